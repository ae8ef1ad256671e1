// Device code of the dispatch layout, shared by the layout kernels and the
// fused layout + dispatch kernel.  See layout.cu for what is computed.
#pragma once

#include "ep_internal.cuh"

namespace ep {

namespace {


struct ChunkPos {
    int64_t src, c, t0;  // source rank, chunk index in the rank, first token
    int nt;              // tokens in this chunk
};

__device__ __forceinline__ ChunkPos chunk_pos(const Dims &d, int64_t ci) {
    ChunkPos p;
    p.src = ci / d.cps;
    p.c = ci % d.cps;
    const int64_t tb = p.c * kChunk;
    p.nt = (int)min((int64_t)kChunk, d.Tr - tb);
    p.t0 = p.src * d.Tr + tb;
    return p;
}

// Visits the elements of a [nt][cols] row-major output block in memory
// order, f(o, tl, q) for element o = tl * cols + q, consecutive threads of
// the CTA (NT of them) on consecutive elements (coalesced stores); (tl, q)
// advance by NT elements per step without a division.
template <int NT = kLayoutThreads, typename F>
__device__ __forceinline__ void walk_block(int nt, int cols, F &&f) {
    const int tid = threadIdx.x;
    const int total = nt * cols;
    int tl = tid / cols, q = tid - tl * cols;
    const int dt = NT / cols, dq = NT - dt * cols;
#pragma unroll 4
    for (int o = tid; o < total; o += NT) {
        f(o, tl, q);
        tl += dt;
        q += dq;
        if (q >= cols) {
            q -= cols;
            ++tl;
        }
    }
}

// Routing ids j0 .. j0+7 of one token row (-1 beyond k, and everywhere when
// !valid), all loads in flight together.  vec (k even and the id array
// 16-byte aligned, so every row is): 16-byte loads of id pairs, half the
// memory transactions of 8-byte loads for a thread reading its own row.
__device__ __forceinline__ void load_ids8(const int64_t *row, int j0, int k, bool valid, bool vec,
                                          int64_t (&ids)[8]) {
    if (vec) {
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            if (valid && j0 + i < k) {
                const longlong2 v = __ldg(reinterpret_cast<const longlong2 *>(row + j0 + i));
                ids[i] = v.x;
                ids[i + 1] = v.y;
            } else {
                ids[i] = ids[i + 1] = -1;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) ids[i] = valid && j0 + i < k ? __ldg(row + j0 + i) : -1;
    }
}

// whether load_ids8 may use 16-byte loads on this routing array
__device__ __forceinline__ bool ids_vec(const Dims &d, const int64_t *topk_idx) {
    return (d.k & 1) == 0 && ((uintptr_t)topk_idx & 15) == 0;
}

// Reads token t's k expert ids in j order; kept entries set bit `bit` in
// their expert column of the token's bitmap word (bm_exp: that word's expert
// columns).  Returns the kept-entry mask and rank / node masks; status bits
// for ids outside [-1, E) and repeated ids.  kid (may be null): receives
// the token's k entries, the expert id where kept, else -1.
__device__ __forceinline__ uint32_t token_sets(const Dims &d, const int64_t *row, bool vec, uint32_t *bm_exp,
                                               uint32_t bit, uint64_t &rmask, uint64_t &nmask, int &st,
                                               int16_t *kid = nullptr) {
    uint32_t kept = 0;
    for (int j0 = 0; j0 < (int)d.k; j0 += 8) {
        // the ids' loads first, all in flight (the shared-memory atomics
        // below would otherwise order each load after the previous atomic)
        int64_t ids[8];
        load_ids8(row, j0, (int)d.k, true, vec, ids);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (j0 + i >= (int)d.k) break;
            const int64_t e = ids[i];
            bool keep = false;
            if (e != -1) {
                if (e < 0 || e >= d.E) {
                    st |= EP_STATUS_BAD_EXPERT;
                } else if (atomicOr(&bm_exp[(uint32_t)e], bit) & bit) {
                    st |= EP_STATUS_DUP_EXPERT;
                } else {
                    keep = true;
                    kept |= 1u << (j0 + i);
                    rmask |= 1ull << rank_of(d, (uint32_t)e);
                    nmask |= 1ull << node_of(d, (uint32_t)e);
                }
            }
            if (kid) kid[j0 + i] = keep ? (int16_t)e : (int16_t)-1;
        }
    }
    return kept;
}

// Fills the chunk's bitmaps, word-major ([kChunkWords][cols]: word w of
// column q at bm[w * cols + q], so the lanes of a warp writing different
// columns of one word hit different banks): ranks [0, R), experts [R, R+E),
// nodes [R+E, cols).  Bitmaps must be zero on entry; ends with
// __syncthreads().
__device__ __forceinline__ void build_bitmaps(const LayoutArgs &a, const ChunkPos &cp, uint32_t *bm,
                                              bool with_nodes, uint64_t &rmask, uint32_t &kept,
                                              int &st, uint64_t &nmask, int16_t *kid = nullptr) {
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    nmask = 0;
    rmask = 0;
    kept = 0;
    st = 0;
    if (tid < cp.nt)
        kept = token_sets(d, a.topk_idx + (cp.t0 + tid) * d.k, ids_vec(d, a.topk_idx), bm + w * d.cols + d.R,
                          1u << lane, rmask, nmask, st, kid ? kid + tid * d.k : nullptr);
    for (int r = 0; r < (int)d.R; ++r) {
        const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
        if (lane == 0) bm[w * d.cols + r] = b;
    }
    if (with_nodes) {
        uint32_t *bn = bm + w * d.cols + d.R + d.E;
        for (int n = 0; n < (int)d.N; ++n) {
            const uint32_t b = __ballot_sync(kFull, (nmask >> n) & 1);
            if (lane == 0) bn[n] = b;
        }
    }
    __syncthreads();
}

// Pass 1 for chunk ci: bitmaps, is_token_in_rank, the chunk's column counts.
__device__ __forceinline__ void layout_count_body(const LayoutArgs &a, int64_t ci, uint32_t *smem) {
    const Dims &d = a.d;
    const ChunkPos cp = chunk_pos(d, ci);
    const int tid = threadIdx.x;
    for (int64_t i = tid; i < d.cols * kChunkWords; i += kLayoutThreads) smem[i] = 0;
    __syncthreads();

    uint64_t rmask, nmask;
    uint32_t kept;
    int st;
    build_bitmaps(a, cp, smem, true, rmask, kept, st, nmask);
    if (st) raise_status(a.dev_status, st);

    // is_token_in_rank in memory order, from the rank columns
    if (a.is_token_in_rank)
        walk_block(cp.nt, (int)d.R, [&](int o, int tl, int r) {
            a.is_token_in_rank[cp.t0 * d.R + o] = (uint8_t)((smem[(tl >> 5) * d.cols + r] >> (tl & 31)) & 1);
        });
    int32_t *out = a.chunk_counts + ci * d.cols;
    for (int64_t q = tid; q < d.cols; q += kLayoutThreads) {
        int cnt = 0;
#pragma unroll
        for (int w = 0; w < kChunkWords; ++w) cnt += __popc(smem[w * d.cols + q]);
        out[q] = cnt;
    }
}

// Adds cc[b * cols + q] over chunks b in [b0, b1) and columns q in [0, ncol)
// into acc[q] (shared), spreading the (chunk, column) pairs over the CTA.
template <bool kCG>
__device__ __forceinline__ void add_counts(const int32_t *__restrict__ cc, int64_t cols, int64_t b0,
                                           int64_t b1, int64_t ncol, int32_t *acc) {
    const int64_t n = (b1 - b0) * ncol;
    constexpr int U = 8;
    for (int64_t i0 = (int64_t)threadIdx.x * U; i0 < n; i0 += (int64_t)kLayoutThreads * U) {
        int32_t v[U];
        int64_t q[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = i0 + u;
            v[u] = 0;
            q[u] = 0;
            if (i < n) {
                const int64_t b = b0 + i / ncol;
                q[u] = i % ncol;
                v[u] = kCG ? __ldcg(cc + b * cols + q[u]) : __ldg(cc + b * cols + q[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v[u]) atomicAdd(&acc[q[u]], v[u]);
    }
}

// Pass 2 for chunk ci: counts of earlier chunks, slots, totals.  kCG: read
// the chunk counts from L2 (written earlier in the same kernel).
template <bool kCG>
__device__ __forceinline__ void layout_slot_body(const LayoutArgs &a, int64_t ci, uint32_t *smem) {
    const Dims &d = a.d;
    const ChunkPos cp = chunk_pos(d, ci);
    const int tid = threadIdx.x, w = tid >> 5;
    const int64_t re = d.R + d.E;                    // rank + expert columns; nodes follow
    uint32_t *bm = smem;                             // [8][cols] bitmaps (word-major)
    int32_t *pre = (int32_t *)(smem + d.cols * kChunkWords);   // [8][cols] slot bases (word-major)
    int32_t *base = pre + d.cols * kChunkWords;      // [cols] earlier chunks, same source
    int32_t *gbase = base + d.cols;                  // [R] earlier tokens, any source

    for (int64_t i = tid; i < d.cols * kChunkWords; i += kLayoutThreads) bm[i] = 0;
    for (int64_t i = tid; i < d.cols + d.R; i += kLayoutThreads) base[i] = 0;
    __syncthreads();

    const int64_t seg0 = cp.src * d.cps;             // first chunk of this source rank
    add_counts<kCG>(a.chunk_counts, d.cols, seg0, ci, d.cols, base);
    add_counts<kCG>(a.chunk_counts, d.cols, 0, seg0, d.R, gbase);

    int16_t *kid = (int16_t *)(gbase + d.R);         // [kChunk][k] kept expert ids, -1 otherwise
    uint64_t rmask, nmask;
    uint32_t kept;
    int st;
    build_bitmaps(a, cp, bm, a.node_slot != nullptr, rmask, kept, st, nmask,
                  a.expert_slot ? kid : nullptr);   // ends with a barrier

    // pre[q, w] = base[q] + number of chunk tokens of column q in words
    // before w; one thread per column walks its 8 words (a running prefix),
    // so each word is read once
    const int64_t ncols = a.node_slot ? d.cols : re;
    for (int q = tid; q < (int)ncols; q += kLayoutThreads) {
        int s = base[q];
#pragma unroll
        for (int x = 0; x < kChunkWords; ++x) {
            pre[x * d.cols + q] = s;
            s += __popc(bm[x * d.cols + q]);
        }
    }
    __syncthreads();

    // the outputs in memory order: position of chunk token tl in column q
    // is its column prefix plus the set bits below it in its word
    const int C = (int)d.cols;
    auto member = [&](int tl, int q) { return (bm[(tl >> 5) * C + q] >> (tl & 31)) & 1; };
    auto pos = [&](int tl, int q) {
        const int x = tl >> 5;
        return pre[x * C + q] + __popc(bm[x * C + q] & ((1u << (tl & 31)) - 1));
    };
    const int64_t o0 = cp.t0;   // first token of the chunk
    if (a.rank_slot || a.token_major_offset)
        walk_block(cp.nt, (int)d.R, [&](int o, int tl, int r) {
            const bool in = member(tl, r);
            const int32_t slot = in ? pos(tl, r) : -1;
            if (a.rank_slot) a.rank_slot[o0 * d.R + o] = slot;
            if (a.token_major_offset) a.token_major_offset[o0 * d.R + o] = in ? slot + gbase[r] : -1;
        });
    if (a.expert_slot)
        walk_block(cp.nt, (int)d.k, [&](int o, int tl, int) {
            const int e = kid[o];
            a.expert_slot[o0 * d.k + o] = e >= 0 ? pos(tl, (int)d.R + e) : -1;
        });
    if (a.node_slot)
        walk_block(cp.nt, (int)d.N, [&](int o, int tl, int n) {
            const int q = (int)re + n;
            a.node_slot[o0 * d.N + o] = member(tl, q) ? pos(tl, q) : -1;
        });

    // totals: the last chunk of each source rank, and the very last chunk
    const int32_t *own = a.chunk_counts + ci * d.cols;
    if (cp.c == d.cps - 1) {
        for (int64_t q = tid; q < d.cols; q += kLayoutThreads) {
            const int32_t v = base[q] + (kCG ? __ldcg(own + q) : own[q]);
            if (q < d.R) {
                if (a.tokens_per_rank) a.tokens_per_rank[cp.src * d.R + q] = v;
            } else if (q < re) {
                if (a.tokens_per_expert) a.tokens_per_expert[cp.src * d.E + (q - d.R)] = v;
            } else {
                if (a.tokens_per_node) a.tokens_per_node[cp.src * d.N + (q - re)] = v;
            }
        }
        if (cp.src == d.R - 1 && a.recv_tokens_per_rank)
            for (int64_t r = tid; r < d.R; r += kLayoutThreads)
                a.recv_tokens_per_rank[r] = gbase[r] + base[r] + (kCG ? __ldcg(own + r) : own[r]);
        // RDMA token counts of this source rank: the (token, node) pairs are
        // the node columns' totals; physical drops the source's own node
        if (tid == 0 && (a.algo_per_rank || a.phys_per_rank)) {
            int64_t algo = 0, own_node = 0;
            for (int64_t n = 0; n < d.N; ++n) {
                const int64_t v = base[re + n] + (kCG ? __ldcg(own + re + n) : own[re + n]);
                algo += v;
                if (n == cp.src / d.G) own_node = v;
            }
            if (a.algo_per_rank) a.algo_per_rank[cp.src] = algo;
            if (a.phys_per_rank) a.phys_per_rank[cp.src] = algo - own_node;
        }
    }
}

// Small problems (every source rank fits one chunk, Tr <= kChunk, and at
// most kSmallScan tokens precede the last source rank): one launch, one CTA
// per source rank.  A source's slots depend on its own tokens only, so a
// CTA writes them straight from its bitmaps; the token-major offsets and the
// receive totals also need the per-rank counts of earlier sources, which
// each CTA counts itself from their routing rows (a few thousand rank sets
// at most) instead of waiting on other CTAs or on a second launch.  Bitmaps
// have ceil(Tr / 32) words per column, so an 8-token rank zeroes and scans
// one word per column instead of eight.

// Rank set of 8 routing ids: ranks of the ids in [0, E) (repeats and -1
// change no set).
__device__ __forceinline__ uint64_t rank_set8(const Dims &d, const int64_t (&ids)[8]) {
    uint64_t m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int64_t e = ids[j];
        if (e >= 0 && e < d.E) m |= 1ull << rank_of(d, (uint32_t)e);
    }
    return m;
}

// Rank set of routing row u, ids j0 .. k-1.
__device__ __forceinline__ uint64_t rank_set_row(const Dims &d, const int64_t *row, int j0) {
    uint64_t m = 0;
    for (; j0 < (int)d.k; j0 += 8) {
        int64_t v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = j0 + i < (int)d.k ? __ldg(row + j0 + i) : -1;
        m |= rank_set8(d, v);
    }
    return m;
}

// Shared memory of small_layout_body, in 32-bit words: bitmaps and their
// column prefixes ([W][cols] each), the earlier sources' tokens per rank
// ([R]) and the own tokens' kept expert ids ([Tr][k], 16-bit).
__host__ __device__ __forceinline__ int64_t small_layout_words(const Dims &d, int W) {
    return 2 * d.cols * W + d.R + (d.Tr * d.k + 1) / 2;
}

// Tokens of earlier sources per thread and batch of small_layout_body: their
// ids are loaded together, so the count waits on memory once per batch
constexpr int kEarlyBatch = 4;

// The small-problem layout of source rank `src` (small_layout(d)): one
// token per thread of the first kLayoutThreads threads of an NT-thread CTA;
// smem holds small_layout_words(d, W) words.  primary: writes the layout outputs
// (slots, offsets, counts, totals, RDMA counts) and counts the earlier
// sources' tokens for the token-major offsets and receive totals.  DT
// (EP_RANK_MAJOR or EP_EXPERT_MAJOR; -1: none): also lists each own token's
// destination rows in that layout, dcnt[tl] of them at dtab[tl * w ...]
// (w = R or k), in shared memory the caller provides.
//
// Phases: (1) membership bitmaps of the own tokens (ballots for ranks and
// nodes, shared-memory atomicOr for experts) and the earlier sources'
// tokens per rank, their ids loaded kEarlyBatch tokens per thread at a
// time; with NT = 2 * kLayoutThreads the second half of the CTA counts
// those while the first builds the bitmaps, so the two run side by side;
// (2) column totals and the prefix of each column over its words; (3) the
// outputs, each array written in its own memory order (consecutive threads,
// consecutive elements), a slot being the column prefix plus the set bits
// below the token in its word.
template <int DT, int NT = kLayoutThreads>
__device__ __forceinline__ void small_layout_body(const LayoutArgs &a, int W, uint32_t *smem, int64_t src,
                                                  bool primary, int32_t *dtab, int32_t *dcnt) {
    static_assert(NT == kLayoutThreads || NT == 2 * kLayoutThreads, "one or two sets of warps");
    constexpr bool kSplit = NT == 2 * kLayoutThreads;
    const Dims &d = a.d;
    // bitmaps [W][cols], word-major: word x of column q at bm[x * C + q]
    // (columns: ranks, then experts, then nodes), so the lanes of a warp
    // touching different columns of one word hit different banks
    const int C = (int)d.cols, ce = (int)d.R, cn = (int)(d.R + d.E);   // first expert / node column
    const int R = (int)d.R, N = (int)d.N;
    uint32_t *bm = smem;
    int32_t *pre = reinterpret_cast<int32_t *>(smem + C * W);   // [W][cols] set bits of earlier words
    int32_t *gbase = pre + C * W;                               // [R] earlier sources' tokens
    int16_t *kid = reinterpret_cast<int16_t *>(gbase + R);       // [Tr][k] kept expert id or -1
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nt = (int)d.Tr;
    const int k = (int)d.k;
    const bool counter = !kSplit || tid >= kLayoutThreads;  // counts earlier sources' tokens
    const int te = kSplit ? tid - kLayoutThreads : tid;     // index among the counting threads
    const int64_t t = src * d.Tr + tid;                      // this thread's token (tid < nt)
    const bool own = tid < nt && (!kSplit || tid < kLayoutThreads);
    const bool want_eslot = primary && a.expert_slot;

    // the first 8 routing ids of the own token and those of the first batch
    // of earlier tokens (te + i * kLayoutThreads), in flight while shared
    // memory is cleared
    const int64_t nearly = primary ? src * d.Tr : 0;        // earlier sources' tokens to count
    const bool vec = ids_vec(d, a.topk_idx);
    int64_t ids[8], eids[kEarlyBatch][8];
    load_ids8(a.topk_idx + t * k, 0, k, own, vec, ids);
#pragma unroll
    for (int b = 0; b < kEarlyBatch; ++b) {
        const int64_t u = te + (int64_t)b * kLayoutThreads;
        load_ids8(a.topk_idx + u * k, 0, k, counter && u < nearly, vec, eids[b]);
    }
    for (int i = tid; i < C * W; i += NT) bm[i] = 0;
    for (int i = tid; i < R; i += NT) gbase[i] = 0;
    __syncthreads();

    // own token: expert bits (an atomicOr's old value exposes a repeat),
    // rank and node sets, kept ids for the expert slots
    uint64_t rmask = 0, nmask = 0;
    uint32_t kept = 0;
    int st = 0;
    const uint32_t bit = 1u << lane;
    auto take = [&](int j, int64_t e) {
        bool keep = false;
        if (e != -1) {
            if (e < 0 || e >= d.E) {
                st |= EP_STATUS_BAD_EXPERT;
            } else if (atomicOr(&bm[w * C + ce + (int)e], bit) & bit) {
                st |= EP_STATUS_DUP_EXPERT;
            } else {
                keep = true;
                kept |= 1u << j;
                rmask |= 1ull << rank_of(d, (uint32_t)e);
                nmask |= 1ull << node_of(d, (uint32_t)e);
            }
        }
        if (want_eslot) kid[tid * k + j] = keep ? (int16_t)e : (int16_t)-1;
    };
    if (own) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < k) take(j, ids[j]);
        for (int j = 8; j < k; ++j) take(j, __ldg(a.topk_idx + t * k + j));
    }
    if (st && primary) raise_status(a.dev_status, st);
    if (w < W) {
        for (int r = 0; r < R; ++r) {
            const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
            if (lane == 0) bm[w * C + r] = b;
        }
        for (int n = 0; n < N; ++n) {
            const uint32_t b = __ballot_sync(kFull, (nmask >> n) & 1);
            if (lane == 0) bm[w * C + cn + n] = b;
        }
    }
    // tokens of earlier sources per destination rank (token-major offsets,
    // receive totals): warp-aggregated counts of their rank sets, a batch of
    // kEarlyBatch tokens per thread per memory round trip
    for (int64_t u0 = 0; counter && u0 < nearly; u0 += (int64_t)kEarlyBatch * kLayoutThreads) {
        uint64_t m[kEarlyBatch];
#pragma unroll
        for (int b = 0; b < kEarlyBatch; ++b) {
            const int64_t u = u0 + te + (int64_t)b * kLayoutThreads;
            m[b] = u < nearly ? rank_set8(d, eids[b]) | rank_set_row(d, a.topk_idx + u * k, 8) : 0;
        }
        const int64_t n0 = u0 + (int64_t)kEarlyBatch * kLayoutThreads;   // the next batch
        if (n0 < nearly) {
#pragma unroll
            for (int b = 0; b < kEarlyBatch; ++b) {
                const int64_t u = n0 + te + (int64_t)b * kLayoutThreads;
                load_ids8(a.topk_idx + u * k, 0, k, u < nearly, vec, eids[b]);
            }
        }
        for (int r = 0; r < R; ++r) {
            int c = 0;
#pragma unroll
            for (int b = 0; b < kEarlyBatch; ++b) c += __popc(__ballot_sync(kFull, (m[b] >> r) & 1));
            if (lane == 0 && c) atomicAdd(&gbase[r], c);
        }
    }
    __syncthreads();

    // column totals and prefixes; the counts (the last source also writes
    // the receive totals: earlier sources' counts plus its own)
    for (int q = tid; q < C; q += NT) {
        int c = 0;
#pragma unroll
        for (int x = 0; x < kChunkWords; ++x) {
            if (x < W) {
                pre[x * C + q] = c;
                c += __popc(bm[x * C + q]);
            }
        }
        if (!primary) continue;
        if (q < R) {
            if (a.tokens_per_rank) a.tokens_per_rank[src * R + q] = c;
            if (src == R - 1 && a.recv_tokens_per_rank) a.recv_tokens_per_rank[q] = gbase[q] + c;
        } else if (q < cn) {
            if (a.tokens_per_expert) a.tokens_per_expert[src * d.E + (q - R)] = c;
        } else {
            if (a.tokens_per_node) a.tokens_per_node[src * N + (q - cn)] = c;
        }
    }
    __syncthreads();
    // position of own token tl in column q
    auto pos = [&](int tl, int q) {
        const int x = tl >> 5;
        return pre[x * C + q] + __popc(bm[x * C + q] & ((1u << (tl & 31)) - 1));
    };

    // destination rows of the own token for the caller's table
    if (DT >= 0 && own) {
        int nd = 0;
        if (DT == EP_RANK_MAJOR) {
            for (int r = 0; r < R; ++r)
                if ((rmask >> r) & 1) dtab[tid * R + nd++] = (int32_t)((r * d.R + src) * d.Tr + pos(tid, r));
        } else {
            auto erow = [&](int j, int64_t e) {
                if ((kept >> j) & 1) dtab[tid * k + nd++] = (int32_t)((e * d.R + src) * d.Tr + pos(tid, ce + (int)e));
            };
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < k) erow(j, ids[j]);
            for (int j = 8; j < k; ++j) erow(j, __ldg(a.topk_idx + t * k + j));
        }
        dcnt[tid] = nd;
    }
    if (!primary) return;

    // the outputs in memory order (walk_block: consecutive threads on
    // consecutive elements)
    const int64_t base_r = src * d.Tr * R;
    if (a.is_token_in_rank || a.rank_slot || a.token_major_offset)
        walk_block<NT>(nt, R, [&](int o, int tl, int r) {
            const bool in = (bm[(tl >> 5) * C + r] >> (tl & 31)) & 1;
            const int32_t slot = in ? pos(tl, r) : -1;
            if (a.is_token_in_rank) a.is_token_in_rank[base_r + o] = (uint8_t)in;
            if (a.rank_slot) a.rank_slot[base_r + o] = slot;
            if (a.token_major_offset) a.token_major_offset[base_r + o] = in ? slot + gbase[r] : -1;
        });
    if (want_eslot)
        walk_block<NT>(nt, k, [&](int o, int tl, int) {
            const int e = kid[o];
            a.expert_slot[src * d.Tr * k + o] = e >= 0 ? pos(tl, ce + e) : -1;
        });
    if (a.node_slot)
        walk_block<NT>(nt, N, [&](int o, int tl, int n) {
            const bool in = (bm[(tl >> 5) * C + cn + n] >> (tl & 31)) & 1;
            a.node_slot[src * d.Tr * N + o] = in ? pos(tl, cn + n) : -1;
        });
    // RDMA token counts: (token, node) pairs are the node columns' totals;
    // physical drops the source's own node
    if (w == 0 && (a.algo_per_rank || a.phys_per_rank)) {
        // node column totals fit 32 bits here (at most Tr tokens each)
        int algo = 0, own_node = 0;
        const int my_node = (int)src / (int)d.G;
        for (int n = lane; n < N; n += 32) {
            const int q = cn + n;
            const int c = pre[(W - 1) * C + q] + __popc(bm[(W - 1) * C + q]);
            algo += c;
            if (n == my_node) own_node = c;
        }
        algo = __reduce_add_sync(kFull, algo);
        own_node = __reduce_add_sync(kFull, own_node);
        if (lane == 0) {
            if (a.algo_per_rank) a.algo_per_rank[src] = algo;
            if (a.phys_per_rank) a.phys_per_rank[src] = algo - own_node;
        }
    }
}

// Warps of the tiny-problem layout team of one source rank.
constexpr int kTinyTeam = 4;

// The layout of source rank `src` for tiny problems (tiny_layout(d)),
// computed by a team of kTinyTeam warps, one token per lane (token
// src * Tr + lane), warp-synchronous: the work splits into four chains that
// share nothing but the routing rows, so the team needs no barrier and the
// step takes the longest chain, not their sum.  Every warp derives the
// token's rank and node sets from its ids itself (a repeated id changes no
// set); rank and node columns are single ballots, a slot the popcount of
// the ballot below the lane.
//   tw 0, experts: expert words in bm_exp (E words of shared memory owned
//         by this warp; atomicOr, whose old value exposes a repeat), the
//         status bits, expert slots and counts, expert-major destination
//         rows;
//   tw 1, earlier sources: the tokens of the earlier source ranks per rank
//         (lane r % 32 keeps rank r's count), then the token-major offsets
//         and the receive totals;
//   tw 2, ranks: is_token_in_rank, rank slots and counts, rank-major
//         destination rows;
//   tw 3, nodes: node slots and counts, RDMA token counts.
// primary: writes the layout outputs; DT (EP_RANK_MAJOR, EP_EXPERT_MAJOR or
// -1), dtab and dcnt as in small_layout_body (written by the warp that
// owns the layout's slots).
template <int DT>
__device__ __forceinline__ void tiny_layout_team(const LayoutArgs &a, uint32_t *bm_exp, int64_t src, int tw,
                                                 bool primary, int32_t *dtab, int32_t *dcnt) {
    const Dims &d = a.d;
    const int lane = threadIdx.x & 31;
    const int k = (int)d.k, R = (int)d.R, N = (int)d.N;
    const int64_t t = src * d.Tr + lane;
    const bool own = lane < (int)d.Tr;
    const bool vec = ids_vec(d, a.topk_idx);
    const uint32_t below = lanemask_lt();
    // roles without outputs of a non-primary team (the fused kernel's
    // further CTAs) have nothing to do
    const bool needed = primary || (tw == 0 && DT == EP_EXPERT_MAJOR) || (tw == 2 && DT == EP_RANK_MAJOR);
    if (!needed) return;

    int64_t ids[8];
    load_ids8(a.topk_idx + t * k, 0, k, own, vec, ids);
    if (tw == 1) {
        // earlier sources' tokens per rank, 32 tokens per round, the next
        // round's ids in flight while the current one is counted
        const int64_t nearly = src * d.Tr;
        int64_t eids[8];
        load_ids8(a.topk_idx + (int64_t)lane * k, 0, k, lane < nearly, vec, eids);
        int g0 = 0, g1 = 0;
        for (int64_t u0 = 0; u0 < nearly; u0 += 32) {
            const int64_t u = u0 + lane, un = u + 32;
            int64_t nids[8];
            load_ids8(a.topk_idx + un * k, 0, k, un < nearly, vec, nids);
            const uint64_t m = u < nearly ? rank_set8(d, eids) | rank_set_row(d, a.topk_idx + u * k, 8) : 0;
            for (int r = 0; r < R; ++r) {
                const int c = __popc(__ballot_sync(kFull, (m >> r) & 1));
                if (lane == (r & 31)) {
                    if (r < 32) g0 += c;
                    else g1 += c;
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) eids[i] = nids[i];
        }
        const uint64_t rmask = own ? rank_set8(d, ids) | rank_set_row(d, a.topk_idx + t * k, 8) : 0;
        for (int r = 0; r < R; ++r) {
            const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
            const int gb = __shfl_sync(kFull, r < 32 ? g0 : g1, r & 31);
            const bool in = (rmask >> r) & 1;
            if (own && a.token_major_offset) a.token_major_offset[t * R + r] = in ? __popc(b & below) + gb : -1;
            if (lane == 0 && src == R - 1 && a.recv_tokens_per_rank) a.recv_tokens_per_rank[r] = gb + __popc(b);
        }
        return;
    }
    if (tw == 0) {
        for (int e = lane; e < (int)d.E; e += 32) bm_exp[e] = 0;
        __syncwarp();
        // the atomics of all entries first (their old values are read after)
        uint32_t kept = 0;
        int st = 0;
        const uint32_t bit = 1u << lane;
        uint32_t old[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            old[j] = 0;
            const int64_t e = ids[j];
            if (own && j < k && e >= 0 && e < d.E) old[j] = atomicOr(&bm_exp[(uint32_t)e], bit);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t e = ids[j];
            if (!own || j >= k || e == -1) continue;
            if (e < 0 || e >= d.E) st |= EP_STATUS_BAD_EXPERT;
            else if (old[j] & bit) st |= EP_STATUS_DUP_EXPERT;
            else kept |= 1u << j;
        }
        for (int j = 8; j < k; ++j) {   // entries beyond the first 8
            const int64_t e = own ? __ldg(a.topk_idx + t * k + j) : -1;
            if (e == -1) continue;
            if (e < 0 || e >= d.E) st |= EP_STATUS_BAD_EXPERT;
            else if (atomicOr(&bm_exp[(uint32_t)e], bit) & bit) st |= EP_STATUS_DUP_EXPERT;
            else kept |= 1u << j;
        }
        if (st && primary) raise_status(a.dev_status, st);
        __syncwarp();   // every lane's expert bits are in place
        int nd = 0;
        auto eslot = [&](int j, int64_t e) {
            const int32_t sl = (kept >> j) & 1 ? __popc(bm_exp[e] & below) : -1;
            if (primary && a.expert_slot) a.expert_slot[t * k + j] = sl;
            if (DT == EP_EXPERT_MAJOR && sl >= 0) dtab[lane * k + nd++] = (int32_t)((e * d.R + src) * d.Tr + sl);
        };
        if (own && ((primary && a.expert_slot) || DT == EP_EXPERT_MAJOR)) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < k) eslot(j, ids[j]);
            for (int j = 8; j < k; ++j) eslot(j, __ldg(a.topk_idx + t * k + j));
        }
        if (DT == EP_EXPERT_MAJOR && own) dcnt[lane] = nd;
        if (primary && a.tokens_per_expert)
            for (int e = lane; e < (int)d.E; e += 32) a.tokens_per_expert[src * d.E + e] = __popc(bm_exp[e]);
        return;
    }
    if (tw == 2) {
        const uint64_t rmask = own ? rank_set8(d, ids) | rank_set_row(d, a.topk_idx + t * k, 8) : 0;
        int nd = 0;
        for (int r = 0; r < R; ++r) {
            const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
            const bool in = (rmask >> r) & 1;
            const int32_t slot = in ? __popc(b & below) : -1;
            if (primary) {
                if (own) {
                    if (a.is_token_in_rank) a.is_token_in_rank[t * R + r] = (uint8_t)in;
                    if (a.rank_slot) a.rank_slot[t * R + r] = slot;
                }
                if (lane == 0 && a.tokens_per_rank) a.tokens_per_rank[src * R + r] = __popc(b);
            }
            if (DT == EP_RANK_MAJOR && in) dtab[lane * R + nd++] = (int32_t)((r * d.R + src) * d.Tr + slot);
        }
        if (DT == EP_RANK_MAJOR && own) dcnt[lane] = nd;
        return;
    }
    // tw == 3: node slots and counts; RDMA token counts ((token, node)
    // pairs; the physical count drops the source's own node)
    uint64_t nmask = 0;
    if (own) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t e = ids[j];
            if (j < k && e >= 0 && e < d.E) nmask |= 1ull << node_of(d, (uint32_t)e);
        }
        for (int j = 8; j < k; ++j) {
            const int64_t e = __ldg(a.topk_idx + t * k + j);
            if (e >= 0 && e < d.E) nmask |= 1ull << node_of(d, (uint32_t)e);
        }
    }
    int algo = 0, own_node = 0;
    const int my_node = (int)src / (int)d.G;
    for (int n = 0; n < N; ++n) {
        const uint32_t b = __ballot_sync(kFull, (nmask >> n) & 1);
        if (own && a.node_slot) a.node_slot[t * N + n] = (nmask >> n) & 1 ? __popc(b & below) : -1;
        if (lane == 0 && a.tokens_per_node) a.tokens_per_node[src * N + n] = __popc(b);
        algo += __popc(b);
        if (n == my_node) own_node = __popc(b);
    }
    if (lane == 0) {
        if (a.algo_per_rank) a.algo_per_rank[src] = algo;
        if (a.phys_per_rank) a.phys_per_rank[src] = algo - own_node;
    }
}

size_t count_smem(const Dims &d) { return (size_t)d.cols * kChunkWords * 4; }

size_t slot_smem(const Dims &d) {
    return (size_t)(d.cols * kChunkWords * 2 + d.cols + d.R) * 4 + (size_t)kChunk * d.k * 2;
}

}  // namespace

}  // namespace ep
