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

// Reads token t's k expert ids in j order; kept entries set bit `bit` in
// their expert column of the token's bitmap word (bm_exp: that word's expert
// columns).  Returns the kept-entry mask and rank / node masks; status bits
// for ids outside [-1, E) and repeated ids.
__device__ __forceinline__ uint32_t token_sets(const Dims &d, const int64_t *row, uint32_t *bm_exp,
                                               uint32_t bit, uint64_t &rmask, uint64_t &nmask, int &st) {
    uint32_t kept = 0;
    for (int j0 = 0; j0 < (int)d.k; j0 += 8) {
        // the ids' loads first, all in flight (the shared-memory atomics
        // below would otherwise order each load after the previous atomic)
        int64_t ids[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ids[i] = j0 + i < (int)d.k ? __ldg(row + j0 + i) : -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t e = ids[i];
            if (e == -1) continue;
            if (e < 0 || e >= d.E) {
                st |= EP_STATUS_BAD_EXPERT;
                continue;
            }
            const uint32_t ue = (uint32_t)e;
            const uint32_t old = atomicOr(&bm_exp[ue], bit);
            if (old & bit) {
                st |= EP_STATUS_DUP_EXPERT;
                continue;
            }
            kept |= 1u << (j0 + i);
            rmask |= 1ull << rank_of(d, ue);
            nmask |= 1ull << node_of(d, ue);
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
                                              int &st, uint64_t &nmask) {
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    nmask = 0;
    rmask = 0;
    kept = 0;
    st = 0;
    if (tid < cp.nt)
        kept = token_sets(d, a.topk_idx + (cp.t0 + tid) * d.k, bm + w * d.cols + d.R, 1u << lane, rmask, nmask,
                          st);
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

    if (tid < cp.nt && a.is_token_in_rank) {
        uint8_t *dst = a.is_token_in_rank + (cp.t0 + tid) * d.R;
        for (int r = 0; r < (int)d.R; ++r) dst[r] = (uint8_t)((rmask >> r) & 1);
    }
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

    uint64_t rmask, nmask;
    uint32_t kept;
    int st;
    build_bitmaps(a, cp, bm, a.node_slot != nullptr, rmask, kept, st, nmask);   // ends with a barrier

    // pre[q, w] = base[q] (+ gbase for the token-major copy below)
    //           + number of chunk tokens of column q in words before w
    const int64_t ncols = a.node_slot ? d.cols : re;
    // one thread per column walks its 8 words (a running prefix), so each
    // word is read once
    for (int q = tid; q < (int)ncols; q += kLayoutThreads) {
        int s = base[q];
#pragma unroll
        for (int x = 0; x < kChunkWords; ++x) {
            pre[x * d.cols + q] = s;
            s += __popc(bm[x * d.cols + q]);
        }
    }
    __syncthreads();

    if (tid < cp.nt) {
        const int64_t t = cp.t0 + tid;
        const uint32_t below = lanemask_lt();
        for (int r = 0; r < (int)d.R; ++r) {
            int32_t slot = -1, off = -1;
            if ((rmask >> r) & 1) {
                const int pos = pre[w * d.cols + r] + __popc(bm[w * d.cols + r] & below);
                slot = pos;
                off = pos + gbase[r];
            }
            if (a.rank_slot) a.rank_slot[t * d.R + r] = slot;
            if (a.token_major_offset) a.token_major_offset[t * d.R + r] = off;
        }
        if (a.expert_slot) {
            const int64_t *row = a.topk_idx + t * d.k;
            for (int j0 = 0; j0 < (int)d.k; j0 += 8) {
                int64_t ids[8];   // loads first, as in token_sets
#pragma unroll
                for (int i = 0; i < 8; ++i) ids[i] = j0 + i < (int)d.k ? __ldg(row + j0 + i) : 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int j = j0 + i;
                    if (j >= (int)d.k) break;
                    int32_t s = -1;
                    if ((kept >> j) & 1) {
                        const int64_t q = d.R + ids[i];
                        s = pre[w * d.cols + q] + __popc(bm[w * d.cols + q] & below);
                    }
                    a.expert_slot[t * d.k + j] = s;
                }
            }
        }
        if (a.node_slot) {
            for (int n = 0; n < (int)d.N; ++n) {
                int32_t s = -1;
                if ((nmask >> n) & 1) {
                    const int64_t q = re + n;
                    s = pre[w * d.cols + q] + __popc(bm[w * d.cols + q] & below);
                }
                a.node_slot[t * d.N + n] = s;
            }
        }
    }

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

// Position of the token at (warp w, lanes below `below`) in column q of
// word-major bitmaps with C columns: the set bits of the column's earlier
// words plus those below it in word w.
__device__ __forceinline__ int column_pos(const uint32_t *bm, int C, int q, int w, uint32_t below) {
    int pos = __popc(bm[w * C + q] & below);
    for (int x = 0; x < w; ++x) pos += __popc(bm[x * C + q]);
    return pos;
}

// The small-problem layout of source rank `src` (small_layout(d)): one
// token per thread of a kLayoutThreads CTA; smem holds cols * W + R words.
// primary: writes the layout outputs (slots, offsets, counts, totals, RDMA
// counts) and counts the earlier sources' tokens for the token-major offsets
// and receive totals.  DT (EP_RANK_MAJOR or EP_EXPERT_MAJOR; -1: none): also
// lists each own token's destination rows in that layout, dcnt[tl] of them
// at dtab[tl * w ...] (w = R or k), in shared memory the caller provides.
template <int DT>
__device__ __forceinline__ void small_layout_body(const LayoutArgs &a, int W, uint32_t *smem, int64_t src,
                                                  bool primary, int32_t *dtab, int32_t *dcnt) {
    const Dims &d = a.d;
    // bitmaps [W][cols], word-major: word x of column q at bm[x * C + q]
    // (columns: ranks, then experts, then nodes), so the lanes of a warp
    // touching different columns of one word hit different banks
    const int C = (int)d.cols, ce = (int)d.R, cn = (int)(d.R + d.E);   // first expert / node column
    uint32_t *bm = smem;
    int32_t *gbase = reinterpret_cast<int32_t *>(smem + d.cols * W);   // [R] earlier sources' tokens
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nt = (int)d.Tr;
    const int k = (int)d.k;
    const int64_t t = src * d.Tr + tid;                      // this thread's token (tid < nt)
    const bool own = tid < nt;

    // the first 8 routing ids of the own token and of the first earlier
    // token, in flight while shared memory is cleared
    const int64_t nearly = primary ? src * d.Tr : 0;        // earlier sources' tokens to count
    int64_t ids[8], eids[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ids[i] = own && i < k ? __ldg(a.topk_idx + t * k + i) : -1;
        eids[i] = tid < nearly && i < k ? __ldg(a.topk_idx + (int64_t)tid * k + i) : -1;
    }
    for (int i = tid; i < C * W; i += kLayoutThreads) bm[i] = 0;
    for (int i = tid; i < d.R; i += kLayoutThreads) gbase[i] = 0;
    __syncthreads();

    // own token: expert bits (an atomicOr's old value exposes a repeat),
    // rank and node sets
    uint64_t rmask = 0, nmask = 0;
    uint32_t kept = 0;
    int st = 0;
    const uint32_t bit = 1u << lane;
    auto take = [&](int j, int64_t e) {
        if (e == -1) return;
        if (e < 0 || e >= d.E) {
            st |= EP_STATUS_BAD_EXPERT;
            return;
        }
        const uint32_t ue = (uint32_t)e;
        if (atomicOr(&bm[w * C + ce + (int)ue], bit) & bit) {
            st |= EP_STATUS_DUP_EXPERT;
            return;
        }
        kept |= 1u << j;
        rmask |= 1ull << rank_of(d, ue);
        nmask |= 1ull << node_of(d, ue);
    };
    if (own) {
#pragma unroll
        for (int j = 0; j < 8; ++j) take(j, ids[j]);   // -1 beyond k
        for (int j = 8; j < k; ++j) take(j, __ldg(a.topk_idx + t * k + j));
    }
    if (st && primary) raise_status(a.dev_status, st);
    if (w < W) {
        for (int r = 0; r < (int)d.R; ++r) {
            const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
            if (lane == 0) bm[w * C + r] = b;
        }
        for (int n = 0; n < (int)d.N; ++n) {
            const uint32_t b = __ballot_sync(kFull, (nmask >> n) & 1);
            if (lane == 0) bm[w * C + cn + n] = b;
        }
    }
    // tokens of earlier sources per destination rank (token-major offsets,
    // receive totals): warp-aggregated counts of their rank sets.  The ids
    // of a thread's next earlier token are loaded while it counts the
    // current one, so the loop waits on memory once, not once per round.
    for (int64_t u0 = 0; u0 < nearly; u0 += kLayoutThreads) {
        const int64_t u = u0 + tid, un = u + kLayoutThreads;
        int64_t nids[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) nids[i] = un < nearly && i < k ? __ldg(a.topk_idx + un * k + i) : -1;
        uint64_t m = 0;
        if (u < nearly) m = rank_set8(d, eids) | rank_set_row(d, a.topk_idx + u * k, 8);
        for (int r = 0; r < (int)d.R; ++r) {
            const int c = __popc(__ballot_sync(kFull, (m >> r) & 1));
            if (lane == 0 && c) atomicAdd(&gbase[r], c);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) eids[i] = nids[i];
    }
    __syncthreads();

    // own token: rank-major slots, token-major offsets, expert and node
    // slots; destination rows for the caller's table
    if (own) {
        const uint32_t below = lanemask_lt();
        int nd = 0;
        for (int r = 0; r < (int)d.R; ++r) {
            const bool in = (rmask >> r) & 1;
            const int32_t slot = in ? column_pos(bm, C, r, w, below) : -1;
            if (primary) {
                if (a.is_token_in_rank) a.is_token_in_rank[t * d.R + r] = (uint8_t)in;
                if (a.rank_slot) a.rank_slot[t * d.R + r] = slot;
                if (a.token_major_offset) a.token_major_offset[t * d.R + r] = in ? slot + gbase[r] : -1;
            }
            if (DT == EP_RANK_MAJOR && in) dtab[(int64_t)tid * d.R + nd++] = (int32_t)((r * d.R + src) * d.Tr + slot);
        }
        if ((primary && a.expert_slot) || DT == EP_EXPERT_MAJOR) {
            auto eslot = [&](int j, int64_t e) {
                const int32_t s = (kept >> j) & 1 ? column_pos(bm, C, ce + (int)e, w, below) : -1;
                if (primary && a.expert_slot) a.expert_slot[t * k + j] = s;
                if (DT == EP_EXPERT_MAJOR && s >= 0) dtab[(int64_t)tid * k + nd++] = (int32_t)((e * d.R + src) * d.Tr + s);
            };
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < k) eslot(j, ids[j]);
            for (int j = 8; j < k; ++j) eslot(j, __ldg(a.topk_idx + t * k + j));
        }
        if (DT >= 0) dcnt[tid] = nd;
        if (primary && a.node_slot)
            for (int n = 0; n < (int)d.N; ++n)
                a.node_slot[t * d.N + n] = (nmask >> n) & 1 ? column_pos(bm, C, cn + n, w, below) : -1;
    }
    if (!primary) return;

    // this source's counts (column totals); the last source also writes the
    // receive totals (earlier sources' counts plus its own)
    for (int q = tid; q < (int)d.cols; q += kLayoutThreads) {
        int c = 0;
        for (int x = 0; x < W; ++x) c += __popc(bm[x * C + q]);
        if (q < d.R) {
            if (a.tokens_per_rank) a.tokens_per_rank[src * d.R + q] = c;
            if (src == d.R - 1 && a.recv_tokens_per_rank) a.recv_tokens_per_rank[q] = gbase[q] + c;
        } else if (q < d.R + d.E) {
            if (a.tokens_per_expert) a.tokens_per_expert[src * d.E + (q - d.R)] = c;
        } else {
            if (a.tokens_per_node) a.tokens_per_node[src * d.N + (q - d.R - d.E)] = c;
        }
    }
    // RDMA token counts: (token, node) pairs are the node columns' totals;
    // physical drops the source's own node
    if (w == 0 && (a.algo_per_rank || a.phys_per_rank)) {
        int64_t algo = 0, own_node = 0;
        const int my_node = (int)src / (int)d.G;
        for (int n = lane; n < (int)d.N; n += 32) {
            int c = 0;
            for (int x = 0; x < W; ++x) c += __popc(bm[x * C + cn + n]);
            algo += c;
            if (n == my_node) own_node = c;
        }
        for (int o = 16; o; o >>= 1) {
            algo += __shfl_xor_sync(kFull, algo, o);
            own_node += __shfl_xor_sync(kFull, own_node, o);
        }
        if (lane == 0) {
            if (a.algo_per_rank) a.algo_per_rank[src] = algo;
            if (a.phys_per_rank) a.phys_per_rank[src] = algo - own_node;
        }
    }
}


// The layout of source rank `src` computed by one warp, warp-synchronous
// (tiny_layout(d)): token src * Tr + lane in each lane.  Rank and node
// columns are single ballots (a slot is the popcount of the ballot below
// the lane), expert columns one word each in bm_exp (E words of shared
// memory owned by this warp), and the earlier source ranks' tokens are
// counted per rank by the same warp, so no block barrier is needed.
// primary, DT, dtab and dcnt as in small_layout_body.
template <int DT>
__device__ __forceinline__ void tiny_layout_warp(const LayoutArgs &a, uint32_t *bm_exp, int64_t src, bool primary,
                                                 int32_t *dtab, int32_t *dcnt) {
    const Dims &d = a.d;
    const int lane = threadIdx.x & 31;
    const int k = (int)d.k, R = (int)d.R, N = (int)d.N;
    const int64_t t = src * d.Tr + lane;
    const bool own = lane < (int)d.Tr;
    const int64_t nearly = primary ? src * d.Tr : 0;   // earlier sources' tokens to count
    // the first 8 ids of the own token and of the lane's first earlier
    // token, in flight while the expert words are cleared
    int64_t ids[8], eids[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ids[i] = own && i < k ? __ldg(a.topk_idx + t * k + i) : -1;
        eids[i] = lane < nearly && i < k ? __ldg(a.topk_idx + (int64_t)lane * k + i) : -1;
    }
    for (int e = lane; e < (int)d.E; e += 32) bm_exp[e] = 0;
    __syncwarp();

    // own token: expert bits (an atomicOr's old value exposes a repeat),
    // rank and node sets
    uint64_t rmask = 0, nmask = 0;
    uint32_t kept = 0;
    int st = 0;
    const uint32_t bit = 1u << lane;
    auto take = [&](int j, int64_t e) {
        if (e == -1) return;
        if (e < 0 || e >= d.E) {
            st |= EP_STATUS_BAD_EXPERT;
            return;
        }
        const uint32_t ue = (uint32_t)e;
        if (atomicOr(&bm_exp[ue], bit) & bit) {
            st |= EP_STATUS_DUP_EXPERT;
            return;
        }
        kept |= 1u << j;
        rmask |= 1ull << rank_of(d, ue);
        nmask |= 1ull << node_of(d, ue);
    };
    if (own) {
#pragma unroll
        for (int j = 0; j < 8; ++j) take(j, ids[j]);   // -1 beyond k
        for (int j = 8; j < k; ++j) take(j, __ldg(a.topk_idx + t * k + j));
    }
    if (st && primary) raise_status(a.dev_status, st);

    // earlier source ranks' tokens per destination rank: lane r % 32 keeps
    // rank r's count (g0 for ranks below 32, g1 above)
    int g0 = 0, g1 = 0;
    for (int64_t u0 = 0; u0 < nearly; u0 += 32) {
        const int64_t u = u0 + lane, un = u + 32;
        int64_t nids[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) nids[i] = un < nearly && i < k ? __ldg(a.topk_idx + un * k + i) : -1;
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
    __syncwarp();   // every lane's expert bits are in place

    const uint32_t below = lanemask_lt();
    int nd = 0;
    for (int r = 0; r < R; ++r) {
        const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
        const int gb = __shfl_sync(kFull, r < 32 ? g0 : g1, r & 31);
        const bool in = (rmask >> r) & 1;
        const int32_t slot = in ? __popc(b & below) : -1;
        if (primary) {
            if (own) {
                if (a.is_token_in_rank) a.is_token_in_rank[t * R + r] = (uint8_t)in;
                if (a.rank_slot) a.rank_slot[t * R + r] = slot;
                if (a.token_major_offset) a.token_major_offset[t * R + r] = in ? slot + gb : -1;
            }
            if (lane == 0) {
                if (a.tokens_per_rank) a.tokens_per_rank[src * R + r] = __popc(b);
                if (src == R - 1 && a.recv_tokens_per_rank) a.recv_tokens_per_rank[r] = gb + __popc(b);
            }
        }
        if (DT == EP_RANK_MAJOR && in) dtab[lane * R + nd++] = (int32_t)((r * d.R + src) * d.Tr + slot);
    }
    if (own && ((primary && a.expert_slot) || DT == EP_EXPERT_MAJOR)) {
        auto eslot = [&](int j, int64_t e) {
            const int32_t s = (kept >> j) & 1 ? __popc(bm_exp[e] & below) : -1;
            if (primary && a.expert_slot) a.expert_slot[t * k + j] = s;
            if (DT == EP_EXPERT_MAJOR && s >= 0) dtab[lane * k + nd++] = (int32_t)((e * d.R + src) * d.Tr + s);
        };
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < k) eslot(j, ids[j]);
        for (int j = 8; j < k; ++j) eslot(j, __ldg(a.topk_idx + t * k + j));
    }
    if (DT >= 0 && own) dcnt[lane] = nd;
    if (!primary) return;

    // node slots and counts; RDMA token counts ((token, node) pairs; the
    // physical count drops the source's own node)
    int64_t algo = 0, own_node = 0;
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
    if (a.tokens_per_expert)
        for (int e = lane; e < (int)d.E; e += 32) a.tokens_per_expert[src * d.E + e] = __popc(bm_exp[e]);
}

size_t count_smem(const Dims &d) { return (size_t)d.cols * kChunkWords * 4; }

size_t slot_smem(const Dims &d) { return (size_t)(d.cols * kChunkWords * 2 + d.cols + d.R) * 4; }

}  // namespace

}  // namespace ep
