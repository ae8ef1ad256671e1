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

// Reads token t's k expert ids in j order; kept entries set bit `bit` of word
// `w` in their expert column.  Returns the kept-entry mask and rank / node
// masks; status bits for ids outside [-1, E) and repeated ids.
__device__ __forceinline__ uint32_t token_sets(const Dims &d, const int64_t *row, uint32_t *bm_exp,
                                               int w, uint32_t bit, uint64_t &rmask,
                                               uint64_t &nmask, int &st) {
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
            const uint32_t old = atomicOr(&bm_exp[ue * kChunkWords + w], bit);
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

// Fills the chunk's bitmaps: ranks [0, R), experts [R, R+E), nodes [R+E, cols).
// Bitmaps must be zero on entry; ends with __syncthreads().
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
        kept = token_sets(d, a.topk_idx + (cp.t0 + tid) * d.k, bm + d.R * kChunkWords, w, 1u << lane,
                          rmask, nmask, st);
    for (int r = 0; r < (int)d.R; ++r) {
        const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
        if (lane == 0) bm[r * kChunkWords + w] = b;
    }
    if (with_nodes) {
        uint32_t *bn = bm + (d.R + d.E) * kChunkWords;
        for (int n = 0; n < (int)d.N; ++n) {
            const uint32_t b = __ballot_sync(kFull, (nmask >> n) & 1);
            if (lane == 0) bn[n * kChunkWords + w] = b;
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
        for (int w = 0; w < kChunkWords; ++w) cnt += __popc(smem[q * kChunkWords + w]);
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
    uint32_t *bm = smem;                             // [cols * 8] bitmaps
    int32_t *pre = (int32_t *)(smem + d.cols * kChunkWords);   // [cols * 8] slot bases
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
    for (int64_t i = tid; i < ncols * kChunkWords; i += kLayoutThreads) {
        const int64_t q = i / kChunkWords;
        const int ww = (int)(i % kChunkWords);
        int s = base[q];
        for (int x = 0; x < ww; ++x) s += __popc(bm[q * kChunkWords + x]);
        pre[i] = s;
    }
    __syncthreads();

    if (tid < cp.nt) {
        const int64_t t = cp.t0 + tid;
        const uint32_t below = lanemask_lt();
        for (int r = 0; r < (int)d.R; ++r) {
            int32_t slot = -1, off = -1;
            if ((rmask >> r) & 1) {
                const int pos = pre[r * kChunkWords + w] + __popc(bm[r * kChunkWords + w] & below);
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
                        s = pre[q * kChunkWords + w] + __popc(bm[q * kChunkWords + w] & below);
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
                    s = pre[q * kChunkWords + w] + __popc(bm[q * kChunkWords + w] & below);
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

size_t count_smem(const Dims &d) { return (size_t)d.cols * kChunkWords * 4; }

size_t slot_smem(const Dims &d) { return (size_t)(d.cols * kChunkWords * 2 + d.cols + d.R) * 4; }

}  // namespace

}  // namespace ep
