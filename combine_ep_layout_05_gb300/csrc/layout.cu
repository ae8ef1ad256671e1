// Dispatch layout and RDMA token counts.
//
// What is computed ("MORI-EP Benchmark", print_bw_values.py; MSCCL++ PR #860
// get_dispatch_layout and the rank-major commit): for every token its set of
// destination ranks {e / (E/R)}, nodes {e / (E/N)} and experts, the counts of
// tokens per (source rank, destination rank / expert / node), and the
// compacted slot of each (token, rank) and (token, expert) pair in ascending
// token order within its source rank.
//
// How: a CTA owns a chunk of kChunk (256) consecutive tokens of one source
// rank, one token per thread.  Membership is recorded as per-column bitmaps
// in shared memory (one bit per token of the chunk, 8 words per column):
// rank and node columns come from warp ballots, expert columns from
// shared-memory atomicOr (whose return value also exposes a repeated expert
// in the same token).  A token's position among the chunk's tokens of a
// column is a popcount of the bits below it.  Pass 1 writes each chunk's
// column counts to a workspace; pass 2 adds the counts of earlier chunks (no
// cross-CTA waiting, so no spin loops) and writes slots and totals; the
// totals of the node columns also give the RDMA token counts.
#include "layout_device.cuh"

namespace ep {

namespace {

// Small problems (every source rank fits one chunk, Tr <= kChunk, and at
// most kSmallScan tokens precede the last source rank): one launch, one CTA
// per source rank.  A source's slots depend on its own tokens only, so a
// CTA writes them straight from its bitmaps; the token-major offsets and the
// receive totals also need the per-rank counts of earlier sources, which
// each CTA counts itself from their routing rows (a few thousand rank sets
// at most) instead of waiting on other CTAs or on a second launch.  Bitmaps
// have ceil(Tr / 32) words per column, so an 8-token rank zeroes and scans
// one word per column instead of eight.
constexpr int kSmallScan = 4096;

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

// Position of the token at (warp w, lanes below `below`) in column q: the
// set bits of the column's earlier words plus those below it in word w.
__device__ __forceinline__ int column_pos(const uint32_t *col, int w, uint32_t below) {
    int pos = __popc(col[w] & below);
    for (int x = 0; x < w; ++x) pos += __popc(col[x]);
    return pos;
}

__global__ void __launch_bounds__(kLayoutThreads, 1) layout_small_kernel(LayoutArgs a, int W) {
    extern __shared__ uint32_t smem[];
    const Dims &d = a.d;
    uint32_t *bm = smem;                                      // [cols][W]: ranks, experts, nodes
    int32_t *gbase = reinterpret_cast<int32_t *>(smem + d.cols * W);   // [R] earlier sources' tokens
    uint32_t *bm_exp = bm + d.R * W, *bm_node = bm + (d.R + d.E) * W;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int64_t src = blockIdx.x;
    const int nt = (int)d.Tr;
    const int k = (int)d.k;
    const int64_t t = src * d.Tr + tid;                      // this thread's token (tid < nt)
    const bool own = tid < nt;

    // the first 8 routing ids of the own token and of the first earlier
    // token, in flight while shared memory is cleared
    const int64_t nearly = src * d.Tr;                       // tokens of earlier sources
    int64_t ids[8], eids[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ids[i] = own && i < k ? __ldg(a.topk_idx + t * k + i) : -1;
        eids[i] = tid < nearly && i < k ? __ldg(a.topk_idx + (int64_t)tid * k + i) : -1;
    }
    for (int i = tid; i < d.E * W; i += kLayoutThreads) bm_exp[i] = 0;
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
        if (atomicOr(&bm_exp[ue * W + w], bit) & bit) {
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
    if (st) raise_status(a.dev_status, st);
    if (w < W) {
        for (int r = 0; r < (int)d.R; ++r) {
            const uint32_t b = __ballot_sync(kFull, (rmask >> r) & 1);
            if (lane == 0) bm[r * W + w] = b;
        }
        for (int n = 0; n < (int)d.N; ++n) {
            const uint32_t b = __ballot_sync(kFull, (nmask >> n) & 1);
            if (lane == 0) bm_node[n * W + w] = b;
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

    // own token: rank-major slots, token-major offsets, expert and node slots
    if (own) {
        const uint32_t below = lanemask_lt();
        for (int r = 0; r < (int)d.R; ++r) {
            const bool in = (rmask >> r) & 1;
            const int32_t slot = in ? column_pos(bm + r * W, w, below) : -1;
            if (a.is_token_in_rank) a.is_token_in_rank[t * d.R + r] = (uint8_t)in;
            if (a.rank_slot) a.rank_slot[t * d.R + r] = slot;
            if (a.token_major_offset) a.token_major_offset[t * d.R + r] = in ? slot + gbase[r] : -1;
        }
        if (a.expert_slot) {
            auto eslot = [&](int j, int64_t e) {
                a.expert_slot[t * k + j] = (kept >> j) & 1 ? column_pos(bm_exp + e * W, w, below) : -1;
            };
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < k) eslot(j, ids[j]);
            for (int j = 8; j < k; ++j) eslot(j, __ldg(a.topk_idx + t * k + j));
        }
        if (a.node_slot)
            for (int n = 0; n < (int)d.N; ++n)
                a.node_slot[t * d.N + n] = (nmask >> n) & 1 ? column_pos(bm_node + n * W, w, below) : -1;
    }

    // this source's counts (column totals); the last source also writes the
    // receive totals (earlier sources' counts plus its own)
    for (int q = tid; q < (int)d.cols; q += kLayoutThreads) {
        int c = 0;
        for (int x = 0; x < W; ++x) c += __popc(bm[q * W + x]);
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
            for (int x = 0; x < W; ++x) c += __popc(bm_node[n * W + x]);
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

__global__ void __launch_bounds__(kLayoutThreads) layout_count_kernel(LayoutArgs a) {
    extern __shared__ uint32_t smem[];
    layout_count_body(a, blockIdx.x, smem);
}

__global__ void __launch_bounds__(kLayoutThreads) layout_slot_kernel(LayoutArgs a) {
    extern __shared__ uint32_t smem[];
    layout_slot_body<false>(a, blockIdx.x, smem);
}

__global__ void __launch_bounds__(kLayoutThreads) rdma_count_kernel(RdmaArgs a) {
    __shared__ unsigned long long s_algo, s_phys;
    const Dims &d = a.d;
    const ChunkPos cp = chunk_pos(d, blockIdx.x);
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) s_algo = s_phys = 0;
    __syncthreads();
    unsigned algo = 0, phys = 0;
    int st = 0;
    if (tid < cp.nt) {
        const int64_t *row = a.topk_idx + (cp.t0 + tid) * d.k;
        uint64_t nmask = 0;
        for (int j = 0; j < (int)d.k; ++j) {
            const int64_t e = row[j];
            if (e == -1) continue;
            if (e < 0 || e >= d.E) {
                st |= EP_STATUS_BAD_EXPERT;
                continue;
            }
            bool dup = false;
            for (int i = 0; i < j; ++i) dup |= (row[i] == e);
            if (dup) {
                st |= EP_STATUS_DUP_EXPERT;
                continue;
            }
            nmask |= 1ull << node_of(d, (uint32_t)e);
        }
        const int64_t my_node = cp.src / d.G;
        algo = __popcll(nmask);
        phys = __popcll(nmask & ~(1ull << my_node));
    }
    if (st) raise_status(a.dev_status, st);
    for (int o = 16; o; o >>= 1) {
        algo += __shfl_xor_sync(kFull, algo, o);
        phys += __shfl_xor_sync(kFull, phys, o);
    }
    if (lane == 0) {
        atomicAdd(&s_algo, (unsigned long long)algo);
        atomicAdd(&s_phys, (unsigned long long)phys);
    }
    __syncthreads();
    if (tid == 0) {
        atomicAdd(a.algo + cp.src, s_algo);
        if (a.phys) atomicAdd(a.phys + cp.src, s_phys);
    }
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs &a, int32_t *, cudaStream_t st) {
    const Dims &d = a.d;
    cudaError_t e;
#ifndef EP_LAYOUT_SMALL
#define EP_LAYOUT_SMALL 1
#endif
    if (EP_LAYOUT_SMALL && d.cps == 1 && (d.R - 1) * d.Tr <= kSmallScan) {
        const int W = (int)((d.Tr + 31) / 32);
        const size_t sm = (size_t)(d.cols * W + d.R) * 4;
        if (sm > 48 * 1024 &&
            (e = cudaFuncSetAttribute(layout_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
            return e;
        layout_small_kernel<<<(unsigned)d.R, kLayoutThreads, sm, st>>>(a, W);
        return cudaGetLastError();
    }
    const unsigned grid = (unsigned)(d.R * d.cps);
    const size_t s1 = count_smem(d), s2 = slot_smem(d);
    if (s1 > 48 * 1024 &&
        (e = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1)))
        return e;
    if (s2 > 48 * 1024 &&
        (e = cudaFuncSetAttribute(layout_slot_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2)))
        return e;
    layout_count_kernel<<<grid, kLayoutThreads, s1, st>>>(a);
    if ((e = cudaGetLastError())) return e;
    layout_slot_kernel<<<grid, kLayoutThreads, s2, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rdma_count(const RdmaArgs &a, cudaStream_t st) {
    const Dims &d = a.d;
    const unsigned grid = (unsigned)(d.R * d.cps);
    rdma_count_kernel<<<grid, kLayoutThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ep
