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

// Tiny problems: a CTA of kTinyTeam warps per source rank, E words of
// shared memory; no block barrier.
__global__ void __launch_bounds__(kTinyTeam * 32, 1) layout_tiny_kernel(LayoutArgs a) {
    extern __shared__ uint32_t smem[];
    tiny_layout_team<-1>(a, smem, blockIdx.x, threadIdx.x >> 5, true, nullptr, nullptr);
}

// Small problems: a CTA per source rank; its second set of kLayoutThreads
// threads counts the earlier sources' tokens while the first builds the
// bitmaps.
__global__ void __launch_bounds__(2 * kLayoutThreads, 1) layout_small_kernel(LayoutArgs a, int W) {
    extern __shared__ uint32_t smem[];
    small_layout_body<-1, 2 * kLayoutThreads>(a, W, smem, blockIdx.x, true, nullptr, nullptr);
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
    if (EP_LAYOUT_SMALL && tiny_layout(d)) {
        layout_tiny_kernel<<<(unsigned)d.R, kTinyTeam * 32, (size_t)d.E * 4, st>>>(a);
        return cudaGetLastError();
    }
    if (EP_LAYOUT_SMALL && small_layout(d)) {
        const int W = (int)((d.Tr + 31) / 32);
        const size_t sm = (size_t)small_layout_words(d, W) * 4;
        if (sm > 48 * 1024 &&
            (e = cudaFuncSetAttribute(layout_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm)))
            return e;
        layout_small_kernel<<<(unsigned)d.R, 2 * kLayoutThreads, sm, st>>>(a, W);
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
