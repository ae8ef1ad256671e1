// Fused dispatch layout + dispatch in one cooperative launch.
//
// The pages pair the layout ("notify") with the dispatch that consumes it
// (MSCCL++ PR #860: notify_dispatch / dispatch, and the cached
// previous_handle path that skips the host wait).  Here the pair is one
// kernel with three phases over a grid whose CTAs are all resident
// (cooperative launch):
//   1. each CTA builds the bitmaps and column counts of its layout chunks;
//   2. after a grid barrier, it adds the earlier chunks' counts and writes
//      slots, counts and RDMA token counts (the same code as ep_layout);
//   3. after a second barrier, all CTAs dispatch all tokens (bulk copies,
//      register copies or FP8, as ep_dispatch chooses), reading the slots
//      other CTAs wrote from L2.
// This removes two launches and the host-visible gap between them; the
// outputs are identical to ep_layout followed by ep_dispatch.  Small
// problems take a kernel without grid barriers instead (below).
//
// The grid barrier is a counter in the workspace (zeroed before the launch)
// polled a bounded number of times; on time-out the kernel raises
// EP_STATUS_TIMEOUT and its CTAs return instead of waiting on.
#include "dispatch_device.cuh"
#include "layout_device.cuh"

namespace ep {

namespace {

constexpr uint32_t kGridBarrierPolls = 1u << 26;   // ~seconds of polling at most

// Every CTA adds one to *count, then thread 0 waits (bounded) until it
// reaches `target`.  Returns false (for the whole CTA) on time-out.
__device__ __forceinline__ bool grid_barrier(unsigned *count, unsigned target, int32_t *status) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(count, 1u);
        const int ok = wait_counter_bounded(count, target, kGridBarrierPolls) ? 1 : 0;
        if (!ok) raise_status(status, EP_STATUS_TIMEOUT);
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

template <int LAYOUT, int MODE>
__global__ void __launch_bounds__(kLayoutThreads, 1)
    layout_dispatch_kernel(LayoutArgs la, DispatchArgs da, unsigned *bar) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int64_t nchunks = la.d.R * la.d.cps;
    for (int64_t ci = blockIdx.x; ci < nchunks; ci += gridDim.x) {
        layout_count_body(la, ci, reinterpret_cast<uint32_t *>(smem));
        __syncthreads();
    }
    if (!grid_barrier(bar, gridDim.x, la.dev_status)) return;
    for (int64_t ci = blockIdx.x; ci < nchunks; ci += gridDim.x) {
        layout_slot_body<true>(la, ci, reinterpret_cast<uint32_t *>(smem));
        __syncthreads();
    }
    if (!grid_barrier(bar, 2 * gridDim.x, la.dev_status)) return;
    // the bulk copies below write shared memory the layout phases used
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    if constexpr (MODE == kFusedBulk) {
        if (warp < kBulkWarps)
            bulk_dispatch_body<LAYOUT, true>(da, smem, warp, (int64_t)blockIdx.x * kBulkWarps + warp,
                                             (int64_t)gridDim.x * kBulkWarps);
    } else if constexpr (MODE == kFusedLsu) {
        lsu_dispatch_body<LAYOUT, true>(da, warp, (int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps);
    } else {
        fp8_dispatch_body<LAYOUT, true>(da, warp, (int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps);
    }
}

// Small problems (small_layout(d), register-copy or FP8 dispatch): one
// launch with no grid barrier.  A source rank's slots depend only on its own
// tokens, so each CTA builds the layout of one source rank itself (P CTAs per
// source; the first writes the layout outputs and counts the earlier
// sources' tokens) and keeps the destination rows of that source's tokens
// in shared memory; its warps then dispatch their share of the source's
// (token, piece) units from that table.  No CTA reads what another writes.
template <int LAYOUT, int MODE, bool WIDE>
__global__ void __launch_bounds__(kLayoutThreads, 1)
    layout_dispatch_small_kernel(LayoutArgs la, DispatchArgs da, int W, int P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const Dims &d = la.d;
    const int64_t src = blockIdx.x / P, part = blockIdx.x % P;
    uint32_t *lsm = reinterpret_cast<uint32_t *>(smem);                 // layout scratch
    int32_t *dcnt = reinterpret_cast<int32_t *>(lsm + small_layout_words(d, W));  // [Tr]
    int32_t *dtab = dcnt + d.Tr;                                          // [Tr][R or k]
    if (tiny_layout(d)) {
        if (threadIdx.x < kTinyTeam * 32)
            tiny_layout_team<LAYOUT>(la, lsm, src, threadIdx.x >> 5, part == 0, dtab, dcnt);
    } else {
        small_layout_body<LAYOUT>(la, W, lsm, src, part == 0, dtab, dcnt);
    }
    __syncthreads();
    DispatchArgs a = da;
    a.dtab = dtab;
    a.dcnt = dcnt;
    a.dtab_w = LAYOUT == EP_RANK_MAJOR ? d.R : d.k;
    const int warp = threadIdx.x >> 5;
    const int64_t first = src * d.Tr * a.pieces + part * kWarps + warp;
    const int64_t end = (src + 1) * d.Tr * a.pieces;
    if constexpr (MODE == kFusedLsu)
        lsu_dispatch_body<kTableDests, false>(a, warp, first, (int64_t)P * kWarps, end);
    else if constexpr (WIDE)
        fp8_dispatch_body_wide<kTableDests>(a, warp, first, (int64_t)P * kWarps, end);
    else
        fp8_dispatch_body<kTableDests, false>(a, warp, first, (int64_t)P * kWarps, end);
}

template <int LAYOUT, int MODE>
cudaError_t launch_fused_small_t(const LayoutArgs &la, const DispatchArgs &da, cudaStream_t st) {
    static_assert(kLayoutThreads == kWarps * 32, "the fused kernel runs layout chunks and dispatch warps");
    const Dims &d = la.d;
    const int W = (int)((d.Tr + 31) / 32);
    const int64_t tw = LAYOUT == EP_RANK_MAJOR ? d.R : d.k;
    const size_t smem = (size_t)(small_layout_words(d, W) + d.Tr + d.Tr * tw) * 4;
    // FP8: 32-channel lanes where x and recv are 32-byte aligned, as ep_dispatch
    const bool wide = MODE == kFusedFp8 && EP_FP8_WIDE && ((uintptr_t)da.x & 31) == 0 &&
                      ((uintptr_t)da.recv & 31) == 0;
    auto kern = wide ? layout_dispatch_small_kernel<LAYOUT, MODE, true> : layout_dispatch_small_kernel<LAYOUT, MODE, false>;
    cudaError_t e;
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
        return e;
    // CTAs per source rank: about one wave of the GPU in all, no more than
    // the source's units keep busy
    const int64_t units = d.Tr * da.pieces;
    int64_t P = ((int64_t)num_sms() + d.R - 1) / d.R;
    const int64_t pmax = (units + kWarps - 1) / kWarps;
    if (P > pmax) P = pmax;
    if (P < 1) P = 1;
    kern<<<(unsigned)(d.R * P), kLayoutThreads, smem, st>>>(la, da, W, (int)P);
    return cudaGetLastError();
}

template <int LAYOUT, int MODE>
cudaError_t launch_fused_t(const LayoutArgs &la, const DispatchArgs &da, unsigned *bar, cudaStream_t st) {
    static_assert(kLayoutThreads == kWarps * 32, "the fused kernel runs layout chunks and dispatch warps");
    const Dims &d = la.d;
    size_t smem = count_smem(d) > slot_smem(d) ? count_smem(d) : slot_smem(d);
    if (MODE == kFusedBulk && smem < (size_t)kBulkWarps * kBulkStages * kBulkPieceBytes)
        smem = (size_t)kBulkWarps * kBulkStages * kBulkPieceBytes;
    auto kern = layout_dispatch_kernel<LAYOUT, MODE>;
    cudaError_t e;
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
        return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLayoutThreads, smem))) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    // enough CTAs for the work, never more than can be resident at once
    const int64_t nchunks = d.R * d.cps;
    const int64_t wpc = MODE == kFusedBulk ? kBulkWarps : kWarps;
    int64_t want = (d.T * da.pieces + wpc - 1) / wpc;
    if (want < nchunks) want = nchunks;
    int64_t grid = (int64_t)num_sms() * per_sm;
    if (grid > want) grid = want;
    if (grid < 1) grid = 1;
    if ((e = cudaMemsetAsync(bar, 0, sizeof(unsigned), st))) return e;
    LayoutArgs la_ = la;
    DispatchArgs da_ = da;
    unsigned *bar_ = bar;
    void *args[] = {&la_, &da_, &bar_};
    return cudaLaunchCooperativeKernel((const void *)kern, dim3((unsigned)grid), dim3(kLayoutThreads), args, smem,
                                       st);
}

// Self-test of the bounded waits: the counter wait of the grid barrier on a
// word nothing increments, and the mbarrier wait of the bulk copies on a
// barrier that expects bytes no copy delivers.  Both must give up after
// `polls` polls; result[0] gets bit 0 / bit 1 for each wait that did.
__global__ void wait_selftest_kernel(unsigned *word, uint32_t polls, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    unsigned res = 0;
    if (!wait_counter_bounded(word + 1, 1u, polls)) {
        res |= 1u;
        raise_status(status, EP_STATUS_TIMEOUT);
    }
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_expect_tx(&bar, 16);   // 16 bytes that no copy will bring
    bool done = false;
    for (uint32_t i = 0; i < polls && !done; ++i) done = mbar_try_wait(&bar, 0);
    if (!done) {
        res |= 2u;
        raise_status(status, EP_STATUS_TIMEOUT);
    }
    word[0] = res;
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned *word, uint32_t polls, int32_t *status, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(word, polls, status);
    return cudaGetLastError();
}

cudaError_t launch_layout_dispatch(int layout, int mode, const LayoutArgs &la, const DispatchArgs &da,
                                   unsigned *bar, cudaStream_t st) {
    if (small_layout(la.d) && mode != kFusedBulk) {
        if (layout == EP_RANK_MAJOR)
            return mode == kFusedLsu ? launch_fused_small_t<EP_RANK_MAJOR, kFusedLsu>(la, da, st)
                                     : launch_fused_small_t<EP_RANK_MAJOR, kFusedFp8>(la, da, st);
        return mode == kFusedLsu ? launch_fused_small_t<EP_EXPERT_MAJOR, kFusedLsu>(la, da, st)
                                 : launch_fused_small_t<EP_EXPERT_MAJOR, kFusedFp8>(la, da, st);
    }
    if (layout == EP_RANK_MAJOR) {
        if (mode == kFusedBulk) return launch_fused_t<EP_RANK_MAJOR, kFusedBulk>(la, da, bar, st);
        if (mode == kFusedLsu) return launch_fused_t<EP_RANK_MAJOR, kFusedLsu>(la, da, bar, st);
        return launch_fused_t<EP_RANK_MAJOR, kFusedFp8>(la, da, bar, st);
    }
    if (mode == kFusedBulk) return launch_fused_t<EP_EXPERT_MAJOR, kFusedBulk>(la, da, bar, st);
    if (mode == kFusedLsu) return launch_fused_t<EP_EXPERT_MAJOR, kFusedLsu>(la, da, bar, st);
    return launch_fused_t<EP_EXPERT_MAJOR, kFusedFp8>(la, da, bar, st);
}

}  // namespace ep
