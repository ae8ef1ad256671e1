// Dispatch: scatter every token row to its destination rows.
//
// What ("MSCCL++ PR #860": throughput dispatch into the rank-major layout,
// one copy per destination rank in a [R dst][R src][Tr] buffer grouped by
// source rank; low-latency dispatch into the expert-major layout, one copy
// per (token, expert), optionally cast to FP8; "MORI-EP Benchmark",
// print_bw_values.py: FP8 is one byte per element plus a 4-byte scale per
// 128 channels).
//
// How: a warp owns one (token, piece) unit and its lanes gather the token's
// destination rows from the layout's slots (ballot-compacted into shared
// memory).  Each source byte is read from HBM once and each destination byte
// written once, by one of two kernels:
//  - bf16 from 2048 tokens on: the bulk-copy (TMA) engine.  Lane 0 loads the
//    row into a shared-memory ring with one cp.async.bulk and stores it to
//    every destination with one bulk store each (evict-first in L2);
//  - otherwise, and for FP8: the row streams through registers with 16-byte
//    loads and 16-byte stores to every destination; rows are split into
//    pieces when there are too few tokens to fill the GPU.
#include "dispatch_device.cuh"
#include "vec8.cuh"

namespace ep {

namespace {

template <int LAYOUT>
__global__ void __launch_bounds__(kWarps * 32, EP_LSU_MINB) dispatch_bf16_kernel(DispatchArgs a) {
    const int warp = threadIdx.x >> 5;
    lsu_dispatch_body<LAYOUT, false>(a, warp, (int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps);
}

template <int LAYOUT>
__global__ void __launch_bounds__(kBulkWarps * 32) dispatch_bf16_bulk_kernel(DispatchArgs a) {
    extern __shared__ __align__(128) unsigned char s_buf[];   // [warp][stage][kBulkPieceBytes]
    const int warp = threadIdx.x >> 5;
    bulk_dispatch_body<LAYOUT, false>(a, s_buf, warp, (int64_t)blockIdx.x * kBulkWarps + warp,
                                      (int64_t)gridDim.x * kBulkWarps);
}

template <int LAYOUT, bool WIDE>
__global__ void __launch_bounds__(kWarps * 32) dispatch_fp8_kernel(DispatchArgs a) {
    const int warp = threadIdx.x >> 5;
    if (WIDE)
        fp8_dispatch_body_wide<LAYOUT>(a, warp, (int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps);
    else
        fp8_dispatch_body<LAYOUT, false>(a, warp, (int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps);
}

template <typename K>
int grid_cap_for(K kernel) {
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, kWarps * 32, 0) != cudaSuccess ||
        blocks < 1)
        blocks = 1;
    return blocks * num_sms();
}

}  // namespace

int num_sms() {
    static std::atomic<int> cache[kCacheDevices];
    return cached_per_device(cache, [](int dev) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    });
}

int dispatch_grid_cap(int layout, int dtype) {
    static std::atomic<int> cache[6][kCacheDevices];
    const int key = layout * 2 + dtype;
    return cached_per_device(cache[key], [&](int) {
        if (dtype == EP_BF16)
            return layout == EP_RANK_MAJOR     ? grid_cap_for(dispatch_bf16_kernel<EP_RANK_MAJOR>)
                   : layout == EP_EXPERT_MAJOR ? grid_cap_for(dispatch_bf16_kernel<EP_EXPERT_MAJOR>)
                                               : grid_cap_for(dispatch_bf16_kernel<kNodeMajor>);
        return layout == EP_RANK_MAJOR ? grid_cap_for(dispatch_fp8_kernel<EP_RANK_MAJOR, false>)
                                       : grid_cap_for(dispatch_fp8_kernel<EP_EXPERT_MAJOR, false>);
    });
}

int dispatch_bulk_piece_bytes() { return kBulkPieceBytes; }

cudaError_t launch_dispatch_bulk(int layout, const DispatchArgs &a, cudaStream_t st) {
    const size_t smem = (size_t)kBulkWarps * kBulkStages * kBulkPieceBytes;
    auto kern = layout == EP_RANK_MAJOR     ? dispatch_bf16_bulk_kernel<EP_RANK_MAJOR>
                : layout == EP_EXPERT_MAJOR ? dispatch_bf16_bulk_kernel<EP_EXPERT_MAJOR>
                                            : dispatch_bf16_bulk_kernel<kNodeMajor>;
    // the shared-memory opt-in and the occupancy, once per device (the
    // attribute is per device; setting it again is harmless)
    static std::atomic<int> per_sm[3][kCacheDevices];
    cudaError_t e = cudaSuccess;
    const int blocks = cached_per_device(per_sm[layout], [&](int) {
        int b = 0;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (!e) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kBulkWarps * 32, smem);
        return e ? 0 : (b > 0 ? b : 1);
    });
    if (e) return e;
    const int64_t units = a.d.T * a.pieces;
    int64_t grid = (units + kBulkWarps - 1) / kBulkWarps;
    const int64_t cap = (int64_t)num_sms() * blocks;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, kBulkWarps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_dispatch(int layout, int dtype, const DispatchArgs &a, int grid, cudaStream_t st) {
    const dim3 blk(kWarps * 32);
    if (dtype == EP_BF16) {
        if (layout == EP_RANK_MAJOR) dispatch_bf16_kernel<EP_RANK_MAJOR><<<grid, blk, 0, st>>>(a);
        else if (layout == EP_EXPERT_MAJOR) dispatch_bf16_kernel<EP_EXPERT_MAJOR><<<grid, blk, 0, st>>>(a);
        else dispatch_bf16_kernel<kNodeMajor><<<grid, blk, 0, st>>>(a);
    } else {
        // 32-channel lanes where the buffers are 32-byte aligned
        const bool wide = EP_FP8_WIDE && ((uintptr_t)a.x & 31) == 0 && ((uintptr_t)a.recv & 31) == 0;
        if (layout == EP_RANK_MAJOR) {
            if (wide) dispatch_fp8_kernel<EP_RANK_MAJOR, true><<<grid, blk, 0, st>>>(a);
            else dispatch_fp8_kernel<EP_RANK_MAJOR, false><<<grid, blk, 0, st>>>(a);
        } else {
            if (wide) dispatch_fp8_kernel<EP_EXPERT_MAJOR, true><<<grid, blk, 0, st>>>(a);
            else dispatch_fp8_kernel<EP_EXPERT_MAJOR, false><<<grid, blk, 0, st>>>(a);
        }
    }
    return cudaGetLastError();
}

}  // namespace ep
