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

template <int LAYOUT>
__global__ void __launch_bounds__(kWarps * 32) dispatch_fp8_kernel(DispatchArgs a) {
    const int warp = threadIdx.x >> 5;
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
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

int dispatch_grid_cap(int layout, int dtype) {
    static int cached[64][6] = {{0}};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    const int key = layout * 2 + dtype;
    if (!cached[dev][key]) {
        if (dtype == EP_BF16)
            cached[dev][key] = layout == EP_RANK_MAJOR     ? grid_cap_for(dispatch_bf16_kernel<EP_RANK_MAJOR>)
                               : layout == EP_EXPERT_MAJOR ? grid_cap_for(dispatch_bf16_kernel<EP_EXPERT_MAJOR>)
                                                           : grid_cap_for(dispatch_bf16_kernel<kNodeMajor>);
        else
            cached[dev][key] = layout == EP_RANK_MAJOR ? grid_cap_for(dispatch_fp8_kernel<EP_RANK_MAJOR>)
                                                       : grid_cap_for(dispatch_fp8_kernel<EP_EXPERT_MAJOR>);
    }
    return cached[dev][key];
}

int dispatch_bulk_piece_bytes() { return kBulkPieceBytes; }

cudaError_t launch_dispatch_bulk(int layout, const DispatchArgs &a, cudaStream_t st) {
    const size_t smem = (size_t)kBulkWarps * kBulkStages * kBulkPieceBytes;
    auto kern = layout == EP_RANK_MAJOR     ? dispatch_bf16_bulk_kernel<EP_RANK_MAJOR>
                : layout == EP_EXPERT_MAJOR ? dispatch_bf16_bulk_kernel<EP_EXPERT_MAJOR>
                                            : dispatch_bf16_bulk_kernel<kNodeMajor>;
    static bool attr_set[3] = {false, false, false};
    cudaError_t e;
    if (!attr_set[layout]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e) return e;
        attr_set[layout] = true;
    }
    static int per_sm[3] = {0, 0, 0};
    if (!per_sm[layout]) {
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kBulkWarps * 32, smem);
        if (e) return e;
        per_sm[layout] = b > 0 ? b : 1;
    }
    const int64_t units = a.d.T * a.pieces;
    int64_t grid = (units + kBulkWarps - 1) / kBulkWarps;
    const int64_t cap = (int64_t)num_sms() * per_sm[layout];
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
        if (layout == EP_RANK_MAJOR) dispatch_fp8_kernel<EP_RANK_MAJOR><<<grid, blk, 0, st>>>(a);
        else dispatch_fp8_kernel<EP_EXPERT_MAJOR><<<grid, blk, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace ep
