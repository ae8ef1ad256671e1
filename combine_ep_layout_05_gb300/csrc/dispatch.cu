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

__device__ __forceinline__ uint32_t bf16_exact_product(float v, float s) {
    // v * s needs up to 28 significant bits.  hi + lo is the exact product
    // (lo from an fma); bf16(hi) is its correct rounding unless hi sits
    // exactly on a bf16 midpoint and lo != 0, in which case lo's sign
    // decides.
    const float hi = __fmul_rn(v, s);
    const float lo = __fmaf_rn(v, s, -hi);
    const uint32_t hb = __float_as_uint(hi);
    uint32_t r = pack_bf16x2(hi, 0.f) & 0xFFFFu;
    if ((hb & 0xFFFFu) == 0x8000u && lo != 0.f) r = (hb >> 16) + (((lo > 0.f) == (hi > 0.f)) ? 1u : 0u);
    return r;
}

__device__ __forceinline__ void e4m3x2_to_f32(uint16_t c2, float &lo, float &hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h; }"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// Identity expert for FP8 payloads: a warp owns one (token, piece) unit and
// converts that piece of each of the token's receive rows (found from the
// dispatch handle as in dispatch), so the work is balanced and small batches
// still spread over the GPU.
template <int LAYOUT>
__global__ void __launch_bounds__(kWarps * 32) dequant_kernel(DispatchArgs a, uint16_t *y) {
    __shared__ int64_t s_rows[kWarps][kMaxDst];
    constexpr int DU = EP_DEQ_U;
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nb = d.H / 128;
    const uint8_t *q = reinterpret_cast<const uint8_t *>(a.recv);
    int64_t *rows = s_rows[warp];
    const int64_t units = d.T * a.pieces;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int nd = gather_dests<LAYOUT>(a, t, t / d.Tr, rows);
        const int64_t hb = p * a.piece_elems, he = min(hb + a.piece_elems, d.H);
        for (int dd = 0; dd < nd; ++dd) {
            const int64_t row = rows[dd];
            for (int64_t h00 = hb + (int64_t)lane * 16; h00 < he; h00 += 512 * DU) {
                uint4 qv[DU];
                float sc[DU];
#pragma unroll
                for (int uu = 0; uu < DU; ++uu) {
                    const int64_t h0 = h00 + 512 * uu;
                    if (h0 < he) {
                        qv[uu] = ld_stream(q + row * d.H + h0);
                        sc[uu] = a.recv_scales[row * nb + h0 / 128];
                    }
                }
#pragma unroll
                for (int uu = 0; uu < DU; ++uu) {
                    const int64_t h0 = h00 + 512 * uu;
                    if (h0 >= he) continue;
                    const uint32_t qw[4] = {qv[uu].x, qv[uu].y, qv[uu].z, qv[uu].w};
                    uint32_t o[8];
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) {
                        float f0, f1, f2, f3;
                        e4m3x2_to_f32((uint16_t)(qw[i2] & 0xFFFF), f0, f1);
                        e4m3x2_to_f32((uint16_t)(qw[i2] >> 16), f2, f3);
                        o[2 * i2] = bf16_exact_product(f0, sc[uu]) | (bf16_exact_product(f1, sc[uu]) << 16);
                        o[2 * i2 + 1] = bf16_exact_product(f2, sc[uu]) | (bf16_exact_product(f3, sc[uu]) << 16);
                    }
                    uint4 *yp = reinterpret_cast<uint4 *>(y + row * d.H + h0);
                    st_v4(yp, make_uint4(o[0], o[1], o[2], o[3]));
                    st_v4(yp + 1, make_uint4(o[4], o[5], o[6], o[7]));
                }
            }
        }
        __syncwarp();
    }
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

cudaError_t launch_dequant(int layout, const DispatchArgs &a, uint16_t *y, cudaStream_t st) {
    int64_t grid = (a.d.T * a.pieces + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (layout == EP_RANK_MAJOR) dequant_kernel<EP_RANK_MAJOR><<<(unsigned)grid, kWarps * 32, 0, st>>>(a, y);
    else dequant_kernel<EP_EXPERT_MAJOR><<<(unsigned)grid, kWarps * 32, 0, st>>>(a, y);
    return cudaGetLastError();
}

}  // namespace ep
