// Dispatch: scatter every token row to its destination rows.
//
// What ("MSCCL++ PR #860": throughput dispatch into the rank-major layout,
// one copy per destination rank in a [R dst][R src][Tr] buffer grouped by
// source rank; low-latency dispatch into the expert-major layout, one copy
// per (token, expert), optionally cast to FP8; "MORI-EP Benchmark",
// print_bw_values.py: FP8 is one byte per element plus a 4-byte scale per
// 128 channels).
//
// How: a warp owns one (token, piece) unit: lanes gather the token's
// destination rows from the layout's slots (ballot-compacted into shared
// memory), then stream the piece of the source row once through registers
// with 16-byte loads and write it to every destination with 16-byte stores,
// so each source byte is read from HBM once and each destination byte
// written once.  Rows are split into pieces only when there are too few
// tokens to fill the GPU.
#include <cfloat>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 8;        // warps per CTA
constexpr int kMaxDst = 64;      // destination rows per token (R <= 64, k <= 32)

// Gathers the destination rows of token t into rows[] (ascending rank or
// entry order); returns their number.  Lanes raise status bits for bad slots
// or expert ids.
template <int LAYOUT>
__device__ __forceinline__ int gather_dests(const DispatchArgs &a, int64_t t, int64_t src,
                                            int64_t *rows) {
    const Dims &d = a.d;
    const int lane = threadIdx.x & 31;
    int nd = 0, st = 0;
    if (LAYOUT == EP_RANK_MAJOR) {
        for (int r0 = 0; r0 < (int)d.R; r0 += 32) {
            const int r = r0 + lane;
            int64_t row = -1;
            if (r < d.R) {
                const int32_t slot = a.rank_slot[t * d.R + r];
                if (slot >= 0 && slot < d.Tr) row = ((int64_t)r * d.R + src) * d.Tr + slot;
                else if (slot != -1) st |= EP_STATUS_BAD_SLOT;
            }
            const unsigned m = __ballot_sync(kFull, row >= 0);
            if (row >= 0) rows[nd + __popc(m & lanemask_lt())] = row;
            nd += __popc(m);
        }
    } else {
        int64_t row = -1;
        if (lane < d.k) {
            const int64_t e = a.topk_idx[t * d.k + lane];
            if (e >= 0 && e < d.E) {
                const int32_t slot = a.expert_slot[t * d.k + lane];
                if (slot >= 0 && slot < d.Tr) row = (e * d.R + src) * d.Tr + slot;
                else if (slot != -1) st |= EP_STATUS_BAD_SLOT;
            } else if (e != -1) {
                st |= EP_STATUS_BAD_EXPERT;
            }
        }
        const unsigned m = __ballot_sync(kFull, row >= 0);
        if (row >= 0) rows[__popc(m & lanemask_lt())] = row;
        nd = __popc(m);
    }
    if (st) raise_status(a.dev_status, st);
    __syncwarp();
    return nd;
}

template <int LAYOUT>
__global__ void __launch_bounds__(kWarps * 32) dispatch_bf16_kernel(DispatchArgs a) {
    __shared__ int64_t s_rows[kWarps][kMaxDst];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t hc = d.H / 8;                     // 16-byte chunks per row
    const int64_t pc = a.piece_elems / 8;           // chunks per piece
    const int64_t units = d.T * a.pieces;
    const uint4 *x = reinterpret_cast<const uint4 *>(a.x);
    uint4 *recv = reinterpret_cast<uint4 *>(a.recv);
    int64_t *rows = s_rows[warp];
    constexpr int U = 4;

    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        const int nd = gather_dests<LAYOUT>(a, t, src, rows);
        const int64_t c0 = p * pc, c1 = min(c0 + pc, hc);
        const uint4 *xs = x + t * hc;
        for (int64_t c = c0 + lane; c < c1; c += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int i = 0; i < U; ++i)
                if (c + 32 * i < c1) v[i] = ld_stream(xs + c + 32 * i);
            for (int dd = 0; dd < nd; ++dd) {
                uint4 *dst = recv + rows[dd] * hc;
#pragma unroll
                for (int i = 0; i < U; ++i)
                    if (c + 32 * i < c1) st_v4(dst + c + 32 * i, v[i]);
            }
        }
        __syncwarp();
    }
}

// FP8: a lane casts 16 consecutive channels; 8 lanes cover one 128-channel
// block, so a warp covers 4 blocks per step.
template <int LAYOUT>
__global__ void __launch_bounds__(kWarps * 32) dispatch_fp8_kernel(DispatchArgs a) {
    __shared__ int64_t s_rows[kWarps][kMaxDst];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane >> 3, sub = lane & 7;
    const int64_t nb = d.H / 128;                   // blocks per row
    const int64_t pb = a.piece_elems / 128;         // blocks per piece
    const int64_t units = d.T * a.pieces;
    uint8_t *recv = reinterpret_cast<uint8_t *>(a.recv);
    int64_t *rows = s_rows[warp];

    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        const int nd = gather_dests<LAYOUT>(a, t, src, rows);
        const int64_t b0 = p * pb, b1 = min(b0 + pb, nb);
        for (int64_t bb = b0; bb < b1; bb += 4) {
            const int64_t b = bb + grp;
            const bool act = b < b1;
            const int64_t e0 = b * 128 + sub * 16;  // first channel of this lane
            uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
            if (act) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(a.x + t * d.H + e0);
                v0 = ld_stream(xp);
                v1 = ld_stream(xp + 1);
            }
            float f[16];
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                f[2 * i] = bf16_lo(w[i]);
                f[2 * i + 1] = bf16_hi(w[i]);
            }
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            const float s = __fdiv_rn(amax, 448.0f);
            const float inv = amax > 0.f ? fminf(__fdiv_rn(448.0f, amax), FLT_MAX) : 0.f;
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = pack_e4m3x2(__fmul_rn(f[4 * i], inv), __fmul_rn(f[4 * i + 1], inv));
                const uint32_t hi = pack_e4m3x2(__fmul_rn(f[4 * i + 2], inv), __fmul_rn(f[4 * i + 3], inv));
                q[i] = lo | (hi << 16);
            }
            if (act) {
                const uint4 qv = make_uint4(q[0], q[1], q[2], q[3]);
                for (int dd = 0; dd < nd; ++dd) {
                    const int64_t row = rows[dd];
                    st_v4(recv + row * d.H + e0, qv);
                    if (sub == 0) a.recv_scales[row * nb + b] = s;
                }
            }
        }
        __syncwarp();
    }
}

// Identity expert for FP8 payloads: one warp per receive row; rows past the
// segment's live count are skipped.
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

__global__ void __launch_bounds__(kWarps * 32) dequant_kernel(DequantArgs a) {
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ndst = a.layout == EP_RANK_MAJOR ? d.R : d.E;
    const int64_t total = ndst * d.R * d.Tr, nb = d.H / 128;
    for (int64_t row = (int64_t)blockIdx.x * kWarps + warp; row < total; row += (int64_t)gridDim.x * kWarps) {
        const int64_t seg = row / d.Tr, i = row % d.Tr;
        const int64_t dst = seg / d.R, src = seg % d.R;
        if (i >= a.counts[src * ndst + dst]) continue;
        for (int64_t h0 = (int64_t)lane * 16; h0 < d.H; h0 += 512) {
            const uint4 qv = ld_stream(a.q + row * d.H + h0);
            const float s = a.s[row * nb + h0 / 128];
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
            uint32_t o[8];
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
                float f0, f1, f2, f3;
                e4m3x2_to_f32((uint16_t)(qw[i2] & 0xFFFF), f0, f1);
                e4m3x2_to_f32((uint16_t)(qw[i2] >> 16), f2, f3);
                o[2 * i2] = bf16_exact_product(f0, s) | (bf16_exact_product(f1, s) << 16);
                o[2 * i2 + 1] = bf16_exact_product(f2, s) | (bf16_exact_product(f3, s) << 16);
            }
            uint4 *yp = reinterpret_cast<uint4 *>(a.y + row * d.H + h0);
            st_v4(yp, make_uint4(o[0], o[1], o[2], o[3]));
            st_v4(yp + 1, make_uint4(o[4], o[5], o[6], o[7]));
        }
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
    static int cached[64][4] = {{0}};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    const int key = layout * 2 + dtype;
    if (!cached[dev][key]) {
        if (dtype == EP_BF16)
            cached[dev][key] = layout == EP_RANK_MAJOR ? grid_cap_for(dispatch_bf16_kernel<EP_RANK_MAJOR>)
                                                       : grid_cap_for(dispatch_bf16_kernel<EP_EXPERT_MAJOR>);
        else
            cached[dev][key] = layout == EP_RANK_MAJOR ? grid_cap_for(dispatch_fp8_kernel<EP_RANK_MAJOR>)
                                                       : grid_cap_for(dispatch_fp8_kernel<EP_EXPERT_MAJOR>);
    }
    return cached[dev][key];
}

cudaError_t launch_dispatch(int layout, int dtype, const DispatchArgs &a, int grid, cudaStream_t st) {
    const dim3 blk(kWarps * 32);
    if (dtype == EP_BF16) {
        if (layout == EP_RANK_MAJOR) dispatch_bf16_kernel<EP_RANK_MAJOR><<<grid, blk, 0, st>>>(a);
        else dispatch_bf16_kernel<EP_EXPERT_MAJOR><<<grid, blk, 0, st>>>(a);
    } else {
        if (layout == EP_RANK_MAJOR) dispatch_fp8_kernel<EP_RANK_MAJOR><<<grid, blk, 0, st>>>(a);
        else dispatch_fp8_kernel<EP_EXPERT_MAJOR><<<grid, blk, 0, st>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantArgs &a, cudaStream_t st) {
    const int64_t ndst = a.layout == EP_RANK_MAJOR ? a.d.R : a.d.E;
    const int64_t total = ndst * a.d.R * a.d.Tr;
    int64_t grid = (total + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    dequant_kernel<<<(unsigned)grid, kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ep
