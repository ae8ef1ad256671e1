// Combine: weighted top-k gather back to token order.
//
// What ("MORI-EP Benchmark", "Combine": the reverse of dispatch, same byte
// counts; MSCCL++ PR #860: combine reads the receiver-side layout, and in the
// expert-major layout each expert returns one copy per dispatched token):
//   out[t] = bf16( sum_j w[t, j] * y[row(t, j)] ), fp32 accumulation.
//
// How: a warp owns one (token, piece) unit.  Lanes j < k read the routing
// entry, drop ids outside [0, E) and repeats (match_any), and resolve the
// receive row.  In the rank-major layout the experts of one rank share a
// row: lanes group by rank (match_any), sum their weights in j order, and
// only the group leader keeps the row, so each live row is read from HBM
// exactly once.  The piece is then produced 8 channels per lane: up to 8
// source rows are loaded back to back (16-byte loads, all in flight), then
// accumulated with fp32 FMAs, rounded to bf16 and stored with one 16-byte
// store.  Deterministic: no atomics, fixed order.
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kWarps = 8;
#ifndef EP_COMBINE_G
#define EP_COMBINE_G 8
#endif
#ifndef EP_COMBINE_MINB
#define EP_COMBINE_MINB 3
#endif
#ifndef EP_COMBINE_LD_HINT
#define EP_COMBINE_LD_HINT 0
#endif

__device__ __forceinline__ void e4m3x2_to_f32_c(uint16_t c2, float &lo, float &hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h; }"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

template <int LAYOUT>
__device__ __forceinline__ int gather_sources(const CombineArgs &a, int64_t t, int64_t src,
                                              int64_t *rows, float *wts) {
    const Dims &d = a.d;
    const int lane = threadIdx.x & 31;
    int st = 0;
    int64_t e = -1;
    float w = 0.f;
    if (lane < d.k) {
        e = a.topk_idx[t * d.k + lane];
        w = a.topk_weights[t * d.k + lane];
    }
    const bool in_range = e >= 0 && e < d.E;
    if (lane < d.k && !in_range && e != -1) st |= EP_STATUS_BAD_EXPERT;
    // repeated expert ids: only the lowest lane of a match group is kept
    const long long key = in_range ? (long long)e : -2 - lane;
    const unsigned same = __match_any_sync(kFull, key);
    const bool dup = in_range && (same & lanemask_lt());
    if (dup) st |= EP_STATUS_DUP_EXPERT;
    const bool kept = in_range && !dup;

    int64_t row = -1;
    float wsum = w;
    if (LAYOUT == EP_RANK_MAJOR) {
        const int r = kept ? (int)((uint32_t)e / (uint32_t)d.Er) : -1;
        const unsigned grp = __match_any_sync(kFull, kept ? r : -100 - lane);
        const bool leader = kept && !(grp & lanemask_lt());
        // weight of the rank: the group's weights summed in j order
        wsum = 0.f;
        for (int j = 0; j < (int)d.k; ++j) {
            const float wj = __shfl_sync(kFull, w, j);
            if (leader && ((grp >> j) & 1)) wsum += wj;
        }
        if (leader) {
            const int32_t slot = a.rank_slot[t * d.R + r];
            if (slot >= 0 && slot < d.Tr) row = ((int64_t)r * d.R + src) * d.Tr + slot;
            else st |= EP_STATUS_BAD_SLOT;
        }
    } else {
        if (kept) {
            const int32_t slot = a.expert_slot[t * d.k + lane];
            if (slot >= 0 && slot < d.Tr) row = (e * d.R + src) * d.Tr + slot;
            else st |= EP_STATUS_BAD_SLOT;
        }
    }
    if (st) raise_status(a.dev_status, st);
    const unsigned m = __ballot_sync(kFull, row >= 0);
    if (row >= 0) {
        const int i = __popc(m & lanemask_lt());
        rows[i] = row;
        wts[i] = wsum;
    }
    __syncwarp();
    return __popc(m);
}

template <int LAYOUT>
__global__ void __launch_bounds__(kWarps * 32, EP_COMBINE_MINB) combine_kernel(CombineArgs a) {
    __shared__ int64_t s_rows[kWarps][32];
    __shared__ float s_w[kWarps][32];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t hc = d.H / 8;
    const int64_t pc = a.piece_elems / 8;
    const int64_t units = d.T * a.pieces;
    const uint4 *y = reinterpret_cast<const uint4 *>(a.y);
    uint4 *out = reinterpret_cast<uint4 *>(a.out);
    int64_t *rows = s_rows[warp];
    float *wts = s_w[warp];
    constexpr int G = EP_COMBINE_G;   // source rows loaded back to back
    const uint64_t pol = l2_policy<EP_COMBINE_LD_HINT>();

    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        const int nd = gather_sources<LAYOUT>(a, t, src, rows, wts);
        const int64_t c0 = p * pc, c1 = min(c0 + pc, hc);
        for (int64_t c = c0 + lane; c < c1; c += 32) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
            for (int g0 = 0; g0 < nd; g0 += G) {
                uint4 v[G];
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if (g0 + i < nd) v[i] = ld_stream_hint(y + rows[g0 + i] * hc + c, pol);
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    if (g0 + i < nd) {
                        const float w = wts[g0 + i];
                        const uint32_t q[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            acc[2 * h] = __fmaf_rn(w, bf16_lo(q[h]), acc[2 * h]);
                            acc[2 * h + 1] = __fmaf_rn(w, bf16_hi(q[h]), acc[2 * h + 1]);
                        }
                    }
                }
            }
            st_v4(out + t * hc + c, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        }
        __syncwarp();
    }
}

// two e2m1 codes (one byte, element 0 in the low nibble) -> two floats
__device__ __forceinline__ void e2m1x2_to_f32(uint32_t byte, float &lo, float &hi) {
    uint32_t h2;
    asm("{ .reg .b8 t; .reg .b16 s; cvt.u16.u32 s, %1; cvt.u8.u16 t, s; cvt.rn.f16x2.e2m1x2 %0, t; }"
        : "=r"(h2)
        : "r"(byte));
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h; }"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// 2^(code - 127) for an e8m0 code 0..254 (code 0 is the denormal 2^-127)
__device__ __forceinline__ float e8m0_value(uint32_t code) {
    return code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);
}

// Combine over a wire-format receive buffer: as combine_kernel, each lane
// producing 16 output channels per step from the rows' codes and scales.
// Codes are decoded by the hardware converters (e4m3x2 / e2m1x2 -> f16x2,
// exact) and accumulated as fma(w * scale, code value, acc).
template <int LAYOUT, int FMT>
__global__ void __launch_bounds__(kWarps * 32, EP_COMBINE_MINB) combine_wire_kernel(CombineArgs a, const uint8_t *wq,
                                                                                   const void *ws) {
    __shared__ int64_t s_rows[kWarps][32];
    __shared__ float s_w[kWarps][32];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t units = d.T * a.pieces;
    const int64_t qrow = FMT == EP_WIRE_MXFP8 ? d.H : d.H / 2;
    int64_t *rows = s_rows[warp];
    float *wts = s_w[warp];
    constexpr int G = 8;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int nd = gather_sources<LAYOUT>(a, t, t / d.Tr, rows, wts);
        const int64_t hb = p * a.piece_elems, he = min(hb + a.piece_elems, d.H);
        for (int64_t h0 = hb + lane * 16; h0 < he; h0 += 512) {
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
            for (int g0 = 0; g0 < nd; g0 += G) {
                uint4 cq[G];
                float sc[G];
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    if (g0 + i < nd) {
                        const int64_t row = rows[g0 + i];
                        if (FMT == EP_WIRE_MXFP8) {
                            cq[i] = ld_stream(wq + row * qrow + h0);
                            sc[i] = e8m0_value(__ldg(static_cast<const uint8_t *>(ws) + row * (d.H / 32) + h0 / 32));
                        } else {
                            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(wq + row * qrow + h0 / 2));
                            cq[i] = make_uint4(v.x, v.y, 0, 0);
                            sc[i] = __uint_as_float(
                                (uint32_t)__ldg(static_cast<const uint16_t *>(ws) + row * (d.H / 16) + h0 / 16) << 16);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    if (g0 + i < nd) {
                        // weight x block scale once per row: exact for a power-of-two
                        // e8m0 scale; for a bf16 scale one fp32 rounding of w * s
                        const float c = wts[g0 + i] * sc[i];
                        if (FMT == EP_WIRE_MXFP8) {
                            const uint32_t qw[4] = {cq[i].x, cq[i].y, cq[i].z, cq[i].w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                float f0, f1, f2, f3;
                                e4m3x2_to_f32_c((uint16_t)(qw[h] & 0xFFFF), f0, f1);
                                e4m3x2_to_f32_c((uint16_t)(qw[h] >> 16), f2, f3);
                                acc[4 * h] = __fmaf_rn(c, f0, acc[4 * h]);
                                acc[4 * h + 1] = __fmaf_rn(c, f1, acc[4 * h + 1]);
                                acc[4 * h + 2] = __fmaf_rn(c, f2, acc[4 * h + 2]);
                                acc[4 * h + 3] = __fmaf_rn(c, f3, acc[4 * h + 3]);
                            }
                        } else {
                            const uint32_t qw[2] = {cq[i].x, cq[i].y};
#pragma unroll
                            for (int h = 0; h < 8; ++h) {
                                float f0, f1;
                                e2m1x2_to_f32((qw[h >> 2] >> (8 * (h & 3))) & 0xFF, f0, f1);
                                acc[2 * h] = __fmaf_rn(c, f0, acc[2 * h]);
                                acc[2 * h + 1] = __fmaf_rn(c, f1, acc[2 * h + 1]);
                            }
                        }
                    }
                }
            }
            uint4 *op = reinterpret_cast<uint4 *>(a.out + t * d.H + h0);
            st_v4(op, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                                 pack_bf16x2(acc[6], acc[7])));
            st_v4(op + 1, make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                                     pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15])));
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

int combine_grid_cap(int layout) {
    static int cached[64][2] = {{0}};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev][layout])
        cached[dev][layout] = layout == EP_RANK_MAJOR ? grid_cap_for(combine_kernel<EP_RANK_MAJOR>)
                                                      : grid_cap_for(combine_kernel<EP_EXPERT_MAJOR>);
    return cached[dev][layout];
}

cudaError_t launch_combine_wire(int layout, int fmt, const CombineArgs &a, const uint8_t *wq, const void *ws,
                                cudaStream_t st) {
    int64_t grid = (a.d.T * a.pieces + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * 3;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const dim3 g((unsigned)grid), b(kWarps * 32);
    if (layout == EP_RANK_MAJOR) {
        if (fmt == EP_WIRE_MXFP8) combine_wire_kernel<EP_RANK_MAJOR, EP_WIRE_MXFP8><<<g, b, 0, st>>>(a, wq, ws);
        else combine_wire_kernel<EP_RANK_MAJOR, EP_WIRE_NVFP4><<<g, b, 0, st>>>(a, wq, ws);
    } else {
        if (fmt == EP_WIRE_MXFP8) combine_wire_kernel<EP_EXPERT_MAJOR, EP_WIRE_MXFP8><<<g, b, 0, st>>>(a, wq, ws);
        else combine_wire_kernel<EP_EXPERT_MAJOR, EP_WIRE_NVFP4><<<g, b, 0, st>>>(a, wq, ws);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(int layout, const CombineArgs &a, int grid, cudaStream_t st) {
    if (layout == EP_RANK_MAJOR) combine_kernel<EP_RANK_MAJOR><<<grid, kWarps * 32, 0, st>>>(a);
    else combine_kernel<EP_EXPERT_MAJOR><<<grid, kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ep
