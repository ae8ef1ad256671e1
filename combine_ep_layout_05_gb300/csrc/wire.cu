// Casting expert outputs to a low-precision combine wire format.
//
// What ("MoE-EP Benchmark", environment reference, MEGA_COMBINE_DTYPE: the
// cross-rank combine wire format may be mxfp8 - 32 e4m3 values sharing one
// e8m0 scale, 2x less combine traffic - or nvfp4 - 16 e2m1 values with a
// bf16 scale, 4x less): each live receive row y (bf16) is cast once, on the
// expert side, before combine reads it back.
//   mxfp8: per block of 32, X = floor(log2(amax)) - 8 clamped to [-127, 127]
//          (e8m0 code X + 127, 0 when amax = 0); q = e4m3(v * 2^-X),
//          nearest-even, saturating at 448.
//   nvfp4: per block of 16, s = bf16(fp32(amax / 6)); inv = fp32(1 / s)
//          (0 when s = 0); q = e2m1(v * inv), nearest-even, saturating at 6;
//          element 2i in the low nibble.
//
// How: a warp owns a (token, piece) unit and walks the token's receive rows
// from the dispatch handle (as the dispatch does); each lane casts 16
// channels per step (mxfp8: two lanes per block, their amax combined with
// one shuffle; nvfp4: one block per lane).
#include "dispatch_device.cuh"

namespace ep {

namespace {

// 2^e as a float for e in [-127, 127] (2^-127 is a denormal)
__device__ __forceinline__ float exp2i(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// e2m1 code (4 bits) of a float: nearest magnitude among 0, .5, 1, 1.5, 2,
// 3, 4, 6 with ties to the even code, saturating at 6.  The thresholds are
// the midpoints; `>` keeps a tie on the lower (even) code and `>=` moves it
// to the upper (even) one.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
    const float a = fabsf(v);
    const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
                       (a > 5.0f);
    return m | (signbit(v) ? 8u : 0u);
}

template <int LAYOUT, int FMT>
__global__ void __launch_bounds__(kWarps * 32) wire_quant_kernel(DispatchArgs a, const uint16_t *y, uint8_t *wq,
                                                                 void *ws) {
    __shared__ int64_t s_rows[kWarps][kMaxDst];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t *rows = s_rows[warp];
    const int64_t units = d.T * a.pieces;
    const int64_t qrow = FMT == EP_WIRE_MXFP8 ? d.H : d.H / 2;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int nd = gather_dests<LAYOUT>(a, t, t / d.Tr, rows);
        const int64_t hb = p * a.piece_elems, he = min(hb + a.piece_elems, d.H);
        for (int dd = 0; dd < nd; ++dd) {
            const int64_t row = rows[dd];
            for (int64_t h00 = hb; h00 < he; h00 += 512) {
                const int64_t h0 = h00 + lane * 16;
                const bool act = h0 < he;
                uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
                if (act) {
                    const uint4 *yp = reinterpret_cast<const uint4 *>(y + row * d.H + h0);
                    v0 = ld_stream(yp);
                    v1 = ld_stream(yp + 1);
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
                if (FMT == EP_WIRE_MXFP8) {
                    // blocks of 32 = two lanes (h0 is a multiple of 32 on even lanes)
                    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
                    int X = -127;
                    if (amax > 0.f) {
                        // floor(log2 amax) = ex - 127 for a normal amax; a subnormal one
                        // (ex = 0) clamps to -127 below either way
                        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF);
                        X = ex - 127 - 8;
                        if (X < -127) X = -127;
                    }
                    const float sc = exp2i(-X);
                    uint32_t q[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t lo = pack_e4m3x2(__fmul_rn(f[4 * i], sc), __fmul_rn(f[4 * i + 1], sc));
                        const uint32_t hi = pack_e4m3x2(__fmul_rn(f[4 * i + 2], sc), __fmul_rn(f[4 * i + 3], sc));
                        q[i] = lo | (hi << 16);
                    }
                    if (act) {
                        st_v4(wq + row * qrow + h0, make_uint4(q[0], q[1], q[2], q[3]));
                        if ((lane & 1) == 0) static_cast<uint8_t *>(ws)[row * (d.H / 32) + h0 / 32] = (uint8_t)(X + 127);
                    }
                } else {
                    const float s32 = __fdiv_rn(amax, 6.0f);
                    const uint32_t sb = pack_bf16x2(s32, 0.f) & 0xFFFFu;
                    const float sf = __uint_as_float(sb << 16);
                    const float inv = sf > 0.f ? __fdiv_rn(1.0f, sf) : 0.f;
                    uint32_t q0 = 0, q1 = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) q0 |= e2m1_code(__fmul_rn(f[i], inv)) << (4 * i);
#pragma unroll
                    for (int i = 0; i < 8; ++i) q1 |= e2m1_code(__fmul_rn(f[8 + i], inv)) << (4 * i);
                    if (act) {
                        *reinterpret_cast<uint2 *>(wq + row * qrow + h0 / 2) = make_uint2(q0, q1);
                        static_cast<uint16_t *>(ws)[row * (d.H / 16) + h0 / 16] = (uint16_t)sb;
                    }
                }
            }
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_wire_quant(int layout, int fmt, const DispatchArgs &a, const uint16_t *y, uint8_t *wq, void *ws,
                              cudaStream_t st) {
    int64_t grid = (a.d.T * a.pieces + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const dim3 g((unsigned)grid), b(kWarps * 32);
    if (layout == EP_RANK_MAJOR) {
        if (fmt == EP_WIRE_MXFP8) wire_quant_kernel<EP_RANK_MAJOR, EP_WIRE_MXFP8><<<g, b, 0, st>>>(a, y, wq, ws);
        else wire_quant_kernel<EP_RANK_MAJOR, EP_WIRE_NVFP4><<<g, b, 0, st>>>(a, y, wq, ws);
    } else {
        if (fmt == EP_WIRE_MXFP8) wire_quant_kernel<EP_EXPERT_MAJOR, EP_WIRE_MXFP8><<<g, b, 0, st>>>(a, y, wq, ws);
        else wire_quant_kernel<EP_EXPERT_MAJOR, EP_WIRE_NVFP4><<<g, b, 0, st>>>(a, y, wq, ws);
    }
    return cudaGetLastError();
}

}  // namespace ep
