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
//          element 2i in the low nibble.  Defined for finite values (e2m1
//          has no infinity or NaN).
//
// How: a warp owns a (token, piece) unit and walks the token's receive rows
// from the dispatch handle (as the dispatch does); each lane casts 16
// channels per step (mxfp8: two lanes per block, their amax combined with
// one shuffle; nvfp4: one block per lane).
#include "dispatch_device.cuh"
#include "vec8.cuh"

namespace ep {

namespace {

// 2^e as a float for e in [-127, 127] (2^-127 is a denormal)
__device__ __forceinline__ float exp2i(int e) {
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// two e2m1 codes in one byte (lo in the low nibble): the hardware
// conversion, nearest-even, saturating at 6
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The nvfp4 block scale s = bf16(fp32(amax / 6)) and inv = fp32(1 / s)
// without a division per block.  A correctly rounded quotient and the bf16
// rounding both commute with scaling by a power of two while the values stay
// normal, so with amax = 2^e * (1 + i/128) (a bf16 value: 7 mantissa bits)
// s = 2^e * bf16(fp32((1 + i/128) / 6)), and with s = 2^f * (1 + j/128)
// inv = 2^-f * fp32(1 / (1 + j/128)).  The two 128-entry tables hold those
// quotients, filled once per CTA by correctly rounded divisions.  Zero,
// non-finite and tiny amax (below 2^-123, where s would be subnormal) take
// the divisions themselves.
struct Nvfp4Tables {
    uint16_t s[128];   // bf16 bits of fp32((1 + i/128) / 6)
    uint32_t r[128];   // fp32 bits of 1 / (1 + j/128)
};

__device__ __forceinline__ void nvfp4_tables_fill(Nvfp4Tables &tb) {
    if (threadIdx.x < 128) {
        const float m = 1.0f + (float)threadIdx.x * (1.0f / 128.0f);
        tb.s[threadIdx.x] = (uint16_t)(pack_bf16x2(__fdiv_rn(m, 6.0f), 0.f) & 0xFFFFu);
        tb.r[threadIdx.x] = __float_as_uint(__fdiv_rn(1.0f, m));
    }
}

__device__ __forceinline__ void nvfp4_scale(const Nvfp4Tables &tb, float amax, uint32_t &sb, float &inv) {
    const uint32_t ab = __float_as_uint(amax);
    const int ex = (int)(ab >> 23);
    if (ex >= 4 && ex <= 254) {
        sb = (uint32_t)((int)tb.s[(ab >> 16) & 0x7F] + (ex - 127) * 128);
        const int es = (int)((sb >> 7) & 0xFF);
        inv = __uint_as_float((uint32_t)((int)tb.r[sb & 0x7F] - (es - 127) * (1 << 23)));
    } else {
        const float s32 = __fdiv_rn(amax, 6.0f);
        sb = pack_bf16x2(s32, 0.f) & 0xFFFFu;
        const float sf = __uint_as_float(sb << 16);
        inv = sf > 0.f ? __fdiv_rn(1.0f, sf) : 0.f;
    }
}

#ifndef EP_WIRE_QG
#define EP_WIRE_QG 4   // rows per batch: their loads are issued back to back
#endif

// Casts one lane's 16 channels (v0, v1: bf16) of one row at channel h0.
// Warp-collective (the mxfp8 block maximum is shared by two lanes): every
// lane calls it, `act` says whether this lane's channels exist.
template <int FMT>
__device__ __forceinline__ void cast_chunk(const Nvfp4Tables &tb, uint4 v0, uint4 v1, int64_t row, int64_t h0,
                                           bool act, int64_t H, uint8_t *wq, void *ws) {
    const int64_t qrow = FMT == EP_WIRE_MXFP8 ? H : H / 2;
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
            if ((threadIdx.x & 1) == 0) static_cast<uint8_t *>(ws)[row * (H / 32) + h0 / 32] = (uint8_t)(X + 127);
        }
    } else {
        uint32_t sb;
        float inv;
        nvfp4_scale(tb, amax, sb, inv);
        uint32_t q0 = 0, q1 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q0 |= e2m1x2(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv)) << (8 * i);
            q1 |= e2m1x2(__fmul_rn(f[8 + 2 * i], inv), __fmul_rn(f[8 + 2 * i + 1], inv)) << (8 * i);
        }
        if (act) {
            *reinterpret_cast<uint2 *>(wq + row * qrow + h0 / 2) = make_uint2(q0, q1);
            static_cast<uint16_t *>(ws)[row * (H / 16) + h0 / 16] = (uint16_t)sb;
        }
    }
}

template <int LAYOUT, int FMT, bool WIDE>
__global__ void __launch_bounds__(kWarps * 32) wire_quant_kernel(DispatchArgs a, const uint16_t *y, uint8_t *wq,
                                                                 void *ws) {
    __shared__ int64_t s_rows[kWarps][kMaxDst];
    __shared__ Nvfp4Tables s_tb;
    if (FMT == EP_WIRE_NVFP4) {
        nvfp4_tables_fill(s_tb);
        __syncthreads();
    }
    constexpr int G = EP_WIRE_QG;
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t *rows = s_rows[warp];
    const int64_t units = d.T * a.pieces;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int nd = gather_dests<LAYOUT>(a, t, t / d.Tr, rows);
        const int64_t hb = p * a.piece_elems, he = min(hb + a.piece_elems, d.H);
        for (int g0 = 0; g0 < nd; g0 += G) {
            for (int64_t h00 = hb; h00 < he; h00 += 512) {
                const int64_t h0 = h00 + lane * 16;
                const bool act = h0 < he;
                uint4 v[G][2];
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    v[i][0] = make_uint4(0, 0, 0, 0);
                    v[i][1] = v[i][0];
                    if (g0 + i < nd && act) {
                        if (WIDE) {   // one 32-byte load
                            uint32_t r[8];
                            ld_stream8(y + rows[g0 + i] * d.H + h0, r);
                            v[i][0] = make_uint4(r[0], r[1], r[2], r[3]);
                            v[i][1] = make_uint4(r[4], r[5], r[6], r[7]);
                        } else {
                            const uint4 *yp = reinterpret_cast<const uint4 *>(y + rows[g0 + i] * d.H + h0);
                            v[i][0] = ld_stream(yp);
                            v[i][1] = ld_stream(yp + 1);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if (g0 + i < nd) cast_chunk<FMT>(s_tb, v[i][0], v[i][1], rows[g0 + i], h0, act, d.H, wq, ws);
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
    // 32-byte loads of a lane's 16 channels where y allows them
    const bool wide = a.d.H % 16 == 0 && a.piece_elems % 16 == 0 && ((uintptr_t)y & 31) == 0;
    if (layout == EP_RANK_MAJOR) {
        if (fmt == EP_WIRE_MXFP8)
            wide ? wire_quant_kernel<EP_RANK_MAJOR, EP_WIRE_MXFP8, true><<<g, b, 0, st>>>(a, y, wq, ws)
                 : wire_quant_kernel<EP_RANK_MAJOR, EP_WIRE_MXFP8, false><<<g, b, 0, st>>>(a, y, wq, ws);
        else
            wide ? wire_quant_kernel<EP_RANK_MAJOR, EP_WIRE_NVFP4, true><<<g, b, 0, st>>>(a, y, wq, ws)
                 : wire_quant_kernel<EP_RANK_MAJOR, EP_WIRE_NVFP4, false><<<g, b, 0, st>>>(a, y, wq, ws);
    } else {
        if (fmt == EP_WIRE_MXFP8)
            wide ? wire_quant_kernel<EP_EXPERT_MAJOR, EP_WIRE_MXFP8, true><<<g, b, 0, st>>>(a, y, wq, ws)
                 : wire_quant_kernel<EP_EXPERT_MAJOR, EP_WIRE_MXFP8, false><<<g, b, 0, st>>>(a, y, wq, ws);
        else
            wide ? wire_quant_kernel<EP_EXPERT_MAJOR, EP_WIRE_NVFP4, true><<<g, b, 0, st>>>(a, y, wq, ws)
                 : wire_quant_kernel<EP_EXPERT_MAJOR, EP_WIRE_NVFP4, false><<<g, b, 0, st>>>(a, y, wq, ws);
    }
    return cudaGetLastError();
}

}  // namespace ep
