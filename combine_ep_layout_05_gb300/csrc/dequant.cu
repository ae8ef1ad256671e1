// Identity expert for an FP8 receive buffer (test and benchmark harness):
// the expert output equals its input, y = bf16(decode(q) * s), the exact
// product rounded once to nearest-even.  Only the rows the dispatch handle
// names are written (as ep_dispatch writes them).
#include "dispatch_device.cuh"
#include "vec8.cuh"

namespace ep {

namespace {

#ifndef EP_DEQ_G
#define EP_DEQ_G 8   // rows per batch
#endif
#ifndef EP_DEQ_U
#define EP_DEQ_U 1   // 16-channel chunks per lane and row
#endif
#ifndef EP_DEQ_V8
#define EP_DEQ_V8 1  // 32-byte stores of a lane's 16 bf16 channels
#endif

// v * s rounded to odd in fp32: the product truncated toward zero, its last
// bit set when the truncation dropped anything (the fma remainder is then
// nonzero).  With 16 more bits than bf16, rounding this to nearest-even bf16
// gives the nearest-even bf16 of the exact product (round-to-odd then
// round-to-nearest, Boldo and Melquiond, "Emulation of FMA and correctly
// rounded sums: proved algorithms using rounding to odd", 2008): one
// rounding of a product that needs up to 28 significant bits.
__device__ __forceinline__ float fmul_odd(float v, float s) {
    const float hz = __fmul_rz(v, s);
    const float r = __fmaf_rn(v, s, -hz);
    return __uint_as_float(__float_as_uint(hz) | (r != 0.f ? 1u : 0u));
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
// still spread over the GPU.  A lane handles EP_DEQ_U 16-channel chunks
// (512 channels apart) of EP_DEQ_G rows at a time: their loads are issued
// back to back, then each chunk is converted and stored.
template <int LAYOUT, bool V8>
__global__ void __launch_bounds__(kWarps * 32) dequant_kernel(DispatchArgs a, uint16_t *y) {
    __shared__ int64_t s_rows[kWarps][kMaxDst];
    constexpr int G = EP_DEQ_G, U = EP_DEQ_U;
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
        for (int g0 = 0; g0 < nd; g0 += G) {
            for (int64_t h00 = hb + (int64_t)lane * 16; h00 < he; h00 += 512 * U) {
                uint4 qv[G][U];
                float sc[G][U];
#pragma unroll
                for (int i = 0; i < G; ++i) {
#pragma unroll
                    for (int x = 0; x < U; ++x) {
                        const int64_t h0 = h00 + 512 * x;
                        if (g0 + i < nd && h0 < he) {
                            const int64_t row = rows[g0 + i];
                            qv[i][x] = ld_stream(q + row * d.H + h0);
                            sc[i][x] = a.recv_scales[row * nb + h0 / 128];
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < G; ++i) {
#pragma unroll
                    for (int x = 0; x < U; ++x) {
                        const int64_t h0 = h00 + 512 * x;
                        if (g0 + i >= nd || h0 >= he) continue;
                        const uint32_t qw[4] = {qv[i][x].x, qv[i][x].y, qv[i][x].z, qv[i][x].w};
                        const float s = sc[i][x];
                        uint32_t o[8];
#pragma unroll
                        for (int i2 = 0; i2 < 4; ++i2) {
                            float f0, f1, f2, f3;
                            e4m3x2_to_f32((uint16_t)(qw[i2] & 0xFFFF), f0, f1);
                            e4m3x2_to_f32((uint16_t)(qw[i2] >> 16), f2, f3);
                            o[2 * i2] = pack_bf16x2(fmul_odd(f0, s), fmul_odd(f1, s));
                            o[2 * i2 + 1] = pack_bf16x2(fmul_odd(f2, s), fmul_odd(f3, s));
                        }
                        uint16_t *yr = y + rows[g0 + i] * d.H + h0;
                        if (V8) {
                            st_v8(yr, o);
                        } else {
                            uint4 *yp = reinterpret_cast<uint4 *>(yr);
                            st_v4(yp, make_uint4(o[0], o[1], o[2], o[3]));
                            st_v4(yp + 1, make_uint4(o[4], o[5], o[6], o[7]));
                        }
                    }
                }
            }
        }
        __syncwarp();
    }
}

}  // namespace

namespace {

// Resident CTAs of the dequant kernel on this device (per layout, 32-byte
// stores or not).
int dequant_cap(int layout, bool v8) {
    static std::atomic<int> cache[4][kCacheDevices];
    return cached_per_device(cache[layout * 2 + (v8 ? 1 : 0)], [&](int) {
        auto occ = [](auto kernel) {
            int blocks = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, kWarps * 32, 0) != cudaSuccess ||
                blocks < 1)
                blocks = 1;
            return blocks * num_sms();
        };
        if (layout == EP_RANK_MAJOR)
            return v8 ? occ(dequant_kernel<EP_RANK_MAJOR, true>) : occ(dequant_kernel<EP_RANK_MAJOR, false>);
        return v8 ? occ(dequant_kernel<EP_EXPERT_MAJOR, true>) : occ(dequant_kernel<EP_EXPERT_MAJOR, false>);
    });
}

}  // namespace

// Splits rows into pieces of 512-channel multiples.  Fewer tokens than
// resident warps: each warp takes (token, piece) units in rounds, a unit
// costing about one memory round trip per 512-channel step plus one for its
// routing entry, and the split minimises rounds x cost per unit, ties going
// to more (shorter) units (8 x 128 tokens, expert-major, 8192 rows: 7
// pieces, 31.5 us, against 5 pieces and 33.7 us with a fixed target of
// 32 units per SM).  More tokens: whole rows, or halves below 32 tokens per
// SM.  The grid is up to 8 CTAs per SM, more than are resident, so CTAs
// that start late take the place of those that finish early (a persistent
// grid of resident CTAs was 7% slower at 4096 tokens/rank: static rounds
// left a longer tail).
void plan_dequant(int layout, DispatchArgs &a, bool v8, int &grid) {
    const Dims &d = a.d;
    const int64_t warps = (int64_t)dequant_cap(layout, v8) * kWarps;
    const int64_t max_pieces = (d.H + 511) / 512;
    a.pieces = 1;
    a.piece_elems = d.H;
    if (d.T > 0 && d.T < warps) {
        int64_t best = -1;
        for (int64_t p = 1; p <= max_pieces; ++p) {
            int64_t per = (d.H + p - 1) / p;
            per = (per + 511) / 512 * 512;
            const int64_t pp = (d.H + per - 1) / per;
            if (pp != p) continue;
            const int64_t rounds = (d.T * pp + warps - 1) / warps;
            const int64_t cost = rounds * ((per + 511) / 512 + 1);
            if (best < 0 || cost <= best) {
                best = cost;
                a.pieces = pp;
                a.piece_elems = per;
            }
        }
    } else if (d.T > 0 && d.T < (int64_t)num_sms() * 32 && max_pieces >= 2) {
        a.piece_elems = ((d.H + 1) / 2 + 511) / 512 * 512;
        a.pieces = (d.H + a.piece_elems - 1) / a.piece_elems;
    }
    int64_t g = (d.T * a.pieces + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * 8;
    grid = (int)(g < 1 ? 1 : g > cap ? cap : g);
}

cudaError_t launch_dequant(int layout, const DispatchArgs &a0, uint16_t *y, cudaStream_t st) {
    // 32-byte stores when y is 32-byte aligned (rows are: H % 128 == 0)
    const bool v8 = EP_DEQ_V8 && ((uintptr_t)y & 31) == 0;
    DispatchArgs a = a0;   // the row split is chosen here
    int grid = 1;
    plan_dequant(layout, a, v8, grid);
    const unsigned g = (unsigned)grid, b = kWarps * 32;
    if (layout == EP_RANK_MAJOR) {
        if (v8) dequant_kernel<EP_RANK_MAJOR, true><<<g, b, 0, st>>>(a, y);
        else dequant_kernel<EP_RANK_MAJOR, false><<<g, b, 0, st>>>(a, y);
    } else {
        if (v8) dequant_kernel<EP_EXPERT_MAJOR, true><<<g, b, 0, st>>>(a, y);
        else dequant_kernel<EP_EXPERT_MAJOR, false><<<g, b, 0, st>>>(a, y);
    }
    return cudaGetLastError();
}

}  // namespace ep
