// Combine from a low-precision wire format: the weighted top-k gather of
// ep_combine reading each receive row as mxfp8 (32 e4m3 codes and one
// e8m0 scale per block) or nvfp4 (16 e2m1 codes and one bf16 scale per
// block) and decoding it on the fly ("MoE-EP Benchmark", environment
// reference, MEGA_COMBINE_DTYPE).
#include "combine_device.cuh"

namespace ep {

namespace {

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
    // rows in flight per lane (nvfp4: 6, which keeps the kernel within its
    // register budget of three CTAs per SM without spilling)
    constexpr int G = FMT == EP_WIRE_MXFP8 ? 8 : 6;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int nd = gather_sources<LAYOUT>(a, t, t / d.Tr, rows, wts);
        const int64_t hb = p * a.piece_elems, he = min(hb + a.piece_elems, d.H);
        for (int64_t h0 = hb + lane * 16; h0 < he; h0 += 512) {
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.f;
            for (int g0 = 0; g0 < nd; g0 += G) {
                constexpr int NW = FMT == EP_WIRE_MXFP8 ? 4 : 2;   // code words per lane and row
                uint32_t cq[G][NW];
                float sc[G];
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    if (g0 + i < nd) {
                        const int64_t row = rows[g0 + i];
                        if (FMT == EP_WIRE_MXFP8) {
                            const uint4 v = ld_stream(wq + row * qrow + h0);
                            cq[i][0] = v.x;
                            cq[i][1] = v.y;
                            cq[i][NW - 2] = v.z;
                            cq[i][NW - 1] = v.w;
                            sc[i] = e8m0_value(__ldg(static_cast<const uint8_t *>(ws) + row * (d.H / 32) + h0 / 32));
                        } else {
                            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(wq + row * qrow + h0 / 2));
                            cq[i][0] = v.x;
                            cq[i][1] = v.y;
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
#pragma unroll
                            for (int h = 0; h < NW; ++h) {
                                const float2 f01 = e4m3x2_to_f32x2((uint16_t)(cq[i][h] & 0xFFFF));
                                const float2 f23 = e4m3x2_to_f32x2((uint16_t)(cq[i][h] >> 16));
                                acc[4 * h] = __fmaf_rn(c, f01.x, acc[4 * h]);
                                acc[4 * h + 1] = __fmaf_rn(c, f01.y, acc[4 * h + 1]);
                                acc[4 * h + 2] = __fmaf_rn(c, f23.x, acc[4 * h + 2]);
                                acc[4 * h + 3] = __fmaf_rn(c, f23.y, acc[4 * h + 3]);
                            }
                        } else {
#pragma unroll
                            for (int v = 0; v < NW; ++v) {
                                uint32_t hp[4];
                                e2m1x8_to_f16x2(cq[i][v], hp);
#pragma unroll
                                for (int b = 0; b < 4; ++b) {
                                    const float2 f = f16x2_to_f32x2(hp[b]);
                                    acc[8 * v + 2 * b] = __fmaf_rn(c, f.x, acc[8 * v + 2 * b]);
                                    acc[8 * v + 2 * b + 1] = __fmaf_rn(c, f.y, acc[8 * v + 2 * b + 1]);
                                }
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

// Staged wire combine: the same sums as combine_wire_kernel, with the row
// loads decoupled from the decode.  A warp walks a flat sequence of steps
// (unit, channel step, group of up to ROWS rows); for each step every lane
// copies its 16 code bytes of each row (and the rows' block scales) into a
// per-warp ring of S shared-memory stages with cp.async, and the warp
// decodes the step issued S - 1 steps earlier.  The copies of later steps,
// including those of the warp's next unit, stay in flight while it decodes.
// A lane decodes the bytes it copied itself; the mxfp8 scale words are
// copied by lanes 0-3 and read by all lanes after cp.async.wait_group and a
// warp barrier.  Nothing waits on another warp or CTA.  Pairs of channels
// are accumulated with packed fp32 FMAs (each half rounded as one fmaf), so
// the sums are bit-identical to combine_wire_kernel's.
//   mxfp8: 16 channels (16 code bytes) per lane, 512 per warp step, the
//          step's 16 e8m0 scale bytes per row.  Needs H % 128 == 0 (whole
//          4-byte scale words per row).
//   nvfp4: 32 channels (16 code bytes) per lane, 1024 per warp step, two
//          bf16 block scales per lane and row.  Needs H % 32 == 0.
// Warps per CTA, stages per warp and rows per step (one CTA per SM: the
// stages fill shared memory).  Measured on GB300 (rank-major, 5.3 rows per
// token): more warps beat deeper rings.  mxfp8 with 20 warps: 287 us at
// 4096 tokens/rank, 86 us at 1024; with 24, 285 and 100 us (fewer units per
// warp leave a longer tail); 26 warps of 6-row steps: 327 us.  nvfp4,
// register-bound at 20 warps: 225.5 us at 4096 tokens/rank with 8-row steps,
// 217.0 us with 6 (fewer predicated row slots per step; the few tokens of 7
// or 8 rows take a second group).  Expert-major tokens always have k rows,
// so they keep 8-row steps.
#ifndef EP_WIRE_MX_WARPS
#define EP_WIRE_MX_WARPS 20
#endif
#ifndef EP_WIRE_MX_STAGES
#define EP_WIRE_MX_STAGES 2
#endif
#ifndef EP_WIRE_NV_WARPS
#define EP_WIRE_NV_WARPS 20
#endif
#ifndef EP_WIRE_NV_STAGES
#define EP_WIRE_NV_STAGES 2
#endif
#ifndef EP_WIRE_NV_RANK_ROWS
#define EP_WIRE_NV_RANK_ROWS 6
#endif
#ifndef EP_WIRE_STAGED
#define EP_WIRE_STAGED 1
#endif

struct WireUnit {   // one (token, piece) unit's rows and weights
    int64_t rows[32];
    float w[32];
    int nd;
    int pad[3];
};

template <int LAYOUT, int FMT>
struct WireStaging {
    // rows per step
    static constexpr int ROWS = FMT == EP_WIRE_NVFP4 && LAYOUT == EP_RANK_MAJOR ? EP_WIRE_NV_RANK_ROWS : 8;
    static constexpr int W = FMT == EP_WIRE_MXFP8 ? EP_WIRE_MX_WARPS : EP_WIRE_NV_WARPS;
    static constexpr int S = FMT == EP_WIRE_MXFP8 ? EP_WIRE_MX_STAGES : EP_WIRE_NV_STAGES;
    // unit descriptors in flight: the S steps between the consumer and the
    // producer can span S units, plus the one the producer enters
    static constexpr int US = S + 1;
    static constexpr int CH = FMT == EP_WIRE_MXFP8 ? 16 : 32;     // channels per lane and step
    static constexpr int SPAN = 32 * CH;                            // channels per warp step
    static constexpr int SCW = FMT == EP_WIRE_MXFP8 ? 4 : 32;      // scale words per row and step
    static constexpr size_t kData = (size_t)S * ROWS * 32 * 16;
    static constexpr size_t kScale = (size_t)S * ROWS * SCW * 4;
    static constexpr size_t kUnits = (size_t)US * sizeof(WireUnit);
    static constexpr size_t kWarpBytes = kData + kScale + kUnits;
};

__device__ __forceinline__ uint32_t sh_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sh_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sh_addr(dst)), "l"(src) : "memory");
}

// the same, to a shared-memory address already converted to the shared window
__device__ __forceinline__ void cp_async16_sh(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async4_sh(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Position of a warp in its step sequence.
struct WireCursor {
    int64_t u;       // unit = token * pieces + piece
    int it, g;       // channel step within the unit's piece, row group
    int slot, nd;    // unit ring slot, rows of the unit
    int64_t hb, he;  // the unit's channel range
    int64_t t;       // the unit's token
};

__device__ __forceinline__ void wire_cursor_unit(const CombineArgs &a, WireCursor &c) {
    c.t = a.pieces == 1 ? c.u : c.u / a.pieces;   // no division for whole rows
    const int64_t p = c.u - c.t * a.pieces;
    c.hb = p * a.piece_elems;
    c.he = min(c.hb + a.piece_elems, a.d.H);
}

// moves to the next step; returns true when that step starts a new unit
template <int LAYOUT, int FMT>
__device__ __forceinline__ bool wire_cursor_next(const CombineArgs &a, WireCursor &c, int64_t stride) {
    using SG = WireStaging<LAYOUT, FMT>;
    const int ng = c.nd > SG::ROWS ? (c.nd + SG::ROWS - 1) / SG::ROWS : 1;
    if (++c.g < ng) return false;
    c.g = 0;
    if (c.hb + (int64_t)(c.it + 1) * SG::SPAN < c.he) {
        ++c.it;
        return false;
    }
    c.it = 0;
    c.u += stride;
    c.slot = c.slot + 1 == SG::US ? 0 : c.slot + 1;
    wire_cursor_unit(a, c);
    return true;
}

template <int LAYOUT, int FMT>
__global__ void __launch_bounds__(WireStaging<LAYOUT, FMT>::W * 32, 1)
    combine_wire_staged_kernel(CombineArgs a, const uint8_t *wq, const uint8_t *ws) {
    using SG = WireStaging<LAYOUT, FMT>;
    constexpr int CH = SG::CH, SPAN = SG::SPAN, SCW = SG::SCW, S = SG::S, W = SG::W, kWireRows = SG::ROWS;
    extern __shared__ __align__(16) unsigned char smem[];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char *base = smem + (size_t)warp * SG::kWarpBytes;
    uint4 *s_data = reinterpret_cast<uint4 *>(base);                                   // [S][rows][32]
    uint32_t *s_scale = reinterpret_cast<uint32_t *>(base + SG::kData);                // [S][rows][SCW]
    WireUnit *s_unit = reinterpret_cast<WireUnit *>(base + SG::kData + SG::kScale);    // [S + 1]
    const int64_t units = d.T * a.pieces;
    const int64_t stride = (int64_t)gridDim.x * W;
    const int64_t qrow = FMT == EP_WIRE_MXFP8 ? d.H : d.H / 2;

    // the warp-wide gather of a unit's rows and weights into its ring slot
    // the warp-wide gather of a unit's rows and weights into its ring slot;
    // each row index is turned into the byte offset of the row's codes (its
    // scales sit at that offset >> kScaleShift: mxfp8 H/32 scale bytes per
    // H code bytes, nvfp4 H/8 per H/2)
    constexpr int kScaleShift = FMT == EP_WIRE_MXFP8 ? 5 : 2;
    auto enter = [&](WireCursor &c) {
        if (c.u >= units) return;
        WireUnit &U = s_unit[c.slot];
        c.nd = gather_sources<LAYOUT>(a, c.t, c.t / d.Tr, U.rows, U.w);
        __syncwarp();
        if (lane < c.nd) U.rows[lane] *= qrow;
        if (lane == 0) U.nd = c.nd;
        __syncwarp();
    };
    // this lane's ring addresses: stage s, row j of a step at
    // s_lane + (s * kWireRows + j) * 512 (16 code bytes per lane), its scale
    // word at c_lane + (s * kWireRows + j) * SCW * 4
    const uint32_t s_lane = sh_addr(s_data) + lane * 16;
    const uint32_t c_lane = sh_addr(s_scale) + (FMT == EP_WIRE_MXFP8 ? (lane & 3) : lane) * 4;

    WireCursor P{(int64_t)blockIdx.x * W + warp, 0, 0, 0, 0, 0, 0, 0};
    wire_cursor_unit(a, P);
    enter(P);
    WireCursor C = P;
    int ps = 0, cs = 0;   // producer / consumer step counters (stage = count % S)

    auto issue = [&]() {
        if (P.u < units) {
            const WireUnit &U = s_unit[P.slot];
            const int stage = ps % S;
            const int64_t hs = P.hb + (int64_t)P.it * SPAN;   // first channel of the step
            const int64_t h0 = hs + lane * CH;
            const int i0 = P.g * kWireRows;
            const int n = min(kWireRows, P.nd - i0);
            // this lane's code bytes and scale word within a row, and whether
            // it copies them (lanes past the piece's end do not; mxfp8: lanes
            // 0-3 copy the step's 16 scale bytes)
            const int64_t qo = FMT == EP_WIRE_MXFP8 ? h0 : h0 / 2;
            const int64_t so = FMT == EP_WIRE_MXFP8 ? hs / 32 + 4 * lane : h0 / 8;
            const bool qon = h0 < P.he;
            const bool son = FMT == EP_WIRE_MXFP8 ? lane < 4 && hs / 32 + 4 * lane < P.he / 32 : qon;
            const uint32_t sd = s_lane + (uint32_t)stage * kWireRows * 512;
            const uint32_t sc = c_lane + (uint32_t)stage * kWireRows * SCW * 4;
#pragma unroll
            for (int j = 0; j < kWireRows; ++j) {
                if (j < n) {
                    const int64_t ro = U.rows[i0 + j];   // byte offset of the row's codes
                    if (qon) cp_async16_sh(sd + j * 512, wq + ro + qo);
                    if (son) cp_async4_sh(sc + j * SCW * 4, ws + (ro >> kScaleShift) + so);
                }
            }
        }
        cp_async_commit();
        ++ps;
        if (P.u < units && wire_cursor_next<LAYOUT, FMT>(a, P, stride)) enter(P);
    };

    for (int s = 0; s < S - 1; ++s) issue();

    float2 acc[CH / 2];   // channel pairs
    const int mx_shift = 8 * ((lane >> 1) & 3);   // mxfp8: this lane's scale byte within its word
    while (C.u < units) {
        issue();
        cp_async_wait<S - 1>();
        __syncwarp();
        const WireUnit &U = s_unit[C.slot];
        const int stage = cs % S;
        const int64_t hs = C.hb + (int64_t)C.it * SPAN;
        const int64_t h0 = hs + lane * CH;
        const int i0 = C.g * kWireRows;
        const int n = min(kWireRows, C.nd - i0);
        const int ng = C.nd > kWireRows ? (C.nd + kWireRows - 1) / kWireRows : 1;
        if (C.g == 0) {
#pragma unroll
            for (int i = 0; i < CH / 2; ++i) acc[i] = make_float2(0.f, 0.f);
        }
        if (h0 < C.he) {
            // this stage's rows: codes at qs[i * 32], the lane's scale word at ss[i * SCW]
            const uint4 *qs = s_data + stage * kWireRows * 32 + lane;
            const uint32_t *ss = s_scale + stage * kWireRows * SCW + (FMT == EP_WIRE_MXFP8 ? lane >> 3 : lane);
#pragma unroll
            for (int i = 0; i < kWireRows; ++i) {
                if (i < n) {
                    const float w = U.w[i0 + i];
                    const uint4 q = qs[i * 32];
                    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
                    if (FMT == EP_WIRE_MXFP8) {
                        // block of this lane's 16 channels: byte lane / 2 of the step's scales
                        const uint32_t code = (ss[i * SCW] >> mx_shift) & 0xFF;
                        const float c = w * e8m0_value(code);
                        const float2 c2 = make_float2(c, c);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            acc[2 * h] = __ffma2_rn(c2, e4m3x2_to_f32x2((uint16_t)(qw[h] & 0xFFFF)), acc[2 * h]);
                            acc[2 * h + 1] = __ffma2_rn(c2, e4m3x2_to_f32x2((uint16_t)(qw[h] >> 16)), acc[2 * h + 1]);
                        }
                    } else {
                        // channels 0-15 use the low bf16 scale, 16-31 the high one
                        const uint32_t sw = ss[i * SCW];
                        const float s0 = w * bf16_lo(sw), s1 = w * bf16_hi(sw);
                        const float2 c0 = make_float2(s0, s0), c1 = make_float2(s1, s1);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t hp[4];
                            e2m1x8_to_f16x2(qw[v], hp);
#pragma unroll
                            for (int b = 0; b < 4; ++b)
                                acc[4 * v + b] = __ffma2_rn(v < 2 ? c0 : c1, f16x2_to_f32x2(hp[b]), acc[4 * v + b]);
                        }
                    }
                }
            }
            if (C.g == ng - 1) {
                uint4 *op = reinterpret_cast<uint4 *>(a.out + C.t * d.H + h0);
#pragma unroll
                for (int v = 0; v < CH / 8; ++v)
                    st_v4(op + v, make_uint4(pack_bf16x2(acc[4 * v].x, acc[4 * v].y),
                                             pack_bf16x2(acc[4 * v + 1].x, acc[4 * v + 1].y),
                                             pack_bf16x2(acc[4 * v + 2].x, acc[4 * v + 2].y),
                                             pack_bf16x2(acc[4 * v + 3].x, acc[4 * v + 3].y)));
            }
        }
        __syncwarp();   // every lane is done with this stage before it is refilled
        ++cs;
        if (wire_cursor_next<LAYOUT, FMT>(a, C, stride) && C.u < units) C.nd = s_unit[C.slot].nd;
    }
    cp_async_wait<0>();
}

template <int LAYOUT, int FMT>
cudaError_t launch_wire_staged(const CombineArgs &a0, const uint8_t *wq, const void *ws, cudaStream_t st) {
    using SG = WireStaging<LAYOUT, FMT>;
    const size_t smem = SG::kWarpBytes * SG::W;
    auto kern = combine_wire_staged_kernel<LAYOUT, FMT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e) return e;
    // pieces of whole warp steps, enough units to give every warp work
    CombineArgs a = a0;
    const Dims &d = a.d;
    const int64_t want_units = (int64_t)num_sms() * SG::W;
    const int64_t max_pieces = (d.H + SG::SPAN - 1) / SG::SPAN;
    int64_t pieces = (want_units + d.T - 1) / d.T;
    if (pieces > max_pieces) pieces = max_pieces;
    if (pieces < 1) pieces = 1;
    int64_t per = (d.H + pieces - 1) / pieces;
    per = (per + SG::SPAN - 1) / SG::SPAN * SG::SPAN;
    a.piece_elems = per;
    a.pieces = (d.H + per - 1) / per;
    int64_t grid = (d.T * a.pieces + SG::W - 1) / SG::W;
    if (grid > num_sms()) grid = num_sms();
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, SG::W * 32, smem, st>>>(a, wq, static_cast<const uint8_t *>(ws));
    return cudaGetLastError();
}

#ifndef EP_WIRE_FILL
#define EP_WIRE_FILL 10
#endif
template <int FMT>
bool staged_fills(const Dims &d) {
    using SG = WireStaging<EP_RANK_MAJOR, FMT>;
    return d.T * ((d.H + SG::SPAN - 1) / SG::SPAN) >= (int64_t)EP_WIRE_FILL * num_sms() * SG::W;
}

}  // namespace

cudaError_t launch_combine_wire(int layout, int fmt, const CombineArgs &a, const uint8_t *wq, const void *ws,
                                cudaStream_t st) {
    // the staged kernel where its aligned scale-word copies apply and there
    // are units for ten rounds of every warp of a full grid (measured: at
    // 2048 tokens and fewer the unstaged kernel, whose 8-warp CTAs spread
    // over more SMs, is faster; at 8192 the staged one)
    const bool ws4 = EP_WIRE_STAGED && ((uintptr_t)ws & 3) == 0;
    if (fmt == EP_WIRE_MXFP8 && a.d.H % 128 == 0 && ws4 && staged_fills<EP_WIRE_MXFP8>(a.d))
        return layout == EP_RANK_MAJOR ? launch_wire_staged<EP_RANK_MAJOR, EP_WIRE_MXFP8>(a, wq, ws, st)
                                       : launch_wire_staged<EP_EXPERT_MAJOR, EP_WIRE_MXFP8>(a, wq, ws, st);
    if (fmt == EP_WIRE_NVFP4 && a.d.H % 32 == 0 && ws4 && staged_fills<EP_WIRE_NVFP4>(a.d))
        return layout == EP_RANK_MAJOR ? launch_wire_staged<EP_RANK_MAJOR, EP_WIRE_NVFP4>(a, wq, ws, st)
                                       : launch_wire_staged<EP_EXPERT_MAJOR, EP_WIRE_NVFP4>(a, wq, ws, st);
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

}  // namespace ep
