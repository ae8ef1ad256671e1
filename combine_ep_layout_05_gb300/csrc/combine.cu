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
// exactly once.  The piece is then produced in 16-byte chunks (8 channels):
// a lane loads one or two chunks of up to 8 or 4 source rows back to back
// (16-byte loads, all in flight), then accumulates them with fp32 FMAs in
// row order, rounds to bf16 and stores each chunk with one 16-byte store.
// Deterministic: no atomics, fixed order.
#include "combine_device.cuh"
#include "vec8.cuh"

namespace ep {

namespace {

#ifndef EP_COMBINE_LD_HINT
#define EP_COMBINE_LD_HINT 0
#endif

// One (token, piece) unit of combine: U 16-byte chunks per lane (32 lanes
// apart) of up to G source rows are loaded back to back, then accumulated in
// row order with fp32 FMAs and stored as bf16.
template <int U, int G>
__device__ __forceinline__ void combine_piece(const uint4 *y, uint4 *out, const int64_t *rows, const float *wts,
                                              int nd, int64_t t, int64_t hc, int64_t c0, int64_t c1, uint64_t pol,
                                              int lane) {
    for (int64_t cb = c0 + lane; cb < c1; cb += 32 * U) {
        float acc[U][8];
#pragma unroll
        for (int x = 0; x < U; ++x)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[x][i] = 0.f;
        for (int g0 = 0; g0 < nd; g0 += G) {
            uint4 v[G][U];
#pragma unroll
            for (int i = 0; i < G; ++i)
#pragma unroll
                for (int x = 0; x < U; ++x)
                    if (g0 + i < nd && cb + 32 * x < c1) v[i][x] = ld_stream_hint(y + rows[g0 + i] * hc + cb + 32 * x, pol);
#pragma unroll
            for (int i = 0; i < G; ++i) {
                if (g0 + i < nd) {
                    const float w = wts[g0 + i];
#pragma unroll
                    for (int x = 0; x < U; ++x) {
                        const uint32_t q[4] = {v[i][x].x, v[i][x].y, v[i][x].z, v[i][x].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            acc[x][2 * h] = __fmaf_rn(w, bf16_lo(q[h]), acc[x][2 * h]);
                            acc[x][2 * h + 1] = __fmaf_rn(w, bf16_hi(q[h]), acc[x][2 * h + 1]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int x = 0; x < U; ++x)
            if (cb + 32 * x < c1)
                st_v4(out + t * hc + cb + 32 * x,
                      make_uint4(pack_bf16x2(acc[x][0], acc[x][1]), pack_bf16x2(acc[x][2], acc[x][3]),
                                 pack_bf16x2(acc[x][4], acc[x][5]), pack_bf16x2(acc[x][6], acc[x][7])));
    }
}

// Channels [hb, he) of a token with 32-byte lanes: each lane owns 16
// contiguous channels of every 512-channel step and keeps 8 32-byte loads
// (slots) in flight: one step of up to 8 rows, or, for tokens with at most
// two_max (<= 4) rows, two steps of up to 4 rows (slots 0-3 the first step,
// 4-7 the second), so that such tokens still have 8 loads in flight.
// The slots' element offsets and weights are laid out once per unit in
// rows[8..15] / wts[8..15] (free: at most 8 rows), so both shapes run the
// same instructions.  MANY (tokens may have more than 8 rows): one step per
// batch, rows beyond 8 in further batches of 8 accumulated into the same
// sums.  Each output is the fp32 FMA chain over the token's rows in order,
// whatever the batching, so the sums equal combine_piece's bit for bit.
template <bool MANY>
__device__ __forceinline__ void combine_row_wide(const uint16_t *y, uint16_t *out, int64_t *rows, float *wts,
                                                 int nd, int two_max, int64_t t, int64_t H, int64_t hb, int64_t he,
                                                 int lane) {
    uint16_t *orow = out + t * H;
    if (MANY) {
        for (int64_t h0 = hb + (int64_t)lane * 16; h0 < he; h0 += 512) {
            float acc[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c] = 0.f;
            for (int g0 = 0; g0 < nd; g0 += 8) {
                uint32_t v[8][8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (g0 + i < nd) ld_stream8(y + rows[g0 + i] * H + h0, v[i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (g0 + i < nd) {
                        const float w = wts[g0 + i];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            acc[2 * c] = __fmaf_rn(w, bf16_lo(v[i][c]), acc[2 * c]);
                            acc[2 * c + 1] = __fmaf_rn(w, bf16_hi(v[i][c]), acc[2 * c + 1]);
                        }
                    }
                }
            }
            uint32_t o[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) o[c] = pack_bf16x2(acc[2 * c], acc[2 * c + 1]);
            st_v8(orow + h0, o);
        }
        return;
    }
    const bool two = nd <= two_max;   // two steps per batch
    int64_t *soff = rows + 8;
    float *sw = wts + 8;
    if (lane < 8) {
        const int i = two ? (lane & 3) : lane;
        soff[lane] = i < nd ? rows[i] * H + (two && lane >= 4 ? 512 : 0) : 0;
        sw[lane] = i < nd ? wts[i] : 0.f;
    }
    __syncwarp();
    const unsigned full = two ? ((1u << nd) - 1) * 0x11u : (1u << nd) - 1;   // slots in use
    const int64_t adv = two ? 1024 : 512;
    for (int64_t h0 = hb + (int64_t)lane * 16; h0 < he; h0 += adv) {
        const bool second = two && h0 + 512 < he;   // the batch's second step lies in the row
        const unsigned vm = two && !second ? full & 0x0Fu : full;
        uint32_t v[8][8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if ((vm >> q) & 1) ld_stream8(y + soff[q] + h0, v[q]);
        float acc[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (q == 4 && two) {   // the first step is complete
                uint32_t o[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) o[c] = pack_bf16x2(acc[2 * c], acc[2 * c + 1]);
                st_v8(orow + h0, o);
#pragma unroll
                for (int c = 0; c < 16; ++c) acc[c] = 0.f;
            }
            if ((vm >> q) & 1) {
                const float w = sw[q];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    acc[2 * c] = __fmaf_rn(w, bf16_lo(v[q][c]), acc[2 * c]);
                    acc[2 * c + 1] = __fmaf_rn(w, bf16_hi(v[q][c]), acc[2 * c + 1]);
                }
            }
        }
        if (!two || second) {   // the batch's last step
            uint32_t o[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) o[c] = pack_bf16x2(acc[2 * c], acc[2 * c + 1]);
            st_v8(orow + h0 + (two ? 512 : 0), o);
        }
    }
}

// U = 2 (two chunks per lane, up to 4 rows per batch): whole rows whose
// buffers are not 32-byte aligned; U = 1 (up to 8 rows per batch): row pieces
// shorter than 2048 channels (small batches), so all lanes stay busy.
// U values of the 32-byte-lane variant (at most 8 rows per token; any
// number), for whole rows and for row pieces of
// 2048 channels or more: up to 8 rows in flight per lane (one batch for a
// top-8 token), two CTAs per SM for the registers that takes.  Measured on
// GB300: at 512 tokens/rank (two pieces of 3584 channels) 71.6 against 75.7
// us with 16-byte lanes; at 4096 tokens/rank (whole rows) XXX against 456.7
// us with up to 4 rows per batch and three CTAs per SM; with shorter pieces
// (the low-latency shape's 1536 channels, 512 at 32 tokens/rank) the
// 16-byte lanes were faster (25.4 against 29.0 us, 10.2 against 12.3 us).
constexpr int kWideRows = 9, kWideRowsMany = 10;

template <int LAYOUT, int U>
__global__ void __launch_bounds__(kWarps * 32, U >= kWideRows ? 2 : EP_COMBINE_MINB) combine_kernel(CombineArgs a) {
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
    const uint64_t pol = l2_policy<EP_COMBINE_LD_HINT>();

    // Two-step batches (combine_row_wide) pay where most tokens have few rows
    // (skewed routing: the warps are latency-bound) and cost where most have
    // many (the memory system is saturated anyway): measured on GB300, tokens
    // of 3-4 rows in two-step batches cut the combine of a Zipf-routed 16 x
    // 4096 workload (mean 2-3 rows) from 521 to 467 us and slowed uniform
    // top-8 routing (5.3 rows) from 441 to 451 us.  So each warp uses them
    // for up to 4 rows while the tokens it has combined average under 4.5
    // rows, else for up to 2.  The sums do not depend on the batching.
    int64_t seen_rows = 0, seen_units = 0;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        const int nd = gather_sources<LAYOUT>(a, t, src, rows, wts);
        const int64_t c0 = p * pc, c1 = min(c0 + pc, hc);
        if (U >= kWideRows) {
            const int two_max = 2 * seen_rows >= 9 * seen_units && seen_units ? 2 : 4;
            seen_rows += nd;
            ++seen_units;
            combine_row_wide<U == kWideRowsMany>(a.y, a.out, rows, wts, nd, two_max, t, d.H, c0 * 8, c1 * 8, lane);
        } else {
            combine_piece<U, U == 1 ? 8 : 4>(y, out, rows, wts, nd, t, hc, c0, c1, pol, lane);
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

namespace {

// Resident CTAs of the narrow (16-byte lane) and wide (32-byte lane) kernels
// on this device: the grid caps of the persistent launches.
int narrow_cap(int layout) {
    static std::atomic<int> cache[2][kCacheDevices];
    return cached_per_device(cache[layout], [&](int) {
        return layout == EP_RANK_MAJOR ? grid_cap_for(combine_kernel<EP_RANK_MAJOR, 1>)
                                       : grid_cap_for(combine_kernel<EP_EXPERT_MAJOR, 1>);
    });
}

int wide_cap(int layout) {
    static std::atomic<int> cache[2][kCacheDevices];
    return cached_per_device(cache[layout], [&](int) {
        return layout == EP_RANK_MAJOR ? grid_cap_for(combine_kernel<EP_RANK_MAJOR, kWideRows>)
                                       : grid_cap_for(combine_kernel<EP_EXPERT_MAJOR, kWideRows>);
    });
}

}  // namespace

#ifndef EP_COMBINE_WIDE
#define EP_COMBINE_WIDE 1
#endif

// Splits each token row into pieces and picks the kernel.  Each warp of the
// persistent grid takes (token, piece) units in fixed rounds; a unit costs
// about one memory round trip for its routing entry and slots plus one per
// step of its piece (512 channels with 32-byte lanes, 256 with 16-byte
// lanes).  The split minimises rounds x cost per unit, so that the grid is
// filled and the last round is not a mostly idle one.
void plan_combine(int layout, CombineArgs &a, int &grid, int &kind) {
    const Dims &d = a.d;
    const bool wide32 = EP_COMBINE_WIDE && d.H % 16 == 0 && ((uintptr_t)a.y & 31) == 0 &&
                        ((uintptr_t)a.out & 31) == 0;
    const int64_t max_pieces = (d.H + 255) / 256;
    int64_t best = -1;
    a.pieces = 1;
    a.piece_elems = d.H;
    kind = wide32 ? kWideRows : 2;
    for (int64_t p = 1; p <= max_pieces && d.T > 0; ++p) {
        int64_t per = (d.H + p - 1) / p;
        per = (per + 255) / 256 * 256;
        const int64_t pp = (d.H + per - 1) / per;
        if (pp != p) continue;   // the same split as a smaller p
        const int k = wide32 && (pp == 1 || per >= 2048) ? kWideRows : pp == 1 ? 2 : 1;
        const int64_t warps = (int64_t)(k == kWideRows ? wide_cap(layout) : narrow_cap(layout)) * kWarps;
        const int64_t step = k == 1 ? 256 : 512;
        const int64_t rounds = (d.T * pp + warps - 1) / warps;
        const int64_t cost = rounds * ((per + step - 1) / step + 1);
        if (best < 0 || cost < best) {
            best = cost;
            a.pieces = pp;
            a.piece_elems = per;
            kind = k;
        }
    }
    // Many rounds of whole rows (bandwidth-bound): rows in two halves, so
    // that the units of the last, partly filled round are half as long.
    // Measured on GB300 with uniform top-8 routing at 4096 tokens/rank:
    // combine 449.9 us whole rows, 442.0 us halves (at 8192 tokens/rank
    // 880 against 866 us).  With Zipf routing (16 x 4096, 2-3 rows per
    // token) halves cost 2.9% (475.9 against 489.7 us): short units make
    // the routing round trip of each unit count; the uniform case decides.
    const int64_t wide_warps = (int64_t)wide_cap(layout) * kWarps;
    if (kind == kWideRows && a.pieces == 1 && d.T >= 4 * wide_warps && d.H >= 2 * 2048) {
        a.piece_elems = ((d.H + 1) / 2 + 255) / 256 * 256;
        a.pieces = (d.H + a.piece_elems - 1) / a.piece_elems;
    }
    const int cap = kind == kWideRows ? wide_cap(layout) : narrow_cap(layout);
    // more than 8 rows per token: the wide kernel's batch loop
    if (kind == kWideRows && (layout == EP_RANK_MAJOR ? (d.k < d.R ? d.k : d.R) : d.k) > 8) kind = kWideRowsMany;
    const int64_t units = d.T * a.pieces;
    const int64_t want = (units + kWarps - 1) / kWarps;
    grid = (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

cudaError_t launch_combine(int layout, CombineArgs &a, cudaStream_t st) {
    int grid = 1, kind = 1;
    plan_combine(layout, a, grid, kind);
    const unsigned b = kWarps * 32;
    if (layout == EP_RANK_MAJOR) {
        if (kind == kWideRows) combine_kernel<EP_RANK_MAJOR, kWideRows><<<grid, b, 0, st>>>(a);
        else if (kind == kWideRowsMany) combine_kernel<EP_RANK_MAJOR, kWideRowsMany><<<grid, b, 0, st>>>(a);
        else if (kind == 2) combine_kernel<EP_RANK_MAJOR, 2><<<grid, b, 0, st>>>(a);
        else combine_kernel<EP_RANK_MAJOR, 1><<<grid, b, 0, st>>>(a);
    } else {
        if (kind == kWideRows) combine_kernel<EP_EXPERT_MAJOR, kWideRows><<<grid, b, 0, st>>>(a);
        else if (kind == kWideRowsMany) combine_kernel<EP_EXPERT_MAJOR, kWideRowsMany><<<grid, b, 0, st>>>(a);
        else if (kind == 2) combine_kernel<EP_EXPERT_MAJOR, 2><<<grid, b, 0, st>>>(a);
        else combine_kernel<EP_EXPERT_MAJOR, 1><<<grid, b, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace ep
