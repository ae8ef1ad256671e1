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

// A whole row with 32-byte lanes: each lane owns 16 contiguous channels of a
// 512-channel step, loads them from up to G rows with one 32-byte load per
// row (all in flight), accumulates in row order and stores them with one
// 32-byte store.  Same sums as combine_piece.
template <int G>
__device__ __forceinline__ void combine_row_wide(const uint16_t *y, uint16_t *out, const int64_t *rows,
                                                 const float *wts, int nd, int64_t t, int64_t H, int64_t hb,
                                                 int64_t he, int lane) {
    for (int64_t h0 = hb + (int64_t)lane * 16; h0 < he; h0 += 512) {
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        for (int g0 = 0; g0 < nd; g0 += G) {
            uint32_t v[G][8];
#pragma unroll
            for (int i = 0; i < G; ++i)
                if (g0 + i < nd) ld_stream8(y + rows[g0 + i] * H + h0, v[i]);
#pragma unroll
            for (int i = 0; i < G; ++i) {
                if (g0 + i < nd) {
                    const float w = wts[g0 + i];
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        acc[2 * h] = __fmaf_rn(w, bf16_lo(v[i][h]), acc[2 * h]);
                        acc[2 * h + 1] = __fmaf_rn(w, bf16_hi(v[i][h]), acc[2 * h + 1]);
                    }
                }
            }
        }
        uint32_t o[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) o[h] = pack_bf16x2(acc[2 * h], acc[2 * h + 1]);
        st_v8(out + t * H + h0, o);
    }
}

// U = 2 (two chunks per lane, up to 4 rows per batch) when a unit is a whole
// row: with few rows per token (skewed routing: ~2.3 rows) one chunk per
// lane left too few loads in flight; U = 1 (up to 8 rows per batch) when
// rows are split into pieces for small batches, so all lanes stay busy.
constexpr int kWideLanes = 8;   // U value of the 32-byte-lane variant (whole rows)
// U value of the 32-byte-lane variant for row pieces of 2048 channels or
// more (rows split in two or three): up to 8 rows in flight per lane, two
// CTAs per SM for the registers that takes.  Measured on GB300 at 512
// tokens/rank (two pieces of 3584 channels): combine 71.6 against 75.7 us
// with 16-byte lanes; with shorter pieces (the low-latency shape's 1536
// channels, 512 at 32 tokens/rank) the 16-byte lanes were faster (25.4
// against 29.0 us, 10.2 against 12.3 us).
constexpr int kWidePieces = 9;

template <int LAYOUT, int U>
__global__ void __launch_bounds__(kWarps * 32, U == kWidePieces ? 2 : EP_COMBINE_MINB) combine_kernel(CombineArgs a) {
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

    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        const int nd = gather_sources<LAYOUT>(a, t, src, rows, wts);
        const int64_t c0 = p * pc, c1 = min(c0 + pc, hc);
        if (U == kWideLanes) combine_row_wide<4>(a.y, a.out, rows, wts, nd, t, d.H, 0, d.H, lane);
        else if (U == kWidePieces) combine_row_wide<8>(a.y, a.out, rows, wts, nd, t, d.H, c0 * 8, c1 * 8, lane);
        else combine_piece<U, U == 1 ? 8 : 4>(y, out, rows, wts, nd, t, hc, c0, c1, pol, lane);
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
    static std::atomic<int> cache[2][kCacheDevices];
    return cached_per_device(cache[layout], [&](int) {
        return layout == EP_RANK_MAJOR ? grid_cap_for(combine_kernel<EP_RANK_MAJOR, 2>)
                                       : grid_cap_for(combine_kernel<EP_EXPERT_MAJOR, 2>);
    });
}

#ifndef EP_COMBINE_WIDE
#define EP_COMBINE_WIDE 1
#endif

cudaError_t launch_combine(int layout, const CombineArgs &a, int grid, cudaStream_t st) {
    const bool whole = a.pieces == 1;
    // 32-byte lanes: rows of 16-channel multiples, 32-byte aligned buffers;
    // whole rows, or pieces of at least 2048 channels
    const bool wide32 = EP_COMBINE_WIDE && a.d.H % 16 == 0 && ((uintptr_t)a.y & 31) == 0 &&
                        ((uintptr_t)a.out & 31) == 0;
    const bool wide = wide32 && whole;
    const bool wide_pieces = wide32 && !whole && a.piece_elems >= 2048;
    const unsigned b = kWarps * 32;
    if (wide_pieces) {
        static std::atomic<int> cap[2][kCacheDevices];
        const int c = cached_per_device(cap[layout], [&](int) {
            return layout == EP_RANK_MAJOR ? grid_cap_for(combine_kernel<EP_RANK_MAJOR, kWidePieces>)
                                           : grid_cap_for(combine_kernel<EP_EXPERT_MAJOR, kWidePieces>);
        });
        const int g = grid < c ? grid : c;
        if (layout == EP_RANK_MAJOR) combine_kernel<EP_RANK_MAJOR, kWidePieces><<<g, b, 0, st>>>(a);
        else combine_kernel<EP_EXPERT_MAJOR, kWidePieces><<<g, b, 0, st>>>(a);
        return cudaGetLastError();
    }
    if (layout == EP_RANK_MAJOR) {
        if (wide) combine_kernel<EP_RANK_MAJOR, kWideLanes><<<grid, b, 0, st>>>(a);
        else if (whole) combine_kernel<EP_RANK_MAJOR, 2><<<grid, b, 0, st>>>(a);
        else combine_kernel<EP_RANK_MAJOR, 1><<<grid, b, 0, st>>>(a);
    } else {
        if (wide) combine_kernel<EP_EXPERT_MAJOR, kWideLanes><<<grid, b, 0, st>>>(a);
        else if (whole) combine_kernel<EP_EXPERT_MAJOR, 2><<<grid, b, 0, st>>>(a);
        else combine_kernel<EP_EXPERT_MAJOR, 1><<<grid, b, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace ep
