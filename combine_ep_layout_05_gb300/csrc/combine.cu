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

cudaError_t launch_combine(int layout, const CombineArgs &a, int grid, cudaStream_t st) {
    if (layout == EP_RANK_MAJOR) combine_kernel<EP_RANK_MAJOR><<<grid, kWarps * 32, 0, st>>>(a);
    else combine_kernel<EP_EXPERT_MAJOR><<<grid, kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ep
