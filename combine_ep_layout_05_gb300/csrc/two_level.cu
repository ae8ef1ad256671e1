// Two-level (node-forwarding) dispatch and combine.
//
// What ("MORI-EP Benchmark", "Bandwidth Computation": the inter-node fabric
// carries one copy per (token, destination node) - the "algo" count - and
// the node then forwards it to the token's ranks; "Combine": the reverse,
// same byte counts.  MSCCL++ PR #860: the internode dispatch forwards
// through the node's NVLink ranks, and combine reduces inside the node
// before the inter-node hop).  With the ranks emulated in one GPU:
//   dispatch hop 1: x[t] -> staging row (n, src, node_slot[t, n]) of every
//                   node n the token goes to (ep_dispatch's kernels with a
//                   node-major destination set);
//   dispatch hop 2: staging row -> rank-major row of each of the token's
//                   ranks in n (forward_kernel below);
//   combine hop 1:  per (token, node), the weighted sum of the node's rank
//                   rows, rounded to bf16 into the staging row (the partial
//                   the node sends back);
//   combine hop 2:  out[t] = bf16(sum over nodes of the partials), fp32.
#include "dispatch_device.cuh"
#include "vec8.cuh"

namespace ep {

namespace {

constexpr int kMaxRanks2 = 64;

// Hop 2 of the dispatch: a warp owns a (token, piece) unit; lanes pair each
// of the token's ranks with its node's staging row, then the piece of each
// staging row is read once and stored to the node's ranks (WIDE: 32-byte
// lanes, 256-bit loads and stores).
template <bool WIDE>
__global__ void __launch_bounds__(kWarps * 32) forward_kernel(DispatchArgs a, const uint16_t *stage,
                                                              uint16_t *recv) {
    __shared__ int64_t s_src[kWarps][kMaxRanks2], s_dst[kWarps][kMaxRanks2];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t hc = d.H / 8, pc = a.piece_elems / 8;
    const int64_t units = d.T * a.pieces;
    const uint4 *sg = reinterpret_cast<const uint4 *>(stage);
    uint4 *rv = reinterpret_cast<uint4 *>(recv);
    constexpr int U = 4;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        int np = 0, st = 0;
        for (int r0 = 0; r0 < (int)d.R; r0 += 32) {
            const int r = r0 + lane;
            int64_t srow = -1, drow = -1;
            if (r < d.R) {
                const int32_t rs = a.rank_slot[t * d.R + r];
                if (rs >= 0 && rs < d.Tr) {
                    const int64_t n = r / d.G;
                    const int32_t ns = a.node_slot[t * d.N + n];
                    if (ns >= 0 && ns < d.Tr) {
                        srow = (n * d.R + src) * d.Tr + ns;
                        drow = ((int64_t)r * d.R + src) * d.Tr + rs;
                    } else {
                        st |= EP_STATUS_BAD_SLOT;
                    }
                } else if (rs != -1) {
                    st |= EP_STATUS_BAD_SLOT;
                }
            }
            const unsigned m = __ballot_sync(kFull, drow >= 0);
            if (drow >= 0) {
                const int i = np + __popc(m & lanemask_lt());
                s_src[warp][i] = srow;
                s_dst[warp][i] = drow;
            }
            np += __popc(m);
        }
        if (st) raise_status(a.dev_status, st);
        __syncwarp();
        if (WIDE) {
            // 32-byte lanes: two 16-channel chunks per lane and step
            constexpr int UW = U / 2;
            const int64_t w0 = p * (a.piece_elems / 16), w1 = min(w0 + a.piece_elems / 16, d.H / 16);
            for (int64_t c = w0 + lane; c < w1; c += 32 * UW) {
                uint32_t v[UW][8];
                int64_t cur = -1;
                for (int i = 0; i < np; ++i) {
                    if (s_src[warp][i] != cur) {
                        cur = s_src[warp][i];
#pragma unroll
                        for (int k = 0; k < UW; ++k)
                            if (c + 32 * k < w1) ld_stream8(stage + cur * d.H + (c + 32 * k) * 16, v[k]);
                    }
#pragma unroll
                    for (int k = 0; k < UW; ++k)
                        if (c + 32 * k < w1) st_v8(recv + s_dst[warp][i] * d.H + (c + 32 * k) * 16, v[k]);
                }
            }
        } else {
            const int64_t c0 = p * pc, c1 = min(c0 + pc, hc);
            for (int64_t c = c0 + lane; c < c1; c += 32 * U) {
                uint4 v[U];
                int64_t cur = -1;
                for (int i = 0; i < np; ++i) {
                    // pairs come in ascending rank order, so a node's pairs are
                    // adjacent: each staging row is read once
                    if (s_src[warp][i] != cur) {
                        cur = s_src[warp][i];
#pragma unroll
                        for (int k = 0; k < U; ++k)
                            if (c + 32 * k < c1) v[k] = ld_stream(sg + cur * hc + c + 32 * k);
                    }
#pragma unroll
                    for (int k = 0; k < U; ++k)
                        if (c + 32 * k < c1) st_v4(rv + s_dst[warp][i] * hc + c + 32 * k, v[k]);
                }
            }
        }
        __syncwarp();
    }
}

// Hop 1 of the combine: a warp owns a (token, piece) unit.  Lanes j < k
// keep the valid, non-repeated entries; entries on one rank share that
// rank's row (weights summed in j order).  The rank rows are ordered by node
// (stable), and for each node the weighted rows are summed in fp32 and
// rounded to bf16 into the node's staging row.  Per channel chunk a lane
// loads the rows of all the token's nodes back to back (up to EP_NODE_G in
// flight), then walks them in node order, storing a node's partial after its
// last row (a bit mask marks those rows).  WIDE: 32-byte lanes (16
// contiguous channels, one 256-bit load per row); otherwise EP_NODE_U
// 16-byte chunks per lane.
#ifndef EP_NODE_G
#define EP_NODE_G 4
#endif
#ifndef EP_NODE_U
#define EP_NODE_U 2
#endif
#ifndef EP_SUM_U
#define EP_SUM_U 4
#endif

template <bool WIDE>
__global__ void __launch_bounds__(kWarps * 32) combine_node_kernel(CombineArgs a, uint16_t *stage) {
    constexpr int G = EP_NODE_G, U = EP_NODE_U;
    __shared__ int64_t s_row[kWarps][32], s_srow[kWarps][32];
    __shared__ float s_w[kWarps][32];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t hc = d.H / 8, pc = a.piece_elems / 8;
    const int64_t units = d.T * a.pieces;
    const uint4 *y = reinterpret_cast<const uint4 *>(a.y);
    uint4 *sg = reinterpret_cast<uint4 *>(stage);
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        int st = 0;
        int64_t e = -1;
        float w = 0.f;
        if (lane < d.k) {
            e = a.topk_idx[t * d.k + lane];
            w = a.topk_weights[t * d.k + lane];
        }
        const bool in_range = e >= 0 && e < d.E;
        if (lane < d.k && !in_range && e != -1) st |= EP_STATUS_BAD_EXPERT;
        const unsigned same = __match_any_sync(kFull, in_range ? (long long)e : -2 - lane);
        const bool dup = in_range && (same & lanemask_lt());
        if (dup) st |= EP_STATUS_DUP_EXPERT;
        const bool kept = in_range && !dup;
        const int r = kept ? (int)rank_of(d, (uint32_t)e) : -1;
        const unsigned grp = __match_any_sync(kFull, kept ? r : -100 - lane);
        const bool leader = kept && !(grp & lanemask_lt());
        float wsum = 0.f;
        for (int j = 0; j < (int)d.k; ++j) {
            const float wj = __shfl_sync(kFull, w, j);
            if (leader && ((grp >> j) & 1)) wsum += wj;
        }
        int64_t row = -1, srow = -1;
        int node = 1 << 30;
        if (leader) {
            const int32_t rs = a.rank_slot[t * d.R + r];
            node = r / (int)d.G;
            const int32_t ns = a.node_slot[t * d.N + node];
            if (rs >= 0 && rs < d.Tr && ns >= 0 && ns < d.Tr) {
                row = ((int64_t)r * d.R + src) * d.Tr + rs;
                srow = ((int64_t)node * d.R + src) * d.Tr + ns;
            } else {
                st |= EP_STATUS_BAD_SLOT;
                node = 1 << 30;
            }
        }
        if (st) raise_status(a.dev_status, st);
        // stable order by node: position = sources with a smaller node, or the
        // same node and a lower lane
        const bool have = row >= 0;
        const unsigned hm = __ballot_sync(kFull, have);
        int pos = 0;
        for (int j = 0; j < 32; ++j) {
            const int nj = __shfl_sync(kFull, node, j);
            if (((hm >> j) & 1) && (nj < node || (nj == node && j < lane))) ++pos;
        }
        // the last row of each node (the highest lane of its node among the
        // kept rows) closes that node's partial
        const unsigned same_node = __match_any_sync(kFull, have ? node : -1 - lane);
        const bool last = have && lane == 31 - __clz(same_node);
        const unsigned lastmask = __reduce_or_sync(kFull, last ? 1u << pos : 0u);
        if (have) {
            s_row[warp][pos] = row;
            s_srow[warp][pos] = srow;
            s_w[warp][pos] = wsum;
        }
        __syncwarp();
        const int nd = __popc(hm);
        if (WIDE) {
            // 32-byte lanes: 16 contiguous channels of up to G rows per batch
            const int64_t w0 = p * (a.piece_elems / 16), w1 = min(w0 + a.piece_elems / 16, d.H / 16);
            for (int64_t c = w0 + lane; c < w1; c += 32) {
                float2 acc[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) acc[h] = make_float2(0.f, 0.f);
                for (int g0 = 0; g0 < nd; g0 += G) {
                    uint32_t v[G][8];
#pragma unroll
                    for (int q = 0; q < G; ++q)
                        if (g0 + q < nd) ld_stream8(a.y + s_row[warp][g0 + q] * d.H + c * 16, v[q]);
#pragma unroll
                    for (int q = 0; q < G; ++q) {
                        if (g0 + q < nd) {
                            const float wq = s_w[warp][g0 + q];
                            const float2 w2 = make_float2(wq, wq);
#pragma unroll
                            for (int h = 0; h < 8; ++h)
                                acc[h] = __ffma2_rn(w2, make_float2(bf16_lo(v[q][h]), bf16_hi(v[q][h])), acc[h]);
                            if ((lastmask >> (g0 + q)) & 1) {
                                uint32_t o[8];
#pragma unroll
                                for (int h = 0; h < 8; ++h) {
                                    o[h] = pack_bf16x2(acc[h].x, acc[h].y);
                                    acc[h] = make_float2(0.f, 0.f);
                                }
                                st_v8(stage + s_srow[warp][g0 + q] * d.H + c * 16, o);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            continue;
        }
        const int64_t c0 = p * pc, c1 = min(c0 + pc, hc);
        // U 16-byte chunks per lane (32 lanes apart) and up to G rows per
        // batch: the few rows of a token still give U * rows loads in flight
        for (int64_t cb = c0 + lane; cb < c1; cb += 32 * U) {
            float2 acc[U][4];
#pragma unroll
            for (int x = 0; x < U; ++x)
#pragma unroll
                for (int h = 0; h < 4; ++h) acc[x][h] = make_float2(0.f, 0.f);
            for (int g0 = 0; g0 < nd; g0 += G) {
                uint4 v[G][U];
#pragma unroll
                for (int q = 0; q < G; ++q)
#pragma unroll
                    for (int x = 0; x < U; ++x)
                        if (g0 + q < nd && cb + 32 * x < c1)
                            v[q][x] = ld_stream(y + s_row[warp][g0 + q] * hc + cb + 32 * x);
#pragma unroll
                for (int q = 0; q < G; ++q) {
                    if (g0 + q < nd) {
                        const float wq = s_w[warp][g0 + q];
                        const float2 w2 = make_float2(wq, wq);
                        const bool last_row = (lastmask >> (g0 + q)) & 1;
#pragma unroll
                        for (int x = 0; x < U; ++x) {
                            const uint32_t qw[4] = {v[q][x].x, v[q][x].y, v[q][x].z, v[q][x].w};
#pragma unroll
                            for (int h = 0; h < 4; ++h)
                                acc[x][h] = __ffma2_rn(w2, make_float2(bf16_lo(qw[h]), bf16_hi(qw[h])), acc[x][h]);
                            if (last_row) {
                                if (cb + 32 * x < c1)
                                    st_v4(sg + s_srow[warp][g0 + q] * hc + cb + 32 * x,
                                          make_uint4(pack_bf16x2(acc[x][0].x, acc[x][0].y),
                                                     pack_bf16x2(acc[x][1].x, acc[x][1].y),
                                                     pack_bf16x2(acc[x][2].x, acc[x][2].y),
                                                     pack_bf16x2(acc[x][3].x, acc[x][3].y)));
#pragma unroll
                                for (int h = 0; h < 4; ++h) acc[x][h] = make_float2(0.f, 0.f);
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
    }
}

// Hop 2 of the combine: out[t] = bf16(sum over the token's nodes, in
// ascending order, of the bf16 partials), fp32 accumulation; several chunks
// per lane in flight (WIDE: 32-byte lanes).
template <bool WIDE>
__global__ void __launch_bounds__(kWarps * 32) combine_sum_kernel(CombineArgs a, const uint16_t *stage) {
    constexpr int U = EP_SUM_U;
    __shared__ int64_t s_srow[kWarps][kMaxRanks2];
    const Dims &d = a.d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t hc = d.H / 8, pc = a.piece_elems / 8;
    const int64_t units = d.T * a.pieces;
    const uint4 *sg = reinterpret_cast<const uint4 *>(stage);
    uint4 *out = reinterpret_cast<uint4 *>(a.out);
    for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units; u += (int64_t)gridDim.x * kWarps) {
        const int64_t t = u / a.pieces, p = u % a.pieces;
        const int64_t src = t / d.Tr;
        int nn = 0;
        for (int n0 = 0; n0 < (int)d.N; n0 += 32) {
            const int n = n0 + lane;
            int64_t srow = -1;
            if (n < d.N) {
                const int32_t ns = a.node_slot[t * d.N + n];
                if (ns >= 0 && ns < d.Tr) srow = ((int64_t)n * d.R + src) * d.Tr + ns;
            }
            const unsigned m = __ballot_sync(kFull, srow >= 0);
            if (srow >= 0) s_srow[warp][nn + __popc(m & lanemask_lt())] = srow;
            nn += __popc(m);
        }
        __syncwarp();
        if (WIDE) {
            // 32-byte lanes, U / 2 chunks of 16 channels per lane and step
            constexpr int UW = U / 2;
            const int64_t w0 = p * (a.piece_elems / 16), w1 = min(w0 + a.piece_elems / 16, d.H / 16);
            for (int64_t cb = w0 + lane; cb < w1; cb += 32 * UW) {
                float acc[UW][16];
#pragma unroll
                for (int x = 0; x < UW; ++x)
#pragma unroll
                    for (int h = 0; h < 16; ++h) acc[x][h] = 0.f;
                for (int i0 = 0; i0 < nn; i0 += 2) {
                    uint32_t v[2][UW][8];
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int x = 0; x < UW; ++x)
                            if (i0 + q < nn && cb + 32 * x < w1)
                                ld_stream8(stage + s_srow[warp][i0 + q] * d.H + (cb + 32 * x) * 16, v[q][x]);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        if (i0 + q < nn) {
#pragma unroll
                            for (int x = 0; x < UW; ++x)
#pragma unroll
                                for (int h = 0; h < 8; ++h) {
                                    acc[x][2 * h] += bf16_lo(v[q][x][h]);
                                    acc[x][2 * h + 1] += bf16_hi(v[q][x][h]);
                                }
                        }
                    }
                }
#pragma unroll
                for (int x = 0; x < UW; ++x) {
                    if (cb + 32 * x < w1) {
                        uint32_t o[8];
#pragma unroll
                        for (int h = 0; h < 8; ++h) o[h] = pack_bf16x2(acc[x][2 * h], acc[x][2 * h + 1]);
                        st_v8(a.out + t * d.H + (cb + 32 * x) * 16, o);
                    }
                }
            }
            __syncwarp();
            continue;
        }
        const int64_t c0 = p * pc, c1 = min(c0 + pc, hc);
        // U 16-byte chunks per lane: a token has ~1 partial per node
        for (int64_t cb = c0 + lane; cb < c1; cb += 32 * U) {
            float acc[U][8];
#pragma unroll
            for (int x = 0; x < U; ++x)
#pragma unroll
                for (int h = 0; h < 8; ++h) acc[x][h] = 0.f;
            // the partials' loads back to back (2 rows x U chunks in flight), then the sums
            for (int i0 = 0; i0 < nn; i0 += 2) {
                uint4 v[2][U];
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int x = 0; x < U; ++x)
                        if (i0 + q < nn && cb + 32 * x < c1) v[q][x] = ld_stream(sg + s_srow[warp][i0 + q] * hc + cb + 32 * x);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (i0 + q < nn) {
#pragma unroll
                        for (int x = 0; x < U; ++x) {
                            const uint32_t qw[4] = {v[q][x].x, v[q][x].y, v[q][x].z, v[q][x].w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                acc[x][2 * h] += bf16_lo(qw[h]);
                                acc[x][2 * h + 1] += bf16_hi(qw[h]);
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
        __syncwarp();
    }
}

int64_t unit_grid2(int64_t units, int per_sm) {
    int64_t g = (units + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    if (g > cap) g = cap;
    return g < 1 ? 1 : g;
}

#ifndef EP_TWO_LEVEL_WIDE
#define EP_TWO_LEVEL_WIDE 1
#endif

// 32-byte lanes: rows and pieces of 16-channel multiples, 32-byte aligned buffers
bool wide_ok(const Dims &d, int64_t piece_elems, const void *p0, const void *p1) {
    return EP_TWO_LEVEL_WIDE && d.H % 16 == 0 && piece_elems % 16 == 0 && ((uintptr_t)p0 & 31) == 0 &&
           ((uintptr_t)p1 & 31) == 0;
}

}  // namespace

cudaError_t launch_forward(const DispatchArgs &a, uint16_t *stage, uint16_t *recv, cudaStream_t st) {
    const unsigned g = (unsigned)unit_grid2(a.d.T * a.pieces, 8);
    if (wide_ok(a.d, a.piece_elems, stage, recv)) forward_kernel<true><<<g, kWarps * 32, 0, st>>>(a, stage, recv);
    else forward_kernel<false><<<g, kWarps * 32, 0, st>>>(a, stage, recv);
    return cudaGetLastError();
}

cudaError_t launch_combine_two_level(const CombineArgs &a, uint16_t *stage, cudaStream_t st) {
    const unsigned g = (unsigned)unit_grid2(a.d.T * a.pieces, 3);
    const bool wide = wide_ok(a.d, a.piece_elems, stage, a.y) && ((uintptr_t)a.out & 31) == 0;
    if (wide) combine_node_kernel<true><<<g, kWarps * 32, 0, st>>>(a, stage);
    else combine_node_kernel<false><<<g, kWarps * 32, 0, st>>>(a, stage);
    cudaError_t e = cudaGetLastError();
    if (e) return e;
    const unsigned g2 = (unsigned)unit_grid2(a.d.T * a.pieces, 8);
    if (wide) combine_sum_kernel<true><<<g2, kWarps * 32, 0, st>>>(a, stage);
    else combine_sum_kernel<false><<<g2, kWarps * 32, 0, st>>>(a, stage);
    return cudaGetLastError();
}

}  // namespace ep
