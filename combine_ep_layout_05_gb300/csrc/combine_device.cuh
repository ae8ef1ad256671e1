// Device code shared by the bf16 combine and the wire-format combines:
// the routing-entry gather that resolves a token's receive rows and
// weights, and the exact decoders of the wire formats' codes.
#pragma once

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kWarps = 8;   // warps per CTA of the register-path kernels
#ifndef EP_COMBINE_MINB
#define EP_COMBINE_MINB 3
#endif

// f16 pair (element 0 in the low half) -> two floats.  The mixed-precision
// add of the f16 value and an fp32 -0.0 is exact for every finite f16 (the
// result of cvt.f32.f16, bit for bit); in a decode microbenchmark on GB300
// it sustained 17-22% more decoded elements per clock than cvt.f32.f16.
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h2) {
    float lo, hi;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; add.rn.f32.f16 %0, l, 0f80000000; add.rn.f32.f16 %1, h, 0f80000000; }"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

// two e4m3 codes (element 0 in the low byte) -> two floats, exact
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t c2) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
    return f16x2_to_f32x2(h2);
}

// the eight e2m1 codes of a word (two per byte, element 0 in the low nibble
// of the low byte) -> four f16 pairs, exact; the word is split into its
// bytes by a register move instead of a shift and mask per byte
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
    asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
        " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
        " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// A token's routing entry as the lanes of a warp hold it before it is
// resolved: lane j < k its expert id and weight, and the token's slots
// (rank-major: lane r % 32 the slot of rank r, s1 for ranks 32..63;
// expert-major: lane j the slot of entry j).
struct RouteRegs {
    int64_t e;
    float w;
    int32_t s0, s1;
};

// Issues the loads of token t's routing entry and slots (the slots with the
// entry, not after it: one memory round trip fewer before the rows can be
// read).
template <int LAYOUT>
__device__ __forceinline__ RouteRegs load_route(const CombineArgs &a, int64_t t) {
    const Dims &d = a.d;
    const int lane = threadIdx.x & 31;
    RouteRegs g{-1, 0.f, -1, -1};
    if (t < 0) return g;
    if (lane < d.k) {
        g.e = a.topk_idx[t * d.k + lane];
        g.w = a.topk_weights[t * d.k + lane];
    }
    if (LAYOUT == EP_RANK_MAJOR) {
        if (lane < d.R) g.s0 = a.rank_slot[t * d.R + lane];
        if (lane + 32 < d.R) g.s1 = a.rank_slot[t * d.R + lane + 32];
    } else if (lane < d.k) {
        g.s0 = a.expert_slot[t * d.k + lane];
    }
    return g;
}

// Resolves token t's routing entry (from load_route) into its receive rows
// and weights: rows[i], wts[i] for i < the returned count, in j order of
// the first entry of each row.  Ids outside [0, E) and repeats are dropped
// (and flagged in the status word); in the rank-major layout the entries
// of one rank share its row, with their weights summed in j order.
template <int LAYOUT>
__device__ __forceinline__ int resolve_sources(const CombineArgs &a, int64_t t, int64_t src, const RouteRegs &g,
                                               int64_t *rows, float *wts) {
    const Dims &d = a.d;
    const int lane = threadIdx.x & 31;
    int st = 0;
    const int64_t e = g.e;
    const float w = g.w;
    const int32_t s0 = g.s0, s1 = g.s1;
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
        const int r = kept ? (int)rank_of(d, (uint32_t)e) : -1;
        const unsigned grp = __match_any_sync(kFull, kept ? r : -100 - lane);
        const bool leader = kept && !(grp & lanemask_lt());
        // weight of the rank: the group's weights summed in j order
        wsum = 0.f;
        for (int j = 0; j < (int)d.k; ++j) {
            const float wj = __shfl_sync(kFull, w, j);
            if (leader && ((grp >> j) & 1)) wsum += wj;
        }
        // slot of rank r: lane r % 32 holds it (in s1 for ranks 32..63)
        const int rr = r < 0 ? 0 : r;
        const int32_t g0 = __shfl_sync(kFull, s0, rr & 31), g1 = __shfl_sync(kFull, s1, rr & 31);
        if (leader) {
            const int32_t slot = rr < 32 ? g0 : g1;
            if (slot >= 0 && slot < d.Tr) row = ((int64_t)r * d.R + src) * d.Tr + slot;
            else st |= EP_STATUS_BAD_SLOT;
        }
    } else {
        if (kept) {
            const int32_t slot = s0;
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
__device__ __forceinline__ int gather_sources(const CombineArgs &a, int64_t t, int64_t src, int64_t *rows,
                                              float *wts) {
    return resolve_sources<LAYOUT>(a, t, src, load_route<LAYOUT>(a, t), rows, wts);
}

// 2^(code - 127) for an e8m0 code 0..254 (code 0 is the denormal 2^-127)
__device__ __forceinline__ float e8m0_value(uint32_t code) {
    return code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);
}

}  // namespace

}  // namespace ep
