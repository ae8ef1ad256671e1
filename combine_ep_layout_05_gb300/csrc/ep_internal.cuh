// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/ep.h"

namespace ep {

// Layout: one CTA of kLayoutThreads threads handles one chunk of up to
// kChunk tokens of a single source rank (chunks never straddle ranks).
constexpr unsigned kFull = 0xffffffffu;   // all lanes of a warp
constexpr int kChunk = 256;
constexpr int kLayoutThreads = 256;
constexpr int kChunkWords = kChunk / 32;   // bitmap words per column
constexpr int kMaxExperts = 1024;
constexpr int kMaxRanks = 64;
constexpr int kMaxTopk = 32;

struct Dims {
    int64_t T, H, k, E, R, G;
    int64_t N, Er, En, Tr;
    int64_t cps;      // chunks per source rank = ceil(Tr / kChunk)
    int64_t cols;     // histogram columns per chunk: R + E + N
    // e / Er and e / En for expert ids 0 <= e < 1024 as (e * mul) >> shift
    // (see div_magic)
    uint32_t er_mul, er_shift, en_mul, en_shift;
};

// Multiplier and shift that divide every integer 0 <= n < 2^10 by d
// (1 <= d <= 1024) exactly: with s = 10 + ceil(log2 d) and m = ceil(2^s / d),
// m * d - 2^s < d <= 2^(s - 10), so floor(n * m / 2^s) = floor(n / d) for
// all n < 2^10 (Granlund and Montgomery, "Division by invariant integers
// using multiplication", 1994); n * m < 2^22 fits 32 bits.
inline void div_magic(int64_t d, uint32_t &mul, uint32_t &shift) {
    uint32_t l = 0;
    while (((int64_t)1 << l) < d) ++l;
    shift = 10 + l;
    mul = (uint32_t)((((uint64_t)1 << shift) + (uint64_t)d - 1) / (uint64_t)d);
}

// rank e / Er and node e / En of an expert id 0 <= e < E <= 1024
__host__ __device__ __forceinline__ uint32_t rank_of(const Dims &d, uint32_t e) { return (e * d.er_mul) >> d.er_shift; }
__host__ __device__ __forceinline__ uint32_t node_of(const Dims &d, uint32_t e) { return (e * d.en_mul) >> d.en_shift; }

struct LayoutArgs {
    Dims d;
    const int64_t *topk_idx;
    uint8_t *is_token_in_rank;
    int32_t *tokens_per_rank, *tokens_per_expert, *tokens_per_node, *recv_tokens_per_rank;
    int32_t *rank_slot, *token_major_offset, *expert_slot, *node_slot;
    int64_t *algo_per_rank, *phys_per_rank;
    int32_t *chunk_counts;   // workspace [R * cps, cols]
    int32_t *dev_status;
};

struct RdmaArgs {
    Dims d;
    const int64_t *topk_idx;
    unsigned long long *algo, *phys;
    int32_t *dev_status;
};

struct DispatchArgs {
    Dims d;
    const uint16_t *x;
    const int64_t *topk_idx;
    const int32_t *rank_slot, *expert_slot, *node_slot;
    void *recv;
    float *recv_scales;
    int32_t *dev_status;
    int64_t pieces;          // work units per token row
    int64_t piece_elems;     // elements per piece (multiple of the warp step)
    // destination rows precomputed per token of one source rank (the
    // one-launch small-problem layout + dispatch): dcnt[tl] rows of token
    // src * Tr + tl at dtab[tl * dtab_w ...]; shared memory of that kernel
    const int32_t *dtab, *dcnt;
    int64_t dtab_w;
};

struct CombineArgs {
    Dims d;
    const uint16_t *y;
    const int64_t *topk_idx;
    const float *topk_weights;
    const int32_t *rank_slot, *expert_slot, *node_slot;
    uint16_t *out;
    int32_t *dev_status;
    int64_t pieces;
    int64_t piece_elems;
};

// destination set of the dispatch kernels besides EP_RANK_MAJOR /
// EP_EXPERT_MAJOR: one row per (token, node) of the node-major staging
// buffer (the first hop of the two-level dispatch)
constexpr int kNodeMajor = 2;
// destination set read from DispatchArgs::dtab (rows computed in the same
// kernel by the small-problem layout)
constexpr int kTableDests = 3;

// Small problems for the one-launch layout (one CTA per source rank): every
// source rank in one chunk and at most this many tokens before the last
// source rank, whose CTA counts them itself.
constexpr int kSmallScan = 4096;
__host__ __device__ __forceinline__ bool small_layout(const Dims &d) {
    return d.cps == 1 && (d.R - 1) * d.Tr <= kSmallScan;
}
// Tiny problems, a warp per source rank with no block barrier: at most 32
// tokens per source rank (one per lane) and at most this many before the
// last source rank.
constexpr int kTinyScan = 256;
__host__ __device__ __forceinline__ bool tiny_layout(const Dims &d) {
    return d.Tr <= 32 && (d.R - 1) * d.Tr <= kTinyScan;
}

// dispatch kinds of the fused layout + dispatch kernel
enum { kFusedBulk = 0, kFusedLsu = 1, kFusedFp8 = 2 };

// launchers (return the CUDA error of the launch)
cudaError_t launch_layout(const LayoutArgs &a, int32_t *chunk_counts, cudaStream_t st);
cudaError_t launch_rdma_count(const RdmaArgs &a, cudaStream_t st);
cudaError_t launch_dispatch(int layout, int dtype, const DispatchArgs &a, int grid, cudaStream_t st);
cudaError_t launch_dispatch_bulk(int layout, const DispatchArgs &a, cudaStream_t st);
int dispatch_bulk_piece_bytes();
// picks the row split (a.pieces, a.piece_elems) and the grid, then launches
cudaError_t launch_combine(int layout, CombineArgs &a, cudaStream_t st);
cudaError_t launch_dequant(int layout, const DispatchArgs &a, uint16_t *y, cudaStream_t st);
cudaError_t launch_layout_dispatch(int layout, int mode, const LayoutArgs &la, const DispatchArgs &da,
                                   unsigned *bar, cudaStream_t st);
cudaError_t launch_wait_selftest(unsigned *word, uint32_t polls, int32_t *status, cudaStream_t st);
cudaError_t launch_forward(const DispatchArgs &a, uint16_t *stage, uint16_t *recv, cudaStream_t st);
cudaError_t launch_combine_two_level(const CombineArgs &a, uint16_t *stage, cudaStream_t st);
cudaError_t launch_wire_quant(int layout, int fmt, const DispatchArgs &a, const uint16_t *y, uint8_t *wq, void *ws,
                              cudaStream_t st);
cudaError_t launch_combine_wire(int layout, int fmt, const CombineArgs &a, const uint8_t *wq, const void *ws,
                                cudaStream_t st);

// Sets the message ep_last_error_string() returns on this thread; returns code.
int set_last_error(int code, const char *fmt, ...);

// occupancy-derived grid caps (per device, cached)
int dispatch_grid_cap(int layout, int dtype);
int num_sms();

// Per-device cache of a positive value computed on first use: slots[dev]
// holds it once known.  Host threads may call concurrently (the slots are
// atomics; two threads that both miss compute the same value).  Devices
// with an index of kCacheDevices or more are not cached: compute(dev) runs
// on every call for them.
constexpr int kCacheDevices = 64;
template <typename F>
int cached_per_device(std::atomic<int> *slots, F compute) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    if (dev < 0 || dev >= kCacheDevices) return compute(dev < 0 ? 0 : dev);
    int v = slots[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
    v = compute(dev);
    if (v > 0) slots[dev].store(v, std::memory_order_release);
    return v;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void raise_status(int32_t *st, int bits) {
    if (st) atomicOr(st, bits);
}

// Polls *count (acquire, device scope) until it reaches target, at most
// `polls` times with a short sleep between polls; false if it never did.
__device__ __forceinline__ bool wait_counter_bounded(const unsigned *count, unsigned target, uint32_t polls) {
    for (uint32_t i = 0;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
        if (v >= target) return true;
        if (i >= polls) return false;
        __nanosleep(64);
    }
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}


__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// L2 eviction policy: 0 = default (normal), 1 = evict_first, 2 = evict_last
template <int KIND>
__device__ __forceinline__ uint64_t l2_policy() {
    uint64_t pol = 0;
    if (KIND == 1) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    if (KIND == 2) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte read-only load with an L2 cache policy (pol = 0: no hint)
__device__ __forceinline__ uint4 ld_stream_hint(const void *p, uint64_t pol) {
    uint4 v;
    if (pol == 0) return ld_stream(p);
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// 16-byte store with an L2 cache policy (pol = 0: no hint)
__device__ __forceinline__ void st_v4_hint(void *p, const uint4 &v, uint64_t pol) {
    if (pol == 0) {
        asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
        return;
    }
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void st_v4(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// bf16 pair (packed in a u32, element 0 in the low half) -> two floats
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// two floats -> bf16 pair, round to nearest even, element 0 in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// two floats -> two e4m3 codes, nearest even, saturating; element 0 low byte
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace ep
