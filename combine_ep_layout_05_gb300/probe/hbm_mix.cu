// HBM bandwidth bound for the dispatch's traffic mix on this GPU.
//
// The rank-major dispatch of the prefill workload (8 ranks x 4096 tokens,
// hidden 7168 bf16, top-8 of 256 experts) reads each 14 KB token row once
// and writes it to ~5.3 destination rows: 16% reads, 84% writes.  The copy
// bandwidth the roofline normally uses is a 50:50 stream.  This program
// measures, with plain streaming kernels and no layout work, what HBM
// sustains for that mix: each token row read once and written to its
// destinations (to consecutive rows, and to the dispatch's own scattered
// rows), next to a pure write, a pure read and a 1:1 copy stream, with
// 16- and 32-byte accesses and 2, 4 and 8 CTAs of 256 threads per SM.
// Destinations: per token, the distinct ranks of 8 distinct experts drawn
// uniformly from 256 (32 per rank), compacted per (destination, source) in
// token order, as the layout assigns them.
// Prints one JSON line; same_mix_bound_gbs is the best mix figure.
// Build: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 hbm_mix.cu -o hbm_mix
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>

#include <cuda_runtime.h>

#define CK(x)                                                                             \
    do {                                                                                  \
        cudaError_t e_ = (x);                                                             \
        if (e_ != cudaSuccess) {                                                          \
            fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
            exit(1);                                                                      \
        }                                                                                 \
    } while (0)

namespace {

constexpr int kRowBytes = 7168 * 2;

template <int B>
struct Vec;
template <>
struct Vec<16> {
    uint32_t v[4];
};
template <>
struct Vec<32> {
    uint32_t v[8];
};

__device__ __forceinline__ void ld(const void *p, Vec<16> &r) {
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3])
                 : "l"(p));
}
__device__ __forceinline__ void ld(const void *p, Vec<32> &r) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]), "=r"(r.v[4]), "=r"(r.v[5]),
                   "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p));
}
__device__ __forceinline__ void st(void *p, const Vec<16> &r) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.v[0]), "r"(r.v[1]), "r"(r.v[2]),
                 "r"(r.v[3])
                 : "memory");
}
__device__ __forceinline__ void st(void *p, const Vec<32> &r) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r.v[0]), "r"(r.v[1]),
                 "r"(r.v[2]), "r"(r.v[3]), "r"(r.v[4]), "r"(r.v[5]), "r"(r.v[6]), "r"(r.v[7])
                 : "memory");
}

// a warp per row; lane c moves bytes [c*B, c*B + B) of every 32*B-byte step
template <int B>
__global__ void write_rows(char *y, int64_t nrows) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    Vec<B> v;
    for (int i = 0; i < B / 4; ++i) v.v[i] = lane + i;
    for (int64_t r = w0; r < nrows; r += nw)
        for (int c = lane * B; c < kRowBytes; c += 32 * B) st(y + r * kRowBytes + c, v);
}

template <int B>
__global__ void read_rows(const char *x, int64_t nrows, uint32_t *sink) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    uint32_t acc = 0;
    for (int64_t r = w0; r < nrows; r += nw)
        for (int c = lane * B; c < kRowBytes; c += 64 * B) {
            Vec<B> a, b;
            ld(x + r * kRowBytes + c, a);
            const bool second = c + 32 * B < kRowBytes;
            if (second) ld(x + r * kRowBytes + c + 32 * B, b);
            acc ^= a.v[0] ^ (second ? b.v[1] : 0u);
        }
    if (acc == 0x9e3779b9u) sink[0] = acc;   // keeps the loads
}

// token row r read once, written to dst[r * 8 + i] for each i with dst >= 0
template <int B>
__global__ void mix_rows(const char *x, char *y, const int32_t *dst, int64_t nrows) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = w0; r < nrows; r += nw) {
        const int32_t mine = lane < 8 ? dst[r * 8 + lane] : -1;
        for (int c = lane * B; c < kRowBytes; c += 64 * B) {
            Vec<B> a, b;
            ld(x + r * kRowBytes + c, a);
            const bool second = c + 32 * B < kRowBytes;
            if (second) ld(x + r * kRowBytes + c + 32 * B, b);
            for (int i = 0; i < 8; ++i) {
                const int32_t d = __shfl_sync(0xffffffffu, mine, i);
                if (d < 0) continue;
                st(y + (int64_t)d * kRowBytes + c, a);
                if (second) st(y + (int64_t)d * kRowBytes + c + 32 * B, b);
            }
        }
    }
}

template <typename F>
float time_ms(F launch, int reps) {
    cudaEvent_t a, b;
    CK(cudaEventCreate(&a));
    CK(cudaEventCreate(&b));
    for (int i = 0; i < 3; ++i) launch();
    CK(cudaGetLastError());
    CK(cudaEventRecord(a));
    for (int i = 0; i < reps; ++i) launch();
    CK(cudaEventRecord(b));
    CK(cudaEventSynchronize(b));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, a, b));
    CK(cudaEventDestroy(a));
    CK(cudaEventDestroy(b));
    return ms / reps;
}

}  // namespace

int main() {
    const int R = 8, Tr = 4096, T = R * Tr, E = 256, k = 8, Er = E / R;
    const int64_t cap = (int64_t)R * R * Tr;
    // destinations of every token: distinct ranks of k distinct uniform experts
    std::mt19937_64 rng(12345);
    std::vector<int32_t> scatter((size_t)T * 8, -1), contiguous((size_t)T * 8, -1), one((size_t)T * 8, -1);
    std::vector<int32_t> count((size_t)R * R, 0);
    int64_t D = 0;
    for (int t = 0; t < T; ++t) {
        const int src = t / Tr;
        bool expert[E] = {false}, rank[R] = {false};
        for (int chosen = 0; chosen < k;) {
            const int e = (int)(rng() % E);
            if (!expert[e]) {
                expert[e] = true;
                rank[e / Er] = true;
                ++chosen;
            }
        }
        int j = 0;
        for (int r = 0; r < R; ++r)
            if (rank[r]) {
                scatter[(size_t)t * 8 + j] = (r * R + src) * Tr + count[(size_t)src * R + r]++;
                contiguous[(size_t)t * 8 + j] = (int32_t)D++;
                ++j;
            }
        one[(size_t)t * 8] = t;
    }
    char *x, *y;
    int32_t *d_scatter, *d_contig, *d_one;
    uint32_t *sink;
    CK(cudaMalloc(&x, (size_t)T * kRowBytes));
    CK(cudaMalloc(&y, (size_t)cap * kRowBytes));
    const size_t mb = scatter.size() * sizeof(int32_t);
    CK(cudaMalloc(&d_scatter, mb));
    CK(cudaMalloc(&d_contig, mb));
    CK(cudaMalloc(&d_one, mb));
    CK(cudaMalloc(&sink, 4));
    CK(cudaMemcpy(d_scatter, scatter.data(), mb, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_contig, contiguous.data(), mb, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_one, one.data(), mb, cudaMemcpyHostToDevice));
    CK(cudaMemset(x, 1, (size_t)T * kRowBytes));
    CK(cudaMemset(y, 0, (size_t)cap * kRowBytes));
    int sms = 0;
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));

    const double rb = kRowBytes, mix_bytes = (double)(T + D) * rb;
    double best_w = 0, best_r = 0, best_c = 0, best_mc = 0, best_ms = 0;
    char rows_json[4096];
    int pos = 0;
    auto run = [&](auto tag, int per_sm) {
        constexpr int B = decltype(tag)::value;
        const int grid = sms * per_sm, blk = 256, reps = 10;
        const float w = time_ms([&] { write_rows<B><<<grid, blk>>>(y, D); }, reps);
        const float r = time_ms([&] { read_rows<B><<<grid, blk>>>(y, D, sink); }, reps);
        const float c = time_ms([&] { mix_rows<B><<<grid, blk>>>(x, y, d_one, T); }, reps);
        const float mc = time_ms([&] { mix_rows<B><<<grid, blk>>>(x, y, d_contig, T); }, reps);
        const float ms = time_ms([&] { mix_rows<B><<<grid, blk>>>(x, y, d_scatter, T); }, reps);
        const double gw = D * rb / (w * 1e6), gr = D * rb / (r * 1e6), gc = 2.0 * T * rb / (c * 1e6);
        const double gmc = mix_bytes / (mc * 1e6), gms = mix_bytes / (ms * 1e6);
        best_w = gw > best_w ? gw : best_w;
        best_r = gr > best_r ? gr : best_r;
        best_c = gc > best_c ? gc : best_c;
        best_mc = gmc > best_mc ? gmc : best_mc;
        best_ms = gms > best_ms ? gms : best_ms;
        pos += snprintf(rows_json + pos, sizeof rows_json - pos,
                        "%s{\"bytes_per_access\": %d, \"ctas_per_sm\": %d, \"write\": %.1f, \"read\": %.1f, "
                        "\"copy\": %.1f, \"mix_contiguous\": %.1f, \"mix_scatter\": %.1f}",
                        pos ? ", " : "", B, per_sm, gw, gr, gc, gmc, gms);
    };
    for (int per_sm : {2, 4, 8}) {
        run(std::integral_constant<int, 16>{}, per_sm);
        run(std::integral_constant<int, 32>{}, per_sm);
    }
    CK(cudaDeviceSynchronize());
    const double bound = best_mc > best_ms ? best_mc : best_ms;
    printf("{\"tokens\": %d, \"rows_written\": %lld, \"row_bytes\": %d, \"mix_bytes\": %.0f, \"unit\": \"GB/s\", "
           "\"write\": %.1f, \"read\": %.1f, \"copy\": %.1f, \"mix_contiguous\": %.1f, \"mix_scatter\": %.1f, "
           "\"same_mix_bound_gbs\": %.1f, \"variants\": [%s]}\n",
           T, (long long)D, kRowBytes, mix_bytes, best_w, best_r, best_c, best_mc, best_ms, bound, rows_json);
    return 0;
}
