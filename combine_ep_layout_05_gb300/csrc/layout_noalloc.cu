// ep_layout_noalloc: ep_layout with its scratch in a static device array.
//
// Some callers cannot allocate device memory when they need the layout:
// code that runs inside a host framework whose allocator owns all device
// memory (an inference server or a plugin that pre-reserves the GPU and
// forbids allocations outside its pools), or latency-critical paths where a
// cudaMalloc, which may synchronise the device, is not acceptable.  This
// entry point needs no workspace from them: its scratch lives in a
// file-scope __device__ array that every GPU loading the library holds until
// the process exits.  Inputs and outputs are still the caller's buffers.
#include <mutex>

#include "ep_internal.cuh"

namespace {

constexpr size_t kScratchBytes = EP_LAYOUT_NOALLOC_MAX_SCRATCH_BYTES;

// One copy per device that loads this library.  Device code could name it
// directly; host code must not pass its name to a kernel (on the host the
// name is a stand-in, not a device address): the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_layout_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[64] = {nullptr};   // device address of g_layout_scratch, per device

// Resolves the scratch array's device address for the current device once
// (the first call on each device does this).
int scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= 64) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (e != cudaSuccess) return (int)e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return 0;
}

}  // namespace

extern "C" int ep_layout_noalloc(const ep_problem *p, const int64_t *topk_idx, uint8_t *is_token_in_rank,
                                 int32_t *tokens_per_rank, int32_t *tokens_per_expert, int32_t *tokens_per_node,
                                 int32_t *recv_tokens_per_rank, int32_t *rank_slot, int32_t *token_major_offset,
                                 int32_t *expert_slot, int32_t *node_slot, int64_t *algo_per_rank,
                                 int64_t *physical_exact_per_rank, int32_t *dev_status, ep_stream_t stream) {
    // 0 for a problem ep_layout rejects; it then reports the reason itself
    const size_t need = ep_layout_workspace_bytes(p);
    if (need > kScratchBytes)
        return ep::set_last_error(EP_ERR_INVALID_ARG,
                                  "ep_layout_noalloc: this problem needs %zu bytes of layout scratch, more than the "
                                  "%zu-byte static scratch; use ep_layout with a caller-allocated workspace",
                                  need, kScratchBytes);
    void *scratch = nullptr;
    if (need > 0) {
        const int e = scratch_for_current_device(&scratch);
        if (e)
            return ep::set_last_error(EP_ERR_CUDA, "ep_layout_noalloc: cudaGetSymbolAddress: %s",
                                      cudaGetErrorString((cudaError_t)e));
    }
    // The scratch holds per-chunk counts; the layout's first kernel writes
    // every entry its second kernel reads, so nothing has to start at zero.
    return ep_layout(p, topk_idx, is_token_in_rank, tokens_per_rank, tokens_per_expert, tokens_per_node,
                     recv_tokens_per_rank, rank_slot, token_major_offset, expert_slot, node_slot, algo_per_rank,
                     physical_exact_per_rank, scratch, kScratchBytes, dev_status, stream);
}
