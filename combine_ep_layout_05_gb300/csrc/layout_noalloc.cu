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
#include <cuda.h>

#include <mutex>

#include "ep_internal.cuh"

namespace {

constexpr size_t kScratchBytes = EP_LAYOUT_NOALLOC_MAX_SCRATCH_BYTES;

// One copy per device that loads this library.  Device code could name it
// directly; host code must not pass its name to a kernel (on the host the
// name is a stand-in, not a device address): the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_layout_scratch[kScratchBytes];

// The device address of g_layout_scratch is a property of the CUDA context
// the module was loaded into.  It is resolved once per device and kept with
// the unique id of that context; when the device's current context is a
// different one (the device was reset and the runtime created a new primary
// context, which loads the module afresh), the address is resolved again
// instead of reusing a stale one.  The two driver calls that read the
// context id come through the runtime's driver entry-point table, so the
// library needs no link against the driver library.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

struct ScratchSlot {
    void *ptr = nullptr;
    unsigned long long ctx_id = 0;
};

std::mutex g_mu;
ScratchSlot g_slot[64];   // per device
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_entry_points_tried = false;

// Unique id of the current context, or 0 if there is none (or the driver
// entry points are unavailable, in which case the address is resolved on
// every call).  Called with g_mu held.
unsigned long long current_context_id() {
    if (!g_entry_points_tried) {
        g_entry_points_tried = true;
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            g_ctx_get_current = (CtxGetCurrentFn)f1;
            g_ctx_get_id = (CtxGetIdFn)f2;
        }
        (void)cudaGetLastError();
    }
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// The scratch array's device address on the current device: resolved on
// the first call on each device (and again after the device's context has
// changed).
int scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= 64) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    ScratchSlot &s = g_slot[dev];
    const unsigned long long id = current_context_id();
    if (!s.ptr || id == 0 || id != s.ctx_id) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (e != cudaSuccess) return (int)e;
        s.ptr = p;
        // the symbol lookup makes the device's primary context current if
        // no context was: read the id after it
        s.ctx_id = id ? id : current_context_id();
    }
    *out = s.ptr;
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
