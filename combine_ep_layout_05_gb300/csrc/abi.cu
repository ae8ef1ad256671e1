// C-ABI entry points: argument checks, problem sizes, launches.
// The semantics of every entry point are documented in include/ep.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "ep_internal.cuh"

// bf16 dispatch goes through the bulk-copy engine from this many tokens on;
// below it (decode and low-latency sizes) 16-byte register copies spread
// over more warps finish sooner.
#ifndef EP_DISPATCH_BULK_MIN_TOKENS
#define EP_DISPATCH_BULK_MIN_TOKENS 2048
#endif

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *where) {
    return fail(EP_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Fills d from p; returns false (with the message set) if p describes no problem.
bool make_dims(const ep_problem *p, ep::Dims &d) {
    if (!p) return fail(EP_ERR_INVALID_ARG, "problem is NULL"), false;
    d.T = p->num_tokens;
    d.H = p->hidden;
    d.k = p->num_topk;
    d.E = p->num_experts;
    d.R = p->num_ranks;
    d.G = p->gpus_per_node;
    if (d.T < 0 || d.H < 8 || d.H % 8 || d.k < 1 || d.k > ep::kMaxTopk || d.E < 1 ||
        d.E > ep::kMaxExperts || d.R < 1 || d.R > ep::kMaxRanks || d.G < 1)
        return fail(EP_ERR_INVALID_ARG,
                    "sizes out of range (T=%lld H=%lld k=%lld E=%lld R=%lld G=%lld): need T>=0, H>=8, H%%8==0, "
                    "1<=k<=32, 1<=E<=1024, 1<=R<=64, G>=1",
                    (long long)d.T, (long long)d.H, (long long)d.k, (long long)d.E, (long long)d.R,
                    (long long)d.G),
               false;
    if (d.E % d.R) return fail(EP_ERR_INVALID_ARG, "num_experts %% num_ranks != 0"), false;
    if (d.R % d.G) return fail(EP_ERR_INVALID_ARG, "num_ranks %% gpus_per_node != 0"), false;
    if (d.T % d.R) return fail(EP_ERR_INVALID_ARG, "num_tokens %% num_ranks != 0"), false;
    d.N = d.R / d.G;
    d.Er = d.E / d.R;
    d.En = d.E / d.N;
    d.Tr = d.T / d.R;
    if (d.Tr > INT32_MAX) return fail(EP_ERR_INVALID_ARG, "tokens per rank exceed int32"), false;
    d.cps = (d.Tr + ep::kChunk - 1) / ep::kChunk;
    d.cols = d.R + d.E + d.N;
    ep::div_magic(d.Er, d.er_mul, d.er_shift);
    ep::div_magic(d.En, d.en_mul, d.en_shift);
    return true;
}

// Splits a token row into pieces when there are too few tokens to give every
// warp slot of the GPU a unit of work.  granule: elements one warp step covers.
void pick_pieces(const ep::Dims &d, int64_t granule, int64_t &pieces, int64_t &piece_elems) {
    const int64_t target = (int64_t)ep::num_sms() * 32;   // warps to keep busy
    const int64_t max_pieces = (d.H + granule - 1) / granule;
    int64_t want = d.T > 0 ? (target + d.T - 1) / d.T : 1;
    if (want > max_pieces) want = max_pieces;
    if (want < 1) want = 1;
    int64_t per = (d.H + want - 1) / want;
    per = (per + granule - 1) / granule * granule;
    piece_elems = per;
    pieces = (d.H + per - 1) / per;
}

int64_t unit_grid(int64_t units, int cap) {
    int64_t g = (units + 7) / 8;
    if (g > cap) g = cap;
    return g < 1 ? 1 : g;
}

}  // namespace

namespace ep {
int set_last_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}
}  // namespace ep

extern "C" {

const char *ep_last_error_string(void) { return g_err; }

int ep_get_status(const int32_t *dev_status, int32_t *status_out, ep_stream_t stream) {
    g_err[0] = 0;
    if (!dev_status || !aligned(dev_status, 4)) return fail(EP_ERR_INVALID_ARG, "dev_status NULL or misaligned");
    cudaStream_t st = (cudaStream_t)stream;
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, dev_status, sizeof word, cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    if (e) return cuda_fail(e, "ep_get_status");
    if (status_out) *status_out = word;
    if (word) return fail(EP_ERR_DEVICE, "the kernels reported status bits 0x%x", (unsigned)word);
    return EP_OK;
}

int64_t ep_recv_rows(const ep_problem *p, int layout) {
    ep::Dims d;
    if (!make_dims(p, d)) return -1;
    if (layout == EP_RANK_MAJOR) return d.R * d.R * d.Tr;
    if (layout == EP_EXPERT_MAJOR) return d.E * d.R * d.Tr;
    fail(EP_ERR_INVALID_ARG, "unknown layout %d", layout);
    return -1;
}

size_t ep_layout_workspace_bytes(const ep_problem *p) {
    ep::Dims d;
    if (!make_dims(p, d)) return 0;
    const size_t b = (size_t)(d.R * d.cps * d.cols) * sizeof(int32_t);
    return (b + 255) / 256 * 256;
}

double ep_rdma_physical_formula(int64_t algo_tokens, int64_t num_nodes) {
    if (num_nodes < 1) return 0.0;
    return (double)(algo_tokens * (num_nodes - 1)) / (double)num_nodes;
}

int ep_layout(const ep_problem *p, const int64_t *topk_idx, uint8_t *is_token_in_rank,
              int32_t *tokens_per_rank, int32_t *tokens_per_expert, int32_t *tokens_per_node,
              int32_t *recv_tokens_per_rank, int32_t *rank_slot, int32_t *token_major_offset,
              int32_t *expert_slot, int32_t *node_slot, int64_t *algo_per_rank,
              int64_t *physical_exact_per_rank, void *workspace, size_t workspace_bytes, int32_t *dev_status,
              ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (d.T == 0) {
        // nothing routed: counts are zero
        cudaError_t e = cudaSuccess;
        if (tokens_per_rank && !e) e = cudaMemsetAsync(tokens_per_rank, 0, d.R * d.R * 4, st);
        if (tokens_per_expert && !e) e = cudaMemsetAsync(tokens_per_expert, 0, d.R * d.E * 4, st);
        if (tokens_per_node && !e) e = cudaMemsetAsync(tokens_per_node, 0, d.R * d.N * 4, st);
        if (recv_tokens_per_rank && !e) e = cudaMemsetAsync(recv_tokens_per_rank, 0, d.R * 4, st);
        if (algo_per_rank && !e) e = cudaMemsetAsync(algo_per_rank, 0, d.R * 8, st);
        if (physical_exact_per_rank && !e) e = cudaMemsetAsync(physical_exact_per_rank, 0, d.R * 8, st);
        return e ? cuda_fail(e, "ep_layout memset") : EP_OK;
    }
    if (!topk_idx || !aligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx NULL or misaligned");
    if (!workspace || !aligned(workspace, 16))
        return fail(EP_ERR_INVALID_ARG, "workspace NULL or not 16-byte aligned");
    if (workspace_bytes < ep_layout_workspace_bytes(p))
        return fail(EP_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes,
                    ep_layout_workspace_bytes(p));
    const void *i32s[] = {tokens_per_rank, tokens_per_expert, tokens_per_node, recv_tokens_per_rank,
                          rank_slot, token_major_offset, expert_slot, node_slot, dev_status};
    for (const void *q : i32s)
        if (!aligned(q, 4)) return fail(EP_ERR_INVALID_ARG, "int32 output not 4-byte aligned");
    if (!aligned(algo_per_rank, 8) || !aligned(physical_exact_per_rank, 8))
        return fail(EP_ERR_INVALID_ARG, "int64 output not 8-byte aligned");
    ep::LayoutArgs a{};
    a.d = d;
    a.topk_idx = topk_idx;
    a.is_token_in_rank = is_token_in_rank;
    a.tokens_per_rank = tokens_per_rank;
    a.tokens_per_expert = tokens_per_expert;
    a.tokens_per_node = tokens_per_node;
    a.recv_tokens_per_rank = recv_tokens_per_rank;
    a.rank_slot = rank_slot;
    a.token_major_offset = token_major_offset;
    a.expert_slot = expert_slot;
    a.node_slot = node_slot;
    a.algo_per_rank = algo_per_rank;
    a.phys_per_rank = physical_exact_per_rank;
    a.chunk_counts = (int32_t *)workspace;
    a.dev_status = dev_status;
    cudaError_t e = ep::launch_layout(a, a.chunk_counts, st);
    return e ? cuda_fail(e, "ep_layout launch") : EP_OK;
}

int ep_rdma_token_count(const ep_problem *p, const int64_t *topk_idx, int64_t *algo_per_rank,
                        int64_t *physical_exact_per_rank, int32_t *dev_status, ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    if (!algo_per_rank || !aligned(algo_per_rank, 8) || !aligned(physical_exact_per_rank, 8))
        return fail(EP_ERR_INVALID_ARG, "algo_per_rank NULL or outputs misaligned");
    if (d.T > 0 && (!topk_idx || !aligned(topk_idx, 8)))
        return fail(EP_ERR_INVALID_ARG, "topk_idx NULL or misaligned");
    if (!aligned(dev_status, 4)) return fail(EP_ERR_INVALID_ARG, "dev_status misaligned");
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(algo_per_rank, 0, d.R * 8, st);
    if (!e && physical_exact_per_rank) e = cudaMemsetAsync(physical_exact_per_rank, 0, d.R * 8, st);
    if (e) return cuda_fail(e, "ep_rdma_token_count memset");
    if (d.T == 0) return EP_OK;
    ep::RdmaArgs a{};
    a.d = d;
    a.topk_idx = topk_idx;
    a.algo = (unsigned long long *)algo_per_rank;
    a.phys = (unsigned long long *)physical_exact_per_rank;
    a.dev_status = dev_status;
    e = ep::launch_rdma_count(a, st);
    return e ? cuda_fail(e, "ep_rdma_token_count launch") : EP_OK;
}

}  // extern "C"

namespace {

// Checks ep_dispatch's arguments and fills a (everything but the launch);
// mode: the kernel that will run.  Returns EP_OK or the error code.
int prepare_dispatch(const ep::Dims &d, int layout, int dtype, const uint16_t *x, const int64_t *topk_idx,
                     const int32_t *rank_slot, const int32_t *expert_slot, void *recv, float *recv_scales,
                     int32_t *dev_status, ep::DispatchArgs &a, int &mode) {
    if (layout != EP_RANK_MAJOR && layout != EP_EXPERT_MAJOR)
        return fail(EP_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (dtype != EP_BF16 && dtype != EP_FP8_E4M3) return fail(EP_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (dtype == EP_FP8_E4M3 && d.H % 128) return fail(EP_ERR_INVALID_ARG, "FP8 needs hidden %% 128 == 0");
    if (d.T == 0) return EP_OK;
    if (!x || !aligned(x, 16)) return fail(EP_ERR_INVALID_ARG, "x NULL or not 16-byte aligned");
    if (!recv || !aligned(recv, 16)) return fail(EP_ERR_INVALID_ARG, "recv NULL or not 16-byte aligned");
    if (layout == EP_RANK_MAJOR && (!rank_slot || !aligned(rank_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "rank_slot NULL or misaligned");
    if (layout == EP_EXPERT_MAJOR && (!topk_idx || !aligned(topk_idx, 8) || !expert_slot || !aligned(expert_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "topk_idx / expert_slot NULL or misaligned");
    if (dtype == EP_FP8_E4M3 && (!recv_scales || !aligned(recv_scales, 4)))
        return fail(EP_ERR_INVALID_ARG, "recv_scales NULL or misaligned");
    if (!aligned(dev_status, 4)) return fail(EP_ERR_INVALID_ARG, "dev_status misaligned");
    a.d = d;
    a.x = x;
    a.topk_idx = topk_idx;
    a.rank_slot = rank_slot;
    a.expert_slot = expert_slot;
    a.recv = recv;
    a.recv_scales = recv_scales;
    a.dev_status = dev_status;
    if (dtype == EP_BF16 && d.T >= EP_DISPATCH_BULK_MIN_TOKENS) {
        // bulk-copy path: whole rows, or the fewest pieces that fit one
        // shared-memory buffer each
        const int64_t maxe = ep::dispatch_bulk_piece_bytes() / 2;
        a.pieces = (d.H + maxe - 1) / maxe;
        a.piece_elems = ((d.H + a.pieces - 1) / a.pieces + 7) / 8 * 8;
        a.pieces = (d.H + a.piece_elems - 1) / a.piece_elems;
        mode = ep::kFusedBulk;
    } else {
        pick_pieces(d, dtype == EP_BF16 ? 256 : 512, a.pieces, a.piece_elems);
        mode = dtype == EP_BF16 ? ep::kFusedLsu : ep::kFusedFp8;
    }
    return EP_OK;
}

int launch_prepared_dispatch(int layout, int dtype, int mode, const ep::DispatchArgs &a, cudaStream_t st) {
    cudaError_t e;
    if (mode == ep::kFusedBulk) {
        e = ep::launch_dispatch_bulk(layout, a, st);
    } else {
        const int64_t grid = unit_grid(a.d.T * a.pieces, ep::dispatch_grid_cap(layout, dtype));
        e = ep::launch_dispatch(layout, dtype, a, (int)grid, st);
    }
    return e ? cuda_fail(e, "ep_dispatch launch") : EP_OK;
}

}  // namespace

extern "C" {

int ep_dispatch(const ep_problem *p, int layout, int dtype, const uint16_t *x, const int64_t *topk_idx,
                const int32_t *rank_slot, const int32_t *expert_slot, void *recv, float *recv_scales,
                int32_t *dev_status, ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    ep::DispatchArgs a{};
    int mode = 0;
    const int rc = prepare_dispatch(d, layout, dtype, x, topk_idx, rank_slot, expert_slot, recv, recv_scales,
                                    dev_status, a, mode);
    if (rc != EP_OK || d.T == 0) return rc;
    return launch_prepared_dispatch(layout, dtype, mode, a, (cudaStream_t)stream);
}

size_t ep_layout_dispatch_workspace_bytes(const ep_problem *p) {
    const size_t w = ep_layout_workspace_bytes(p);
    return w ? w + 256 : 0;
}

int ep_layout_dispatch(const ep_problem *p, int layout, int dtype, const uint16_t *x, const int64_t *topk_idx,
                       uint8_t *is_token_in_rank, int32_t *tokens_per_rank, int32_t *tokens_per_expert,
                       int32_t *tokens_per_node, int32_t *recv_tokens_per_rank, int32_t *rank_slot,
                       int32_t *token_major_offset, int32_t *expert_slot, int32_t *node_slot,
                       int64_t *algo_per_rank, int64_t *physical_exact_per_rank, void *recv, float *recv_scales,
                       void *workspace, size_t workspace_bytes, int32_t *dev_status, ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t lw = ep_layout_workspace_bytes(p);
    if (d.T == 0)
        return ep_layout(p, topk_idx, is_token_in_rank, tokens_per_rank, tokens_per_expert, tokens_per_node,
                         recv_tokens_per_rank, rank_slot, token_major_offset, expert_slot, node_slot,
                         algo_per_rank, physical_exact_per_rank, workspace, workspace_bytes, dev_status, stream);
    if (!topk_idx || !aligned(topk_idx, 8)) return fail(EP_ERR_INVALID_ARG, "topk_idx NULL or misaligned");
    if (!workspace || !aligned(workspace, 16))
        return fail(EP_ERR_INVALID_ARG, "workspace NULL or not 16-byte aligned");
    if (workspace_bytes < ep_layout_dispatch_workspace_bytes(p))
        return fail(EP_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes,
                    ep_layout_dispatch_workspace_bytes(p));
    const void *i32s[] = {tokens_per_rank, tokens_per_expert, tokens_per_node, recv_tokens_per_rank,
                          rank_slot, token_major_offset, expert_slot, node_slot, dev_status};
    for (const void *q : i32s)
        if (!aligned(q, 4)) return fail(EP_ERR_INVALID_ARG, "int32 output not 4-byte aligned");
    if (!aligned(algo_per_rank, 8) || !aligned(physical_exact_per_rank, 8))
        return fail(EP_ERR_INVALID_ARG, "int64 output not 8-byte aligned");
    ep::DispatchArgs da{};
    int mode = 0;
    int rc = prepare_dispatch(d, layout, dtype, x, topk_idx, rank_slot, expert_slot, recv, recv_scales, dev_status,
                              da, mode);
    if (rc != EP_OK) return rc;
    ep::LayoutArgs la{};
    la.d = d;
    la.topk_idx = topk_idx;
    la.is_token_in_rank = is_token_in_rank;
    la.tokens_per_rank = tokens_per_rank;
    la.tokens_per_expert = tokens_per_expert;
    la.tokens_per_node = tokens_per_node;
    la.recv_tokens_per_rank = recv_tokens_per_rank;
    la.rank_slot = rank_slot;
    la.token_major_offset = token_major_offset;
    la.expert_slot = expert_slot;
    la.node_slot = node_slot;
    la.algo_per_rank = algo_per_rank;
    la.phys_per_rank = physical_exact_per_rank;
    la.chunk_counts = (int32_t *)workspace;
    la.dev_status = dev_status;
    unsigned *bar = (unsigned *)((char *)workspace + lw);
    cudaError_t e = ep::launch_layout_dispatch(layout, mode, la, da, bar, st);
    if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorNotSupported) {
        // no room for a resident grid: the same work as two calls
        (void)cudaGetLastError();
        rc = ep_layout(p, topk_idx, is_token_in_rank, tokens_per_rank, tokens_per_expert, tokens_per_node,
                       recv_tokens_per_rank, rank_slot, token_major_offset, expert_slot, node_slot, algo_per_rank,
                       physical_exact_per_rank, workspace, workspace_bytes, dev_status, stream);
        if (rc != EP_OK) return rc;
        return launch_prepared_dispatch(layout, dtype, mode, da, st);
    }
    return e ? cuda_fail(e, "ep_layout_dispatch launch") : EP_OK;
}

int ep_combine(const ep_problem *p, int layout, const uint16_t *y, const int64_t *topk_idx,
               const float *topk_weights, const int32_t *rank_slot, const int32_t *expert_slot,
               uint16_t *out, int32_t *dev_status, ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    if (layout != EP_RANK_MAJOR && layout != EP_EXPERT_MAJOR)
        return fail(EP_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (d.T == 0) return EP_OK;
    if (!y || !aligned(y, 16)) return fail(EP_ERR_INVALID_ARG, "y NULL or not 16-byte aligned");
    if (!out || !aligned(out, 16)) return fail(EP_ERR_INVALID_ARG, "out NULL or not 16-byte aligned");
    if (!topk_idx || !aligned(topk_idx, 8) || !topk_weights || !aligned(topk_weights, 4))
        return fail(EP_ERR_INVALID_ARG, "topk_idx / topk_weights NULL or misaligned");
    if (layout == EP_RANK_MAJOR && (!rank_slot || !aligned(rank_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "rank_slot NULL or misaligned");
    if (layout == EP_EXPERT_MAJOR && (!expert_slot || !aligned(expert_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "expert_slot NULL or misaligned");
    if (!aligned(dev_status, 4)) return fail(EP_ERR_INVALID_ARG, "dev_status misaligned");
    ep::CombineArgs a{};
    a.d = d;
    a.y = y;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.rank_slot = rank_slot;
    a.expert_slot = expert_slot;
    a.out = out;
    a.dev_status = dev_status;
    cudaError_t e = ep::launch_combine(layout, a, (cudaStream_t)stream);
    return e ? cuda_fail(e, "ep_combine launch") : EP_OK;
}

int ep_dequant_fp8(const ep_problem *p, int layout, const int64_t *topk_idx, const int32_t *rank_slot,
                   const int32_t *expert_slot, const uint8_t *recv, const float *recv_scales, uint16_t *y,
                   ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    if (layout != EP_RANK_MAJOR && layout != EP_EXPERT_MAJOR)
        return fail(EP_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (d.H % 128) return fail(EP_ERR_INVALID_ARG, "FP8 needs hidden %% 128 == 0");
    if (d.T == 0) return EP_OK;
    if (!recv || !aligned(recv, 16) || !recv_scales || !aligned(recv_scales, 4) || !y || !aligned(y, 16))
        return fail(EP_ERR_INVALID_ARG, "recv / recv_scales / y NULL or misaligned");
    if (layout == EP_RANK_MAJOR && (!rank_slot || !aligned(rank_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "rank_slot NULL or misaligned");
    if (layout == EP_EXPERT_MAJOR && (!topk_idx || !aligned(topk_idx, 8) || !expert_slot || !aligned(expert_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "topk_idx / expert_slot NULL or misaligned");
    ep::DispatchArgs a{};
    a.d = d;
    a.x = nullptr;
    a.topk_idx = topk_idx;
    a.rank_slot = rank_slot;
    a.expert_slot = expert_slot;
    a.recv = const_cast<uint8_t *>(recv);
    a.recv_scales = const_cast<float *>(recv_scales);
    a.dev_status = nullptr;
    cudaError_t e = ep::launch_dequant(layout, a, y, (cudaStream_t)stream);
    return e ? cuda_fail(e, "ep_dequant_fp8 launch") : EP_OK;
}

int ep_selftest_wait_timeout(uint32_t *words, uint32_t polls, int32_t *dev_status, ep_stream_t stream) {
    g_err[0] = 0;
    if (!words || !aligned(words, 4) || !aligned(dev_status, 4))
        return fail(EP_ERR_INVALID_ARG, "words NULL or misaligned");
    if (polls > (1u << 20)) return fail(EP_ERR_INVALID_ARG, "polls must be at most 2^20 for a self-test");
    cudaError_t e = cudaMemsetAsync(words, 0, 2 * sizeof(uint32_t), (cudaStream_t)stream);
    if (!e) e = ep::launch_wait_selftest((unsigned *)words, polls, dev_status, (cudaStream_t)stream);
    return e ? cuda_fail(e, "ep_selftest_wait_timeout launch") : EP_OK;
}

int ep_combine_quantize(const ep_problem *p, int layout, int fmt, const uint16_t *y, const int64_t *topk_idx,
                        const int32_t *rank_slot, const int32_t *expert_slot, uint8_t *wq, void *wscales,
                        ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    if (layout != EP_RANK_MAJOR && layout != EP_EXPERT_MAJOR)
        return fail(EP_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (fmt != EP_WIRE_MXFP8 && fmt != EP_WIRE_NVFP4) return fail(EP_ERR_INVALID_ARG, "unknown wire format %d", fmt);
    if (d.H % (fmt == EP_WIRE_MXFP8 ? 32 : 16))
        return fail(EP_ERR_INVALID_ARG, "hidden must be a multiple of the wire block");
    if (d.T == 0) return EP_OK;
    if (!y || !aligned(y, 16) || !wq || !aligned(wq, 16) || !wscales || !aligned(wscales, 2))
        return fail(EP_ERR_INVALID_ARG, "y / wq / wscales NULL or misaligned");
    if (layout == EP_RANK_MAJOR && (!rank_slot || !aligned(rank_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "rank_slot NULL or misaligned");
    if (layout == EP_EXPERT_MAJOR && (!topk_idx || !aligned(topk_idx, 8) || !expert_slot || !aligned(expert_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "topk_idx / expert_slot NULL or misaligned");
    ep::DispatchArgs a{};
    a.d = d;
    a.x = nullptr;
    a.topk_idx = topk_idx;
    a.rank_slot = rank_slot;
    a.expert_slot = expert_slot;
    a.recv = nullptr;
    a.recv_scales = nullptr;
    a.dev_status = nullptr;
    pick_pieces(d, 512, a.pieces, a.piece_elems);
    cudaError_t e = ep::launch_wire_quant(layout, fmt, a, y, wq, wscales, (cudaStream_t)stream);
    return e ? cuda_fail(e, "ep_combine_quantize launch") : EP_OK;
}

int ep_combine_wire(const ep_problem *p, int layout, int fmt, const uint8_t *wq, const void *wscales,
                    const int64_t *topk_idx, const float *topk_weights, const int32_t *rank_slot,
                    const int32_t *expert_slot, uint16_t *out, int32_t *dev_status, ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    if (layout != EP_RANK_MAJOR && layout != EP_EXPERT_MAJOR)
        return fail(EP_ERR_INVALID_ARG, "unknown layout %d", layout);
    if (fmt != EP_WIRE_MXFP8 && fmt != EP_WIRE_NVFP4) return fail(EP_ERR_INVALID_ARG, "unknown wire format %d", fmt);
    if (d.H % (fmt == EP_WIRE_MXFP8 ? 32 : 16))
        return fail(EP_ERR_INVALID_ARG, "hidden must be a multiple of the wire block");
    if (d.T == 0) return EP_OK;
    if (!wq || !aligned(wq, 16) || !wscales || !aligned(wscales, 2) || !out || !aligned(out, 16))
        return fail(EP_ERR_INVALID_ARG, "wq / wscales / out NULL or misaligned");
    if (!topk_idx || !aligned(topk_idx, 8) || !topk_weights || !aligned(topk_weights, 4))
        return fail(EP_ERR_INVALID_ARG, "topk_idx / topk_weights NULL or misaligned");
    if (layout == EP_RANK_MAJOR && (!rank_slot || !aligned(rank_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "rank_slot NULL or misaligned");
    if (layout == EP_EXPERT_MAJOR && (!expert_slot || !aligned(expert_slot, 4)))
        return fail(EP_ERR_INVALID_ARG, "expert_slot NULL or misaligned");
    if (!aligned(dev_status, 4)) return fail(EP_ERR_INVALID_ARG, "dev_status misaligned");
    ep::CombineArgs a{};
    a.d = d;
    a.y = nullptr;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.rank_slot = rank_slot;
    a.expert_slot = expert_slot;
    a.out = out;
    a.dev_status = dev_status;
    pick_pieces(d, 512, a.pieces, a.piece_elems);
    cudaError_t e = ep::launch_combine_wire(layout, fmt, a, wq, wscales, (cudaStream_t)stream);
    return e ? cuda_fail(e, "ep_combine_wire launch") : EP_OK;
}

int64_t ep_stage_rows(const ep_problem *p) {
    ep::Dims d;
    if (!make_dims(p, d)) return -1;
    return d.N * d.R * d.Tr;
}

int ep_dispatch_two_level(const ep_problem *p, const uint16_t *x, const int32_t *rank_slot,
                          const int32_t *node_slot, uint16_t *stage, uint16_t *recv, int32_t *dev_status,
                          ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    if (d.T == 0) return EP_OK;
    if (!x || !aligned(x, 16) || !stage || !aligned(stage, 16) || !recv || !aligned(recv, 16))
        return fail(EP_ERR_INVALID_ARG, "x / stage / recv NULL or not 16-byte aligned");
    if (!rank_slot || !aligned(rank_slot, 4) || !node_slot || !aligned(node_slot, 4))
        return fail(EP_ERR_INVALID_ARG, "rank_slot / node_slot NULL or misaligned");
    if (!aligned(dev_status, 4)) return fail(EP_ERR_INVALID_ARG, "dev_status misaligned");
    cudaStream_t st = (cudaStream_t)stream;
    // hop 1: one copy per (token, node) into the node-major staging buffer
    ep::DispatchArgs a{};
    a.d = d;
    a.x = x;
    a.rank_slot = rank_slot;
    a.node_slot = node_slot;
    a.recv = stage;
    a.dev_status = dev_status;
    cudaError_t e;
    if (d.T >= EP_DISPATCH_BULK_MIN_TOKENS) {
        const int64_t maxe = ep::dispatch_bulk_piece_bytes() / 2;
        a.pieces = (d.H + maxe - 1) / maxe;
        a.piece_elems = ((d.H + a.pieces - 1) / a.pieces + 7) / 8 * 8;
        a.pieces = (d.H + a.piece_elems - 1) / a.piece_elems;
        e = ep::launch_dispatch_bulk(ep::kNodeMajor, a, st);
    } else {
        pick_pieces(d, 256, a.pieces, a.piece_elems);
        e = ep::launch_dispatch(ep::kNodeMajor, EP_BF16, a, (int)unit_grid(d.T * a.pieces,
                                ep::dispatch_grid_cap(ep::kNodeMajor, EP_BF16)), st);
    }
    if (e) return cuda_fail(e, "ep_dispatch_two_level hop 1");
    // hop 2: each staged row to the token's ranks inside the node
    pick_pieces(d, 256, a.pieces, a.piece_elems);
    e = ep::launch_forward(a, stage, recv, st);
    return e ? cuda_fail(e, "ep_dispatch_two_level hop 2") : EP_OK;
}

int ep_combine_two_level(const ep_problem *p, const uint16_t *y, const int64_t *topk_idx,
                         const float *topk_weights, const int32_t *rank_slot, const int32_t *node_slot,
                         uint16_t *stage, uint16_t *out, int32_t *dev_status, ep_stream_t stream) {
    g_err[0] = 0;
    ep::Dims d;
    if (!make_dims(p, d)) return EP_ERR_INVALID_ARG;
    if (d.T == 0) return EP_OK;
    if (!y || !aligned(y, 16) || !stage || !aligned(stage, 16) || !out || !aligned(out, 16))
        return fail(EP_ERR_INVALID_ARG, "y / stage / out NULL or not 16-byte aligned");
    if (!topk_idx || !aligned(topk_idx, 8) || !topk_weights || !aligned(topk_weights, 4))
        return fail(EP_ERR_INVALID_ARG, "topk_idx / topk_weights NULL or misaligned");
    if (!rank_slot || !aligned(rank_slot, 4) || !node_slot || !aligned(node_slot, 4))
        return fail(EP_ERR_INVALID_ARG, "rank_slot / node_slot NULL or misaligned");
    if (!aligned(dev_status, 4)) return fail(EP_ERR_INVALID_ARG, "dev_status misaligned");
    ep::CombineArgs a{};
    a.d = d;
    a.y = y;
    a.topk_idx = topk_idx;
    a.topk_weights = topk_weights;
    a.rank_slot = rank_slot;
    a.node_slot = node_slot;
    a.out = out;
    a.dev_status = dev_status;
    pick_pieces(d, 256, a.pieces, a.piece_elems);
    cudaError_t e = ep::launch_combine_two_level(a, stage, (cudaStream_t)stream);
    return e ? cuda_fail(e, "ep_combine_two_level launch") : EP_OK;
}

}  // extern "C"
