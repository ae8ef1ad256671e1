/*
 * ep.h - MoE expert-parallel dispatch layout, dispatch and combine on one GPU.
 *
 * The R expert-parallel ranks (and N = R / G nodes of G GPUs) are logical
 * partitions of one GPU's memory.  Token t belongs to source rank
 * src = t / Tr, where Tr = T / R tokens per rank.  Expert e lives on rank
 * e / (E / R) and on node e / (E / N).
 *
 * Conventions shared by every entry point
 *  - Every pointer argument is a device pointer that the caller allocated
 *    and owns, unless stated otherwise.  The library allocates nothing and
 *    keeps no pointer after the call returns.  Inputs are not modified.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns EP_OK once its kernels are enqueued.
 *  - EP_ERR_INVALID_ARG: the sizes describe no problem, or a required
 *    pointer is NULL or misaligned.  Nothing was enqueued.
 *  - EP_ERR_CUDA: a launch failed; nothing more of the call was enqueued.
 *  - ep_last_error_string() describes the last failure on this thread.
 *  - Errors found by the kernels (bad expert id, repeated expert id, slot
 *    out of range, a bounded wait on an asynchronous copy that ran out:
 *    EP_STATUS_TIMEOUT) are OR-ed as EP_STATUS_* bits into *dev_status, an int32
 *    in device memory that the caller zeroes and reads after synchronising
 *    (ep_get_status does both the synchronisation and the read, and
 *    returns EP_ERR_DEVICE when a bit is set).  dev_status may be NULL
 *    (errors then go unreported).  Entries that raise a status bit are
 *    skipped; the rest of the call completes.
 *
 * Problem limits: 1 <= k <= 32, 1 <= R <= 64, E % R == 0, E <= 1024,
 * R % G == 0, T % R == 0, H % 8 == 0 (H % 128 == 0 for FP8), N <= 64.
 *
 * The pages this follows: "MORI-EP Benchmark" (rocm.github.io/mori),
 * "MoE-EP Benchmark" (moe_ep_benchmark README) and MSCCL++ PR #860 "ep(bench):
 * add mscclpp high-throughput (rank-major) backend to the unified Python EP
 * benchmark".
 */
#ifndef EP_H
#define EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, so callers need no CUDA header. */
typedef struct CUstream_st *ep_stream_t;

typedef struct ep_problem {
    int64_t num_tokens;    /* T: tokens of all source ranks, T = R * Tr      */
    int64_t hidden;        /* H: channels per token                          */
    int64_t num_topk;      /* k: routed experts per token                    */
    int64_t num_experts;   /* E                                              */
    int64_t num_ranks;     /* R: logical expert-parallel ranks               */
    int64_t gpus_per_node; /* G: ranks per logical node; N = R / G           */
} ep_problem;

enum { EP_OK = 0, EP_ERR_INVALID_ARG = 1, EP_ERR_CUDA = 2, EP_ERR_DEVICE = 3 };
enum { EP_STATUS_BAD_EXPERT = 1, EP_STATUS_DUP_EXPERT = 2, EP_STATUS_BAD_SLOT = 4, EP_STATUS_TIMEOUT = 8 };
enum { EP_RANK_MAJOR = 0, EP_EXPERT_MAJOR = 1 };
enum { EP_BF16 = 0, EP_FP8_E4M3 = 1 };
enum { EP_WIRE_MXFP8 = 1, EP_WIRE_NVFP4 = 2 };

/* Text for the last failing call on this thread ("" if none). */
const char *ep_last_error_string(void);

/*
 * ep_get_status - waits for `stream` and reads the status word the kernels
 * OR their EP_STATUS_* bits into.  Host-side; it synchronises, so it must
 * not be called while `stream` is being captured into a CUDA graph.
 *
 * dev_status: the device int32 passed to the earlier calls (not NULL).
 * status_out: host int32 that receives the word (may be NULL).
 * Returns EP_OK when no bit is set, EP_ERR_DEVICE when one is (the bits
 * say which errors the kernels found: their entries were skipped, the rest
 * of the work completed), EP_ERR_CUDA when the synchronisation or the read
 * failed (an earlier kernel fault surfaces here), EP_ERR_INVALID_ARG for a
 * NULL or misaligned dev_status.  The word is not cleared.
 */
int ep_get_status(const int32_t *dev_status, int32_t *status_out, ep_stream_t stream);

/*
 * Rows of the receive buffer: R * R * Tr for EP_RANK_MAJOR
 * ([R dst][R src][Tr] rows), E * R * Tr for EP_EXPERT_MAJOR
 * ([E][R src][Tr] rows).  Returns -1 for an invalid problem or layout.
 * Host-only.
 */
int64_t ep_recv_rows(const ep_problem *p, int layout);

/* Bytes of device workspace ep_layout needs (0 for an invalid problem). */
size_t ep_layout_workspace_bytes(const ep_problem *p);

/*
 * ep_layout - dispatch layout of all R source ranks.
 * ("MORI-EP Benchmark", print_bw_values.py: expert -> rank map
 * topk_idx // (E / R) with -1 kept, per-token dedupe, per-rank counts and
 * their all-reduce; MSCCL++ PR #860: get_dispatch_layout, and the
 * rank-major commit, whose slots are grouped by source rank.)
 *
 * In:  topk_idx [T, k] int64, -1 = no expert.  An id outside [-1, E) raises
 *      EP_STATUS_BAD_EXPERT and is ignored; an id repeated in a row raises
 *      EP_STATUS_DUP_EXPERT and only its first occurrence counts.
 * Out (each may be NULL to skip it):
 *   is_token_in_rank     [T, R] uint8   1 if t goes to rank r
 *   tokens_per_rank      [R, R] int32   [src, dst] tokens src sends to dst
 *   tokens_per_expert    [R, E] int32   [src, e] tokens src routes to e
 *   tokens_per_node      [R, N] int32   [src, n] tokens src sends to node n
 *   recv_tokens_per_rank [R]    int32   column sums of tokens_per_rank
 *   rank_slot            [T, R] int32   rank-major slot: number of earlier
 *                                       tokens of the same source that go to
 *                                       r; -1 if t does not go to r
 *   token_major_offset   [T, R] int32   compacted offset on r: number of
 *                                       earlier tokens of any source that go
 *                                       to r; -1 likewise
 *   expert_slot          [T, k] int32   expert-major slot of entry j: number
 *                                       of earlier tokens of the same source
 *                                       routed to the same expert; -1 for
 *                                       ignored entries
 *   node_slot            [T, N] int32   node-major slot: number of earlier
 *                                       tokens of the same source that go to
 *                                       node n; -1 if t does not go to n
 *   algo_per_rank        [R]    int64   RDMA token counts, as
 *   physical_exact_per_rank [R] int64   ep_rdma_token_count defines them
 *                                       (sums of tokens_per_node rows)
 * workspace: device scratch of at least ep_layout_workspace_bytes(p) bytes,
 *   16-byte aligned; overwritten (problems of one chunk per source rank,
 *   Tr <= 256 with at most 4096 tokens before the last source rank, run in
 *   one kernel that does not touch it).
 * One kernel for such small problems (a block per source rank), otherwise
 * two (per-chunk histogram, then scan and slots); no cross-block waiting.
 * All outputs are exact integers, identical on every run.
 */
int ep_layout(const ep_problem *p, const int64_t *topk_idx,
              uint8_t *is_token_in_rank, int32_t *tokens_per_rank,
              int32_t *tokens_per_expert, int32_t *tokens_per_node,
              int32_t *recv_tokens_per_rank, int32_t *rank_slot,
              int32_t *token_major_offset, int32_t *expert_slot,
              int32_t *node_slot, int64_t *algo_per_rank,
              int64_t *physical_exact_per_rank, void *workspace,
              size_t workspace_bytes, int32_t *dev_status, ep_stream_t stream);

/*
 * ep_rdma_token_count - RDMA token counts per source rank.
 * ("MORI-EP Benchmark", "Bandwidth Computation" / "Algo BW vs Physical BW"
 * / "Why DeepEP and Mori RDMA token counts are equivalent".)
 *
 * algo_per_rank[src]           [R] int64: unique (token, node) pairs of src's
 *                              tokens, node = e / (E / N), local node included
 * physical_exact_per_rank[src] [R] int64: the same without src's own node
 *                              (src / G); may be NULL
 * Both outputs are overwritten (zeroed on `stream` first).
 */
int ep_rdma_token_count(const ep_problem *p, const int64_t *topk_idx,
                        int64_t *algo_per_rank, int64_t *physical_exact_per_rank,
                        int32_t *dev_status, ep_stream_t stream);

/*
 * The page's physical estimate algo * (N - 1) / N, the integer product
 * first ("MORI-EP Benchmark", "Algo BW vs Physical BW").  Host-only.
 */
double ep_rdma_physical_formula(int64_t algo_tokens, int64_t num_nodes);

/*
 * ep_dispatch - scatter token rows into the receive buffer.
 * (MSCCL++ PR #860: intranode/throughput dispatch, the rank-major layout
 * "fixed [num_ranks, max_tokens_per_rank, hidden] slot grouped by source
 * rank", and the low-latency expert-major dispatch with optional FP8;
 * "MORI-EP Benchmark", print_bw_values.py: FP8 carries one byte per element
 * and a 4-byte scale per 128 channels.)
 *
 * EP_RANK_MAJOR: one copy of x[t] per rank r with rank_slot[t, r] >= 0, to
 *   row (r * R + src) * Tr + rank_slot[t, r].  Reads rank_slot; topk_idx and
 *   expert_slot are not read (may be NULL).
 * EP_EXPERT_MAJOR: one copy per entry j with expert e = topk_idx[t, j] in
 *   [0, E) and expert_slot[t, j] >= 0, to row (e * R + src) * Tr +
 *   expert_slot[t, j].  rank_slot is not read (may be NULL).
 * A slot >= Tr or < -1 raises EP_STATUS_BAD_SLOT and that copy is skipped.
 *
 * EP_BF16:     x [T, H] bf16 -> recv [rows, H] bf16.  recv_scales unused.
 * EP_FP8_E4M3: per token and 128-channel block b: amax = max |x|,
 *   s = amax / 448, inv = 448 / amax (0 if amax = 0, at most FLT_MAX), each an
 *   fp32 division rounded to nearest; q = e4m3(x * inv), the fp32 product
 *   rounded to nearest, converted with round-to-nearest-even, saturating at
 *   +-448.  recv [rows, H] uint8 codes, recv_scales [rows, H / 128] fp32.
 *   The row is cast once; every copy is identical.
 * Rows the layout does not name are not written.  x and recv: 16-byte
 * aligned.
 */
int ep_dispatch(const ep_problem *p, int layout, int dtype, const uint16_t *x,
                const int64_t *topk_idx, const int32_t *rank_slot,
                const int32_t *expert_slot, void *recv, float *recv_scales,
                int32_t *dev_status, ep_stream_t stream);

/* Bytes of device workspace ep_layout_dispatch needs (0 for an invalid problem). */
size_t ep_layout_dispatch_workspace_bytes(const ep_problem *p);

/*
 * ep_layout_dispatch - ep_layout and ep_dispatch in one launch.
 * (MSCCL++ PR #860: the layout ("notify") paired with the dispatch that
 * consumes it.)
 *
 * Arguments and outputs are those of ep_layout followed by ep_dispatch on
 * the same stream, and the outputs are identical.  The dispatch reads the
 * slots the layout writes, so rank_slot (EP_RANK_MAJOR) or expert_slot
 * (EP_EXPERT_MAJOR) must not be NULL.  workspace: at least
 * ep_layout_dispatch_workspace_bytes(p) bytes, 16-byte aligned.
 * Problems ep_layout runs in one kernel, with a register-copy or FP8
 * dispatch: one launch without grid barriers, several CTAs per source rank
 * that each build that rank's layout in shared memory (the first also
 * writes the outputs) and dispatch a share of its tokens.  Otherwise one
 * cooperative launch whose CTAs meet at two grid barriers (layout histogram
 * -> slots -> dispatch); the barriers poll a bounded number of times and
 * raise EP_STATUS_TIMEOUT instead of waiting forever.  If the GPU cannot
 * hold the grid resident, the call runs ep_layout and ep_dispatch instead.
 */
int ep_layout_dispatch(const ep_problem *p, int layout, int dtype, const uint16_t *x,
                       const int64_t *topk_idx, uint8_t *is_token_in_rank,
                       int32_t *tokens_per_rank, int32_t *tokens_per_expert,
                       int32_t *tokens_per_node, int32_t *recv_tokens_per_rank,
                       int32_t *rank_slot, int32_t *token_major_offset,
                       int32_t *expert_slot, int32_t *node_slot, int64_t *algo_per_rank,
                       int64_t *physical_exact_per_rank, void *recv, float *recv_scales,
                       void *workspace, size_t workspace_bytes, int32_t *dev_status,
                       ep_stream_t stream);

/*
 * ep_combine - weighted top-k gather back to token order.
 * ("MORI-EP Benchmark", "Combine": the reverse of dispatch with the same
 * byte counts; MSCCL++ PR #860: combine consumes the receiver-side layout,
 * and in the expert-major layout each expert returns one copy per token.)
 *
 * out[t] = bf16( sum over kept entries j of topk_weights[t, j] * y[row] ),
 * summed in fp32 and rounded to nearest-even once.  row is the rank-major
 * row of (t, e_j / (E / R)) (several experts on one rank share it: their
 * weights are summed in j order and the row is read once) or the
 * expert-major row of (t, e_j).  Entries are kept as in ep_layout.  A token
 * with no kept entry gets zeros.
 * y [rows, H] bf16 (the receive-buffer shape); topk_weights [T, k] fp32;
 * out [T, H] bf16.  y and out 16-byte aligned.
 */
int ep_combine(const ep_problem *p, int layout, const uint16_t *y,
               const int64_t *topk_idx, const float *topk_weights,
               const int32_t *rank_slot, const int32_t *expert_slot,
               uint16_t *out, int32_t *dev_status, ep_stream_t stream);

/*
 * Two-level (node-forwarding) dispatch and combine.  ("MORI-EP Benchmark",
 * "Bandwidth Computation": the inter-node fabric carries one copy per
 * (token, destination node) - the "algo" count - which the node forwards
 * to the token's ranks; "Combine": the reverse with the same byte counts.)
 *
 * stage: the node-major staging buffer [N][R src][Tr][H] bf16
 * (ep_stage_rows(p) rows); row (n * R + src) * Tr + node_slot[t, n].
 * ep_dispatch_two_level: hop 1 copies x[t] to the staging row of every node
 *   the token goes to; hop 2 copies each staging row to the rank-major rows
 *   of the token's ranks in that node (reading the staging row).  recv ends
 *   up identical to ep_dispatch(EP_RANK_MAJOR, EP_BF16).
 * ep_combine_two_level: hop 1 writes, per (token, node), the weighted sum of
 *   the node's rank rows (fp32, weights of one rank summed in j order),
 *   rounded to bf16, into the staging row; hop 2 writes out[t] = bf16(sum of
 *   the token's node partials in ascending node order), fp32.
 * rank_slot and node_slot from ep_layout; y [R * R * Tr, H] bf16.
 */
int64_t ep_stage_rows(const ep_problem *p);
int ep_dispatch_two_level(const ep_problem *p, const uint16_t *x, const int32_t *rank_slot,
                          const int32_t *node_slot, uint16_t *stage, uint16_t *recv,
                          int32_t *dev_status, ep_stream_t stream);
int ep_combine_two_level(const ep_problem *p, const uint16_t *y, const int64_t *topk_idx,
                         const float *topk_weights, const int32_t *rank_slot,
                         const int32_t *node_slot, uint16_t *stage, uint16_t *out,
                         int32_t *dev_status, ep_stream_t stream);

/*
 * Low-precision combine wire formats ("MoE-EP Benchmark", environment
 * reference, MEGA_COMBINE_DTYPE: mxfp8 = 32 e4m3 values x one e8m0 scale,
 * nvfp4 = 16 e2m1 values x one bf16 scale).  The expert side casts its bf16
 * output rows once (ep_combine_quantize); combine reads the cast rows
 * (ep_combine_wire), moving 1.03 (mxfp8) or 0.625 (nvfp4) bytes per channel
 * instead of 2.
 *
 * EP_WIRE_MXFP8: per block of 32 channels, X = floor(log2(amax)) - 8
 *   clamped to [-127, 127], stored as the e8m0 code X + 127 (0 when
 *   amax = 0); codes e4m3(v * 2^-X), nearest-even, saturating at 448.
 *   wq [rows, H] uint8, wscales [rows, H / 32] uint8.  H % 32 == 0.
 * EP_WIRE_NVFP4: per block of 16 channels, s = bf16(fp32(amax / 6));
 *   inv = fp32(1 / s) (0 when s = 0); codes e2m1(v * inv), nearest-even,
 *   saturating at 6; two codes per byte, channel 2i in the low nibble.
 *   wq [rows, H / 2] uint8, wscales [rows, H / 16] bf16.  H % 16 == 0.
 *
 * ep_combine_quantize casts the rows the dispatch handle names (as
 * ep_dequant_fp8 does) from y [rows, H] bf16.  ep_combine_wire is
 * ep_combine with y[row] replaced by the decoded wire row (exact in fp32):
 * out[t] = bf16(sum_j w_tj * decode(row)), fp32 accumulation.
 * wq and out 16-byte aligned.
 */
int ep_combine_quantize(const ep_problem *p, int layout, int fmt, const uint16_t *y,
                        const int64_t *topk_idx, const int32_t *rank_slot,
                        const int32_t *expert_slot, uint8_t *wq, void *wscales,
                        ep_stream_t stream);
int ep_combine_wire(const ep_problem *p, int layout, int fmt, const uint8_t *wq,
                    const void *wscales, const int64_t *topk_idx,
                    const float *topk_weights, const int32_t *rank_slot,
                    const int32_t *expert_slot, uint16_t *out, int32_t *dev_status,
                    ep_stream_t stream);

/*
 * ep_dequant_fp8 - the identity expert for an FP8 receive buffer (test and
 * benchmark harness: expert output y = input): y = bf16(decode(q) * s),
 * the exact product rounded once to nearest-even.  Only the rows the
 * dispatch handle names are written: the rank-major rows of rank_slot, or
 * the expert-major rows of (topk_idx, expert_slot), as in ep_dispatch.
 * recv [rows, H] uint8, recv_scales [rows, H / 128] fp32, y [rows, H] bf16.
 */
int ep_dequant_fp8(const ep_problem *p, int layout, const int64_t *topk_idx,
                   const int32_t *rank_slot, const int32_t *expert_slot,
                   const uint8_t *recv, const float *recv_scales, uint16_t *y,
                   ep_stream_t stream);

/*
 * ep_layout_noalloc - ep_layout for callers that cannot allocate device
 * memory.  (No counterpart on the pages: an addition of this library.)
 *
 * Who needs it: code that runs inside a host framework whose allocator owns
 * the device memory (an inference server or a plugin that reserves the GPU
 * up front and forbids allocations outside its pools), and latency-critical
 * callers for which a cudaMalloc, which may synchronise the device, is not
 * acceptable.  Such callers cannot provide ep_layout's workspace.
 *
 * Same arguments, outputs and semantics as ep_layout, without `workspace`:
 * the scratch is a file-scope __device__ array of
 * EP_LAYOUT_NOALLOC_MAX_SCRATCH_BYTES bytes, held by every GPU that loads
 * the library until the process exits.  The call allocates nothing (no
 * cudaMalloc / cudaFree, no allocating library routine).
 *  - Limit: problems whose ep_layout_workspace_bytes() exceeds the array are
 *    rejected with EP_ERR_INVALID_ARG and a message saying so; the limit
 *    covers R * ceil(Tr / 256) * (R + E + N) * 4 <= 4 MiB, e.g. 8 or 16
 *    ranks x 8192 tokens/rank with 256 experts.
 *  - Set-up: the first call on each device, with that device current,
 *    resolves the array's device address (cudaGetSymbolAddress) and keeps
 *    it together with the id of the device's CUDA context; make that first
 *    call before any stream capture.  If the device's context later changes
 *    (after cudaDeviceReset the runtime creates a new one, into which the
 *    library's module is loaded again), the next call resolves the address
 *    again rather than using the old one.  A failure there returns
 *    EP_ERR_CUDA.
 *  - Sharing: every call on a device uses the same array, which keeps the
 *    previous call's contents.  Nothing in it needs to start at zero (the
 *    first layout kernel writes every entry the second reads).  Calls that
 *    overlap on the GPU (for example on two streams at once) race on the
 *    array and give wrong results: order them.
 */
#define EP_LAYOUT_NOALLOC_MAX_SCRATCH_BYTES ((size_t)4 << 20)

int ep_layout_noalloc(const ep_problem *p, const int64_t *topk_idx,
                      uint8_t *is_token_in_rank, int32_t *tokens_per_rank,
                      int32_t *tokens_per_expert, int32_t *tokens_per_node,
                      int32_t *recv_tokens_per_rank, int32_t *rank_slot,
                      int32_t *token_major_offset, int32_t *expert_slot,
                      int32_t *node_slot, int64_t *algo_per_rank,
                      int64_t *physical_exact_per_rank, int32_t *dev_status,
                      ep_stream_t stream);

/*
 * ep_selftest_wait_timeout - failure-detection self-test (no counterpart on
 * the pages).  Runs the two bounded waits the kernels use - the grid
 * barrier's counter poll and the bulk copies' mbarrier poll - against a
 * counter nothing increments and an mbarrier whose bytes never arrive, each
 * limited to `polls` polls (at most 2^20).  Both must give up: words[0]
 * gets bit 0 (counter wait) and bit 1 (mbarrier wait), *dev_status gets
 * EP_STATUS_TIMEOUT, and the GPU context stays usable.  words: 2 uint32 of
 * device memory (zeroed by the call).
 */
int ep_selftest_wait_timeout(uint32_t *words, uint32_t polls, int32_t *dev_status,
                             ep_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_H */
