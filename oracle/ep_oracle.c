/*
 * CPU oracle for MoE expert-parallel dispatch layout, dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, sequential
 * statement of what the GPU path computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Sources (page title, section):
 *  - "MORI-EP Benchmark", print_bw_values.py: expert -> rank map
 *    rank_idx = topk_idx // (num_experts // num_ranks), -1 kept as -1,
 *    per-token dedupe; per-rank send counts (rank_idx == i).sum(); global
 *    receive count by all-reduce of the per-rank counts; expert -> node map
 *    rdma_idx = topk_idx // (num_experts // num_nodes), dedupe, count of
 *    non-empty entries ("algo" RDMA tokens, local node included) and the
 *    same count with the local node masked out ("physical").
 *  - "MORI-EP Benchmark", "Algo BW vs Physical BW": physical tokens =
 *    algo tokens x (num_nodes - 1) / num_nodes.
 *  - "MORI-EP Benchmark", "Why DeepEP and Mori RDMA token counts are
 *    equivalent": both count unique (token, destination-node) pairs.
 *  - "MORI-EP Benchmark", print_bw_values.py byte counts: FP8 payload is one
 *    byte per element plus a 4-byte scale per 128 channels.
 *  - MSCCL++ PR #860, rank-major commit: each dispatched token lands in a
 *    fixed [num_ranks, max_tokens_per_rank, hidden] slot grouped by source
 *    rank; the token-major layout uses the compacted prefix offset.
 *  - MSCCL++ PR #860, low-latency combine accounting: one copy per
 *    (token, expert) in the expert-major layout.
 *
 * Readings where the pages leave a step open (each restated where used):
 *  - slots are compacted positions in ascending source-token order;
 *  - an expert id outside [-1, E) is flagged and ignored; a repeated expert
 *    id in one row is flagged and only its first occurrence counts;
 *  - FP8: amax over each 128-channel block, s = amax / 448 and
 *    inv = 448 / amax in fp32 (inv = 0 when amax = 0, capped at FLT_MAX),
 *    q = e4m3(x * inv) with round-to-nearest-even and saturation to +-448;
 *  - combine sums w_j * y_row in fp64 and rounds once to bf16.
 *
 * bf16 values are uint16 bit patterns; e4m3 values are uint8 codes.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* status bits (the same contract the library documents for dev_status) */
#define OR_BAD_EXPERT 1
#define OR_DUP_EXPERT 2
#define OR_BAD_SLOT 4
/* return value for arguments that do not describe a problem */
#define OR_BAD_ARGS (-1)

#define OR_RANK_MAJOR 0
#define OR_EXPERT_MAJOR 1
#define OR_BF16 0
#define OR_FP8 1

/* ------------------------------------------------------------------ */
/* number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 bits -> value (exact). */
static double bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

double oracle_bf16_to_double(uint16_t b) { return bf16_value(b); }

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double y) {
    double f = floor(y);
    double d = y - f;
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/*
 * double -> bf16 with a single round-to-nearest-even.
 * bf16: 1 sign, 8 exponent (bias 127), 7 fraction bits; subnormal step 2^-133.
 */
uint16_t oracle_bf16_from_double(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a < ldexp(1.0, -126)) {                 /* subnormal range */
        double n = round_half_even(ldexp(a, 133));  /* 0..128; 128 = min normal */
        return (uint16_t)(sign | (uint16_t)n);
    }
    int ex;
    frexp(a, &ex);                              /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                             /* a in [2^e, 2^(e+1)) */
    double n = round_half_even(ldexp(a, 7 - e));    /* 128..256 */
    if (n == 256.0) { n = 128.0; e += 1; }
    if (e > 127) return (uint16_t)(sign | 0x7F80);  /* rounds to infinity */
    return (uint16_t)(sign | (uint16_t)((e + 127) << 7) | (uint16_t)(n - 128.0));
}

/*
 * OCP 8-bit floating point, E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN, largest finite 448 (S.1111.110),
 * subnormals m/8 * 2^-6.
 */
double oracle_e4m3_decode(uint8_t c) {
    int s = c >> 7, E = (c >> 3) & 15, M = c & 7;
    double v;
    if (E == 15 && M == 7) return NAN;
    if (E == 0) v = ldexp((double)M, -9);          /* M/8 * 2^-6 */
    else v = ldexp(8.0 + M, E - 10);               /* (1 + M/8) * 2^(E-7) */
    return s ? -v : v;
}

/* float -> e4m3, nearest-even, values beyond the largest finite saturate. */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                      /* subnormal step 2^-9 */
        double n = round_half_even(ldexp(a, 9)); /* 0..8; 8 = min normal */
        return sign | (uint8_t)n;
    }
    int ex;
    frexp(a, &ex);
    int e = ex - 1;                                /* -6 .. 8 */
    double n = round_half_even(ldexp(a, 3 - e));   /* 8..16 */
    if (n == 16.0) { n = 8.0; e += 1; }
    int E = e + 7, M = (int)n - 8;
    if (E > 15 || (E == 15 && M == 7)) return sign | 0x7E;   /* saturate */
    return sign | (uint8_t)((E << 3) | M);
}

/* ------------------------------------------------------------------ */
/* problem                                                             */
/* ------------------------------------------------------------------ */

static int check_problem(int64_t T, int64_t k, int64_t E, int64_t R, int64_t G) {
    if (T < 0 || k < 1 || k > 32 || E < 1 || R < 1 || R > 64 || G < 1) return 0;
    if (E % R || R % G || T % R) return 0;
    if ((R / G) > 64) return 0;
    return 1;
}

/*
 * The valid experts of token row t, in j order: an id of -1 means "no
 * expert"; any other id outside [0, E) is flagged and ignored; an id seen
 * earlier in the row is flagged and ignored.  valid[j] = 1 for kept entries.
 */
static int row_experts(const int64_t *row, int64_t k, int64_t E, unsigned char *valid) {
    int st = 0;
    for (int64_t j = 0; j < k; ++j) {
        int64_t e = row[j];
        valid[j] = 0;
        if (e == -1) continue;
        if (e < 0 || e >= E) { st |= OR_BAD_EXPERT; continue; }
        int seen = 0;
        for (int64_t i = 0; i < j; ++i)
            if (valid[i] && row[i] == e) seen = 1;
        if (seen) { st |= OR_DUP_EXPERT; continue; }
        valid[j] = 1;
    }
    return st;
}

/*
 * Dispatch layout for all R source ranks at once (token t belongs to source
 * rank src = t / Tr, Tr = T / R).
 *
 *  is_token_in_rank[t, r]   1 if some expert of t lives on rank r = e / (E/R)
 *  tokens_per_rank[src, r]  tokens of src that go to rank r
 *  tokens_per_expert[src,e] tokens of src routed to expert e
 *  tokens_per_node[src, n]  tokens of src that go to node n = e / (E/N)
 *  recv_tokens_per_rank[r]  sum over src of tokens_per_rank[src, r]
 *                           (the all-reduce of the per-rank counts)
 *  rank_slot[t, r]          rank-major slot: number of earlier tokens of the
 *                           same source rank that also go to r; -1 if t does
 *                           not go to r
 *  token_major_offset[t, r] compacted offset on r: number of earlier tokens
 *                           of any source rank that go to r; -1 likewise
 *  expert_slot[t, j]        expert-major slot of entry j: number of earlier
 *                           tokens of the same source rank routed to the
 *                           same expert; -1 for ignored entries
 *  node_slot[t, n]          node-major slot: number of earlier tokens of the
 *                           same source rank that go to node n; -1 if t
 *                           does not go to n
 *
 * Every output pointer may be NULL.  Returns the status bits, or -1 for
 * arguments that describe no problem.
 */
int oracle_layout(int64_t T, int64_t k, int64_t E, int64_t R, int64_t G,
                  const int64_t *topk_idx,
                  uint8_t *is_token_in_rank, int32_t *tokens_per_rank,
                  int32_t *tokens_per_expert, int32_t *tokens_per_node,
                  int32_t *recv_tokens_per_rank, int32_t *rank_slot,
                  int32_t *token_major_offset, int32_t *expert_slot, int32_t *node_slot) {
    if (!check_problem(T, k, E, R, G)) return OR_BAD_ARGS;
    const int64_t N = R / G, Er = E / R, En = E / N, Tr = T / R;
    int st = 0;
    unsigned char valid[32];
    unsigned char *in_rank = calloc((size_t)R, 1);
    unsigned char *in_node = calloc((size_t)N, 1);
    int64_t *seg_rank = calloc((size_t)R, sizeof(int64_t));
    int64_t *glob_rank = calloc((size_t)R, sizeof(int64_t));
    int64_t *seg_exp = calloc((size_t)E, sizeof(int64_t));
    int64_t *seg_node = calloc((size_t)N, sizeof(int64_t));

    for (int64_t src = 0; src < R; ++src) {
        memset(seg_rank, 0, (size_t)R * sizeof(int64_t));
        memset(seg_exp, 0, (size_t)E * sizeof(int64_t));
        memset(seg_node, 0, (size_t)N * sizeof(int64_t));
        for (int64_t t = src * Tr; t < (src + 1) * Tr; ++t) {
            const int64_t *row = topk_idx + t * k;
            st |= row_experts(row, k, E, valid);
            memset(in_rank, 0, (size_t)R);
            memset(in_node, 0, (size_t)N);
            for (int64_t j = 0; j < k; ++j) {
                if (!valid[j]) continue;
                in_rank[row[j] / Er] = 1;      /* rank_idx = topk_idx // (E/R) */
                in_node[row[j] / En] = 1;      /* rdma_idx = topk_idx // (E/N) */
            }
            for (int64_t r = 0; r < R; ++r) {
                if (is_token_in_rank) is_token_in_rank[t * R + r] = in_rank[r];
                int32_t slot = -1, off = -1;
                if (in_rank[r]) {
                    slot = (int32_t)seg_rank[r]++;
                    off = (int32_t)glob_rank[r]++;
                }
                if (rank_slot) rank_slot[t * R + r] = slot;
                if (token_major_offset) token_major_offset[t * R + r] = off;
            }
            for (int64_t n = 0; n < N; ++n) {
                /* node-major slot: earlier tokens of this source going to n */
                if (node_slot) node_slot[t * N + n] = in_node[n] ? (int32_t)seg_node[n] : -1;
                seg_node[n] += in_node[n];
            }
            for (int64_t j = 0; j < k; ++j) {
                int32_t s = -1;
                if (valid[j]) s = (int32_t)seg_exp[row[j]]++;
                if (expert_slot) expert_slot[t * k + j] = s;
            }
        }
        for (int64_t r = 0; r < R; ++r)
            if (tokens_per_rank) tokens_per_rank[src * R + r] = (int32_t)seg_rank[r];
        for (int64_t e = 0; e < E; ++e)
            if (tokens_per_expert) tokens_per_expert[src * E + e] = (int32_t)seg_exp[e];
        for (int64_t n = 0; n < N; ++n)
            if (tokens_per_node) tokens_per_node[src * N + n] = (int32_t)seg_node[n];
    }
    if (recv_tokens_per_rank)
        for (int64_t r = 0; r < R; ++r) recv_tokens_per_rank[r] = (int32_t)glob_rank[r];

    free(in_rank); free(in_node); free(seg_rank); free(glob_rank); free(seg_exp); free(seg_node);
    return st;
}

/*
 * RDMA token counts per source rank.  algo = number of unique
 * (token, destination node) pairs, the local node included; physical_exact =
 * the same with the source's own node (src / G) left out.
 */
int oracle_rdma_token_count(int64_t T, int64_t k, int64_t E, int64_t R, int64_t G,
                            const int64_t *topk_idx, int64_t *algo_per_rank,
                            int64_t *physical_exact_per_rank) {
    if (!check_problem(T, k, E, R, G)) return OR_BAD_ARGS;
    const int64_t N = R / G, En = E / N, Tr = T / R;
    int st = 0;
    unsigned char valid[32];
    unsigned char *in_node = calloc((size_t)N, 1);
    for (int64_t src = 0; src < R; ++src) {
        int64_t algo = 0, phys = 0, my_node = src / G;
        for (int64_t t = src * Tr; t < (src + 1) * Tr; ++t) {
            const int64_t *row = topk_idx + t * k;
            st |= row_experts(row, k, E, valid);
            memset(in_node, 0, (size_t)N);
            for (int64_t j = 0; j < k; ++j)
                if (valid[j]) in_node[row[j] / En] = 1;
            for (int64_t n = 0; n < N; ++n) {
                algo += in_node[n];
                if (n != my_node) phys += in_node[n];
            }
        }
        if (algo_per_rank) algo_per_rank[src] = algo;
        if (physical_exact_per_rank) physical_exact_per_rank[src] = phys;
    }
    free(in_node);
    return st;
}

/* physical = algo x (num_nodes - 1) / num_nodes, the integer product first. */
double oracle_rdma_physical_formula(int64_t algo, int64_t num_nodes) {
    return (double)(algo * (num_nodes - 1)) / (double)num_nodes;
}

/*
 * FP8 cast of one token row: for each 128-channel block b, amax = max |x|,
 * s[b] = amax / 448, inv = 448 / amax (0 when amax = 0, capped at FLT_MAX),
 * q = e4m3(x * inv).  All arithmetic in fp32, each operation rounded to
 * nearest.
 */
void oracle_quant_fp8_row(int64_t H, const uint16_t *x, uint8_t *q, float *s) {
    for (int64_t b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int64_t i = 0; i < 128; ++i) {
            float v = fabsf((float)bf16_value(x[b * 128 + i]));
            if (v > amax) amax = v;
        }
        volatile float sb = amax / 448.0f;
        float inv = 0.0f;
        if (amax > 0.0f) {
            volatile float t = 448.0f / amax;
            inv = t;
            if (inv > FLT_MAX) inv = FLT_MAX;
        }
        s[b] = sb;
        for (int64_t i = 0; i < 128; ++i) {
            volatile float p = (float)bf16_value(x[b * 128 + i]) * inv;
            q[b * 128 + i] = oracle_e4m3_encode(p);
        }
    }
}

/* Destination row of (t, r) in the rank-major buffer [R dst][R src][Tr][H]. */
static int64_t rank_major_row(int64_t r, int64_t src, int64_t Tr, int64_t R, int64_t slot) {
    return (r * R + src) * Tr + slot;
}

/* Destination row of (t, e) in the expert-major buffer [E][R src][Tr][H]. */
static int64_t expert_major_row(int64_t e, int64_t src, int64_t Tr, int64_t R, int64_t slot) {
    return (e * R + src) * Tr + slot;
}

/*
 * Dispatch: copy token row x[t] to every destination row.
 *  rank-major:   one copy per rank r with rank_slot[t, r] >= 0
 *  expert-major: one copy per kept entry j (expert e = topk_idx[t, j]) with
 *                expert_slot[t, j] >= 0
 * bf16 payload: recv is uint16 [rows, H].  FP8 payload: recv is uint8
 * [rows, H] and recv_scales float [rows, H / 128]; the row is cast once and
 * every copy is identical.  A slot outside [-1, Tr) is flagged and skipped.
 * Only tokens t in [t0, t1) are dispatched.
 */
int oracle_dispatch(int64_t T, int64_t H, int64_t k, int64_t E, int64_t R, int64_t G,
                    int layout, int dtype, const uint16_t *x, const int64_t *topk_idx,
                    const int32_t *rank_slot, const int32_t *expert_slot,
                    void *recv, float *recv_scales, int64_t t0, int64_t t1) {
    if (!check_problem(T, k, E, R, G) || H < 1 || H % 8) return OR_BAD_ARGS;
    if (dtype == OR_FP8 && H % 128) return OR_BAD_ARGS;
    if (t0 < 0) t0 = 0;
    if (t1 > T) t1 = T;
    const int64_t Tr = T / R, nb = H / 128;
    int st = 0;
    unsigned char valid[32];
    uint8_t *qrow = malloc((size_t)H);
    float *srow = malloc((size_t)(nb > 0 ? nb : 1) * sizeof(float));
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t src = t / Tr;
        if (dtype == OR_FP8) oracle_quant_fp8_row(H, x + t * H, qrow, srow);
        int64_t ndst = (layout == OR_RANK_MAJOR) ? R : k;
        if (layout == OR_EXPERT_MAJOR) st |= row_experts(topk_idx + t * k, k, E, valid);
        for (int64_t d = 0; d < ndst; ++d) {
            int64_t row;
            int32_t slot;
            if (layout == OR_RANK_MAJOR) {
                slot = rank_slot[t * R + d];
                if (slot == -1) continue;
                if (slot < -1 || slot >= Tr) { st |= OR_BAD_SLOT; continue; }
                row = rank_major_row(d, src, Tr, R, slot);
            } else {
                if (!valid[d]) continue;
                slot = expert_slot[t * k + d];
                if (slot == -1) continue;
                if (slot < -1 || slot >= Tr) { st |= OR_BAD_SLOT; continue; }
                row = expert_major_row(topk_idx[t * k + d], src, Tr, R, slot);
            }
            if (dtype == OR_BF16) {
                memcpy((uint16_t *)recv + row * H, x + t * H, (size_t)H * 2);
            } else {
                memcpy((uint8_t *)recv + row * H, qrow, (size_t)H);
                memcpy(recv_scales + row * nb, srow, (size_t)nb * sizeof(float));
            }
        }
    }
    free(qrow); free(srow);
    return st;
}

/*
 * Identity expert for an FP8 payload: y = bf16(decode(q) * s), the product
 * taken exactly in fp64 and rounded once.  Only live rows are touched: in
 * segment (d, src) the first count[src, d] rows, where count is
 * tokens_per_rank [R, R] (rank-major, d = destination rank) or
 * tokens_per_expert [R, E] (expert-major, d = expert).
 */
int oracle_dequant_fp8(int64_t T, int64_t H, int64_t E, int64_t R, int layout,
                       const int32_t *counts, const uint8_t *q, const float *s, uint16_t *y) {
    if (R < 1 || T % R || H % 128) return OR_BAD_ARGS;
    const int64_t Tr = T / R, nb = H / 128;
    const int64_t ndst = (layout == OR_RANK_MAJOR) ? R : E;
    for (int64_t d = 0; d < ndst; ++d)
        for (int64_t src = 0; src < R; ++src) {
            int64_t c = counts[src * ndst + d];
            for (int64_t i = 0; i < c && i < Tr; ++i) {
                int64_t row = (d * R + src) * Tr + i;
                for (int64_t h = 0; h < H; ++h) {
                    double v = oracle_e4m3_decode(q[row * H + h]) * (double)s[row * nb + h / 128];
                    y[row * H + h] = oracle_bf16_from_double(v);
                }
            }
        }
    return 0;
}

/*
 * Weighted combine back to token order, for tokens t in [t0, t1):
 *   out[t] = sum over kept entries j of w[t, j] * y[row(t, j)]
 * with row(t, j) the rank-major row of (t, e_j / (E/R)) or the expert-major
 * row of (t, e_j).  The sum is taken in fp64 in j order; out_bf16 gets one
 * round-to-nearest-even of it, out_f64 (may be NULL) the fp64 value.  Rows
 * are indexed with the output token's own slots.  out arrays are indexed by
 * absolute token (row t of the [T, H] output).
 */
int oracle_combine(int64_t T, int64_t H, int64_t k, int64_t E, int64_t R, int64_t G,
                   int layout, const uint16_t *y, const int64_t *topk_idx,
                   const float *topk_weights, const int32_t *rank_slot,
                   const int32_t *expert_slot, uint16_t *out_bf16, double *out_f64,
                   int64_t t0, int64_t t1) {
    if (!check_problem(T, k, E, R, G) || H < 1 || H % 8) return OR_BAD_ARGS;
    if (t0 < 0) t0 = 0;
    if (t1 > T) t1 = T;
    const int64_t Tr = T / R, Er = E / R;
    int st = 0;
    unsigned char valid[32];
    int64_t rows[32];
    double *acc = malloc((size_t)H * sizeof(double));
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t src = t / Tr;
        const int64_t *row = topk_idx + t * k;
        st |= row_experts(row, k, E, valid);
        for (int64_t j = 0; j < k; ++j) {
            rows[j] = -1;
            if (!valid[j]) continue;
            int32_t slot;
            if (layout == OR_RANK_MAJOR) {
                int64_t r = row[j] / Er;
                slot = rank_slot[t * R + r];
                if (slot < 0 || slot >= Tr) { st |= OR_BAD_SLOT; continue; }
                rows[j] = rank_major_row(r, src, Tr, R, slot);
            } else {
                slot = expert_slot[t * k + j];
                if (slot < 0 || slot >= Tr) { st |= OR_BAD_SLOT; continue; }
                rows[j] = expert_major_row(row[j], src, Tr, R, slot);
            }
        }
        for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            if (rows[j] < 0) continue;
            double w = (double)topk_weights[t * k + j];
            const uint16_t *yr = y + rows[j] * H;
            for (int64_t h = 0; h < H; ++h) acc[h] += w * bf16_value(yr[h]);
        }
        for (int64_t h = 0; h < H; ++h) {
            if (out_bf16) out_bf16[t * H + h] = oracle_bf16_from_double(acc[h]);
            if (out_f64) out_f64[t * H + h] = acc[h];
        }
    }
    free(acc);
    return st;
}

/* ------------------------------------------------------------------ */
/* low-precision combine wire formats ("MoE-EP Benchmark", environment */
/* reference, MEGA_COMBINE_DTYPE: mxfp8 = 32 e4m3 values sharing one   */
/* e8m0 scale; nvfp4 = 16 e2m1 values with a bf16 scale)               */
/* ------------------------------------------------------------------ */

#define OR_WIRE_MXFP8 1
#define OR_WIRE_NVFP4 2

/* E8M0 (OCP MX scale): 2^(code - 127); code 255 is NaN. */
double oracle_e8m0_decode(uint8_t c) {
    if (c == 255) return NAN;
    return ldexp(1.0, (int)c - 127);
}

/*
 * E2M1 (OCP MX FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; no
 * infinities or NaN.  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 */
double oracle_e2m1_decode(uint8_t c) {
    int s = (c >> 3) & 1, E = (c >> 1) & 3, M = c & 1;
    double v = (E == 0) ? 0.5 * M : ldexp(1.0 + 0.5 * M, E - 1);
    return s ? -v : v;
}

/* float -> e2m1 code (low 4 bits), nearest with ties to the even mantissa,
 * saturating at 6. */
uint8_t oracle_e2m1_encode(float x) {
    uint8_t sign = signbit(x) ? 8 : 0;
    double a = fabs((double)x);
    if (a >= 6.0) return sign | 7;
    if (a < 1.0) {                          /* subnormal step 0.5 */
        double n = round_half_even(a * 2.0);  /* 0..2; 2 = 1.0 */
        return sign | (uint8_t)n;           /* 0 -> 0, 1 -> 0.5, 2 -> code 2 (1.0) */
    }
    int ex;
    frexp(a, &ex);
    int e = ex - 1;                         /* 0..2 */
    double n = round_half_even(ldexp(a, 1 - e));   /* 2..4 */
    if (n == 4.0) { n = 2.0; e += 1; }
    if (e > 2) return sign | 7;
    return sign | (uint8_t)(((e + 1) << 1) | ((int)n - 2));
}

/*
 * MXFP8 cast of one row of bf16 values: for each block of 32, amax = max
 * |v|; shared exponent X = floor(log2(amax)) - 8 (8 = exponent of e4m3's
 * largest power of two), clamped to [-127, 127], stored as e8m0 code
 * X + 127 (code 0 when amax = 0); q = e4m3(v * 2^-X) (exact scaling,
 * nearest-even, saturating at 448).  q [H], s [H / 32].
 */
void oracle_quant_mxfp8_row(int64_t H, const uint16_t *y, uint8_t *q, uint8_t *s) {
    for (int64_t b = 0; b < H / 32; ++b) {
        double amax = 0.0;
        for (int64_t i = 0; i < 32; ++i) {
            double v = fabs(bf16_value(y[b * 32 + i]));
            if (v > amax) amax = v;
        }
        int X = -127;
        if (amax > 0.0) {
            int ex;
            frexp(amax, &ex);               /* amax in [2^(ex-1), 2^ex) */
            X = (ex - 1) - 8;
            if (X < -127) X = -127;
            if (X > 127) X = 127;
        }
        s[b] = (uint8_t)(X + 127);
        for (int64_t i = 0; i < 32; ++i)
            q[b * 32 + i] = oracle_e4m3_encode((float)ldexp(bf16_value(y[b * 32 + i]), -X));
    }
}

/*
 * NVFP4 cast ("16e2m1xbf16"): for each block of 16, amax = max |v|; scale
 * s = bf16(amax / 6), the division in fp32 rounded to nearest and then
 * rounded to nearest-even bf16; inv = 1 / s in fp32 (0 when s = 0);
 * q = e2m1(v * inv), the fp32 product rounded to nearest.  Two codes per
 * byte, element 2i in the low nibble.  q [H / 2], s [H / 16] (bf16 bits).
 */
void oracle_quant_nvfp4_row(int64_t H, const uint16_t *y, uint8_t *q, uint16_t *s) {
    for (int64_t b = 0; b < H / 16; ++b) {
        float amax = 0.0f;
        for (int64_t i = 0; i < 16; ++i) {
            float v = fabsf((float)bf16_value(y[b * 16 + i]));
            if (v > amax) amax = v;
        }
        volatile float t = amax / 6.0f;
        uint16_t sb = oracle_bf16_from_double((double)t);
        s[b] = sb;
        float sf = (float)bf16_value(sb);
        float inv = 0.0f;
        if (sf > 0.0f) {
            volatile float r = 1.0f / sf;
            inv = r;
        }
        for (int64_t i = 0; i < 16; i += 2) {
            volatile float p0 = (float)bf16_value(y[b * 16 + i]) * inv;
            volatile float p1 = (float)bf16_value(y[b * 16 + i + 1]) * inv;
            q[(b * 16 + i) / 2] = (uint8_t)(oracle_e2m1_encode(p0) | (oracle_e2m1_encode(p1) << 4));
        }
    }
}

/* Dequantised value of element h of a wire row. */
static double wire_value(int fmt, int64_t H, const uint8_t *q, const void *s, int64_t h) {
    if (fmt == OR_WIRE_MXFP8)
        return oracle_e4m3_decode(q[h]) * oracle_e8m0_decode(((const uint8_t *)s)[h / 32]);
    uint8_t c = (h & 1) ? (q[h / 2] >> 4) : (q[h / 2] & 15);
    return oracle_e2m1_decode(c) * bf16_value(((const uint16_t *)s)[h / 16]);
}

/*
 * Combine from a wire-format receive buffer: as oracle_combine, with
 * y[row] replaced by the dequantised wire row (exact in fp64).  q: [rows,
 * H] (mxfp8) or [rows, H / 2] (nvfp4) bytes; s: [rows, H / 32] e8m0 codes
 * or [rows, H / 16] bf16 bits.
 */
int oracle_combine_wire(int64_t T, int64_t H, int64_t k, int64_t E, int64_t R, int64_t G,
                        int layout, int fmt, const uint8_t *q, const void *s,
                        const int64_t *topk_idx, const float *topk_weights,
                        const int32_t *rank_slot, const int32_t *expert_slot,
                        uint16_t *out_bf16, double *out_f64, int64_t t0, int64_t t1) {
    if (fmt != OR_WIRE_MXFP8 && fmt != OR_WIRE_NVFP4) return OR_BAD_ARGS;
    /* whole blocks: 32 channels (mxfp8) or 16 (nvfp4) */
    const int64_t blk = fmt == OR_WIRE_MXFP8 ? 32 : 16;
    if (!check_problem(T, k, E, R, G) || H < blk || H % blk) return OR_BAD_ARGS;
    if (t0 < 0) t0 = 0;
    if (t1 > T) t1 = T;
    const int64_t Tr = T / R, Er = E / R;
    const int64_t qrow = fmt == OR_WIRE_MXFP8 ? H : H / 2;
    const int64_t srow = fmt == OR_WIRE_MXFP8 ? H / 32 : H / 16;
    const int64_t sbytes = fmt == OR_WIRE_MXFP8 ? 1 : 2;
    int st = 0;
    unsigned char valid[32];
    int64_t rows[32];
    double *acc = malloc((size_t)H * sizeof(double));
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t src = t / Tr;
        const int64_t *row = topk_idx + t * k;
        st |= row_experts(row, k, E, valid);
        for (int64_t j = 0; j < k; ++j) {
            rows[j] = -1;
            if (!valid[j]) continue;
            int32_t slot;
            if (layout == OR_RANK_MAJOR) {
                int64_t r = row[j] / Er;
                slot = rank_slot[t * R + r];
                if (slot < 0 || slot >= Tr) { st |= OR_BAD_SLOT; continue; }
                rows[j] = rank_major_row(r, src, Tr, R, slot);
            } else {
                slot = expert_slot[t * k + j];
                if (slot < 0 || slot >= Tr) { st |= OR_BAD_SLOT; continue; }
                rows[j] = expert_major_row(row[j], src, Tr, R, slot);
            }
        }
        for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            if (rows[j] < 0) continue;
            double w = (double)topk_weights[t * k + j];
            const uint8_t *qr = q + rows[j] * qrow;
            const char *sr = (const char *)s + rows[j] * srow * sbytes;
            for (int64_t h = 0; h < H; ++h) acc[h] += w * wire_value(fmt, H, qr, sr, h);
        }
        for (int64_t h = 0; h < H; ++h) {
            if (out_bf16) out_bf16[t * H + h] = oracle_bf16_from_double(acc[h]);
            if (out_f64) out_f64[t * H + h] = acc[h];
        }
    }
    free(acc);
    return st;
}

/* Casts the listed rows of y [*, H] into the wire format (q, s laid out as
 * in oracle_combine_wire). */
int oracle_quant_wire_rows(int fmt, int64_t H, int64_t n, const int64_t *rows, const uint16_t *y,
                           uint8_t *q, void *s) {
    if (fmt != OR_WIRE_MXFP8 && fmt != OR_WIRE_NVFP4) return OR_BAD_ARGS;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t r = rows[i];
        if (fmt == OR_WIRE_MXFP8)
            oracle_quant_mxfp8_row(H, y + r * H, q + r * H, (uint8_t *)s + r * (H / 32));
        else
            oracle_quant_nvfp4_row(H, y + r * H, q + r * (H / 2), (uint16_t *)s + r * (H / 16));
    }
    return 0;
}


/* ------------------------------------------------------------------ */
/* two-level (node-forwarding) dispatch and combine                    */
/* ("MORI-EP Benchmark", "Bandwidth Computation": a token crosses the  */
/* inter-node fabric once per destination node - the algo count - and  */
/* is then forwarded to the ranks inside the node; "Combine": the      */
/* reverse, with the same byte counts)                                 */
/* ------------------------------------------------------------------ */

/* Row of (t, n) in the node-major staging buffer [N][R src][Tr][H]. */
static int64_t node_major_row(int64_t n, int64_t src, int64_t Tr, int64_t R, int64_t slot) {
    return (n * R + src) * Tr + slot;
}

/*
 * Hop 1: x[t] to the staging row of every node t goes to.  Hop 2: each
 * staging row to the rank-major rows of the token's ranks in that node
 * (read from the staging row, not from x).  bf16 payload only.
 */
int oracle_dispatch_two_level(int64_t T, int64_t H, int64_t k, int64_t E, int64_t R, int64_t G,
                              const uint16_t *x, const int32_t *rank_slot, const int32_t *node_slot,
                              uint16_t *stage, uint16_t *recv) {
    if (!check_problem(T, k, E, R, G) || H < 1 || H % 8) return OR_BAD_ARGS;
    const int64_t N = R / G, Tr = T / R;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t src = t / Tr;
        for (int64_t n = 0; n < N; ++n) {
            int32_t ns = node_slot[t * N + n];
            if (ns < 0) continue;
            uint16_t *srow = stage + node_major_row(n, src, Tr, R, ns) * H;
            memcpy(srow, x + t * H, (size_t)H * 2);                       /* hop 1 */
            for (int64_t r = n * G; r < (n + 1) * G; ++r) {
                int32_t rs = rank_slot[t * R + r];
                if (rs < 0) continue;
                memcpy(recv + rank_major_row(r, src, Tr, R, rs) * H, srow, (size_t)H * 2);   /* hop 2 */
            }
        }
    }
    return 0;
}

/*
 * Hop 1 (inside node n): partial[t, n] = sum over kept entries j whose
 * expert lives on node n of w_j * y[rank-major row of (t, rank(e_j))],
 * in fp64, rounded once to bf16 into the staging row of (t, n).
 * Hop 2 (at the source): out[t] = sum over nodes n of partial[t, n] in
 * fp64 (ascending n), rounded once to bf16.  out_f64 (may be NULL) gets the
 * fp64 sum of the rounded partials.
 */
int oracle_combine_two_level(int64_t T, int64_t H, int64_t k, int64_t E, int64_t R, int64_t G,
                             const uint16_t *y, const int64_t *topk_idx, const float *topk_weights,
                             const int32_t *rank_slot, const int32_t *node_slot, uint16_t *stage,
                             uint16_t *out_bf16, double *out_f64, int64_t t0, int64_t t1) {
    if (!check_problem(T, k, E, R, G) || H < 1 || H % 8) return OR_BAD_ARGS;
    if (t0 < 0) t0 = 0;
    if (t1 > T) t1 = T;
    const int64_t N = R / G, Tr = T / R, Er = E / R, En = E / N;
    int st = 0;
    unsigned char valid[32];
    double *acc = malloc((size_t)H * sizeof(double));
    double *tot = malloc((size_t)H * sizeof(double));
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t src = t / Tr;
        const int64_t *row = topk_idx + t * k;
        st |= row_experts(row, k, E, valid);
        for (int64_t h = 0; h < H; ++h) tot[h] = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            int32_t ns = node_slot[t * N + n];
            if (ns < 0) continue;
            for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                if (!valid[j] || row[j] / En != n) continue;
                int64_t r = row[j] / Er;
                int32_t rs = rank_slot[t * R + r];
                if (rs < 0 || rs >= Tr) { st |= OR_BAD_SLOT; continue; }
                const uint16_t *yr = y + rank_major_row(r, src, Tr, R, rs) * H;
                double w = (double)topk_weights[t * k + j];
                for (int64_t h = 0; h < H; ++h) acc[h] += w * bf16_value(yr[h]);
            }
            uint16_t *srow = stage + node_major_row(n, src, Tr, R, ns) * H;
            for (int64_t h = 0; h < H; ++h) {
                srow[h] = oracle_bf16_from_double(acc[h]);
                tot[h] += bf16_value(srow[h]);
            }
        }
        for (int64_t h = 0; h < H; ++h) {
            if (out_bf16) out_bf16[t * H + h] = oracle_bf16_from_double(tot[h]);
            if (out_f64) out_f64[t * H + h] = tot[h];
        }
    }
    free(acc);
    free(tot);
    return st;
}
