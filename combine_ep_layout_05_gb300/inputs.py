"""Seeded synthetic inputs for MoE expert-parallel dispatch / combine.

This module is shared by the CUDA path's callers (tests, benchmark) and by the
CPU oracle's tests. It holds only random draws and the routing gate that turns
draws into top-k expert choices; none of the dispatch-layout, dispatch or
combine arithmetic lives here.

Workload shapes follow the pages' statement of the problem: tokens
``x[T, hidden]`` in bf16 drawn from N(0, 1) ("MORI-EP Benchmark",
print_bw_values.py, random-data block), ``topk_idx[T, k]`` int64 with -1
meaning "no expert" (same script, ``deep_ep.topk_idx_t == torch.int64``), and
``topk_weights[T, k]`` fp32.

Routing: per token, E logits are drawn i.i.d. N(0, 1) (plus ``log p_e`` for a
Zipf expert popularity); the k largest give ``topk_idx`` ordered by descending
logit (ties, a measure-zero event, go to the lower expert id) and the weights
are the softmax over those k logits. Top-k of exchangeable draws is a uniformly
random k-subset, which is what "uniform routing" means here.

bf16 values are carried as raw ``uint16`` bit patterns in numpy arrays.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "sweep_workloads",
    "make_tokens",
    "make_routing",
    "make_group_limited_routing",
    "make_uniform_weights",
    "make_random_rows",
    "make_workload_inputs",
    "bf16_bits_from_f32",
    "f32_from_bf16_bits",
]

# Stream ids keep the draws for x, routing, weights and expert outputs
# independent of each other for one seed.
_STREAM_X, _STREAM_ROUTE, _STREAM_W, _STREAM_Y = 0, 1, 2, 3


@dataclass(frozen=True)
class Workload:
    """One synthetic problem: R ranks x Tr tokens per rank, hidden H, E experts, top-k."""

    name: str
    ranks: int            # R logical EP ranks
    tokens_per_rank: int  # Tr (also the rank-major segment capacity)
    hidden: int           # H
    experts: int          # E
    topk: int             # k
    gpus_per_node: int    # G; nodes N = R / G
    layout: str           # "rank_major" | "expert_major"
    dtype: str            # dispatch payload: "bf16" | "fp8_e4m3"
    zipf_s: float | None = None
    seed: int = 0
    notes: str = field(default="", compare=False)
    routing: str = "topk"  # "topk" (of N(0,1) logits) | "group_limited" (top min(N, 4) node groups first)

    @property
    def tokens(self) -> int:
        return self.ranks * self.tokens_per_rank

    @property
    def nodes(self) -> int:
        return self.ranks // self.gpus_per_node


# The five workloads. gpus_per_node = ranks (one node) wherever the statement
# of a workload does not give a node count.
WORKLOADS = {
    "decode_r4_t8": Workload("decode_r4_t8", 4, 8, 7168, 256, 8, 4, "rank_major", "bf16",
                             notes="decode size, 32 tokens"),
    "ll_r8_t128_fp8": Workload("ll_r8_t128_fp8", 8, 128, 7168, 256, 8, 8, "expert_major", "fp8_e4m3",
                               notes="low-latency expert-major layout, FP8 dispatch, bf16 combine"),
    "prefill_r8_t4096": Workload("prefill_r8_t4096", 8, 4096, 7168, 256, 8, 8, "rank_major", "bf16",
                                 notes="high-throughput prefill, 32768 tokens"),
    "twolevel_n2g8_t4096_zipf": Workload("twolevel_n2g8_t4096_zipf", 16, 4096, 7168, 256, 8, 8,
                                         "rank_major", "bf16", zipf_s=1.0,
                                         notes="2 nodes x 8 GPUs, Zipf(1) expert popularity"),
    # the pages' node-group-limited routing at the two-level shape with 8
    # nodes, where keeping the top min(N, 4) = 4 node groups binds (with 2
    # nodes every group is kept)
    "grouped_n8g2_t4096": Workload("grouped_n8g2_t4096", 16, 4096, 7168, 256, 8, 2, "rank_major", "bf16",
                                   routing="group_limited",
                                   notes="8 nodes x 2 GPUs, top-4 node groups, then top-8 experts"),
}


def sweep_workloads(hidden: int = 7168, experts: int = 256, dtype: str = "bf16",
                    lo: int = 1, hi: int = 8192):
    """Tokens-per-rank sweep points (powers of two), 8 ranks, rank-major."""
    out = []
    tr = lo
    while tr <= hi:
        out.append(Workload(f"sweep_h{hidden}_e{experts}_{dtype}_t{tr}", 8, tr, hidden, experts, 8, 8,
                            "rank_major", dtype, seed=0))
        tr *= 2
    return out


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs must be finite (the generators only produce finite values).
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def make_tokens(T: int, H: int, seed: int = 0, chunk_rows: int = 4096) -> np.ndarray:
    """x[T, H] ~ N(0, 1) rounded to bf16; returns uint16 bits, C-contiguous."""
    rng = _rng(seed, _STREAM_X)
    out = np.empty((T, H), dtype=np.uint16)
    for r0 in range(0, T, chunk_rows):
        r1 = min(T, r0 + chunk_rows)
        out[r0:r1] = bf16_bits_from_f32(rng.standard_normal((r1 - r0, H), dtype=np.float32))
    return out


def _topk_from_logits(logits: np.ndarray, k: int):
    """k largest logits per row, ordered by descending logit, ties to lower id."""
    T, E = logits.shape
    part = np.argpartition(-logits, k - 1, axis=1)[:, :k]
    sel = np.take_along_axis(logits, part, axis=1)
    # order within the k: descending logit, then ascending id
    order = np.lexsort((part, -sel), axis=1)
    idx = np.take_along_axis(part, order, axis=1)
    val = np.take_along_axis(sel, order, axis=1)
    return idx.astype(np.int64), val


def _softmax(v: np.ndarray) -> np.ndarray:
    v64 = v.astype(np.float64)
    v64 = v64 - v64.max(axis=1, keepdims=True)
    e = np.exp(v64)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def make_routing(T: int, E: int, k: int, seed: int = 0, zipf_s: float | None = None,
                 chunk_rows: int = 8192):
    """Top-k routing from N(0,1) logits (+ log p_e for Zipf(s) popularity).

    Zipf popularity: p_e proportional to 1 / (e + 1)**s over expert ids
    e = 0..E-1, so low expert ids (and therefore low ranks and node 0) are the
    popular ones.

    Returns (topk_idx int64 [T, k], topk_weights float32 [T, k]).
    """
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    rng = _rng(seed, _STREAM_ROUTE)
    bias = None
    if zipf_s is not None:
        p = 1.0 / np.power(np.arange(1, E + 1, dtype=np.float64), zipf_s)
        p /= p.sum()
        bias = np.log(p).astype(np.float32)
    idx = np.empty((T, k), dtype=np.int64)
    w = np.empty((T, k), dtype=np.float32)
    for r0 in range(0, T, chunk_rows):
        r1 = min(T, r0 + chunk_rows)
        logits = rng.standard_normal((r1 - r0, E), dtype=np.float32)
        if bias is not None:
            logits += bias
        i, v = _topk_from_logits(logits, k)
        idx[r0:r1] = i
        w[r0:r1] = _softmax(v)
    return idx, w


def make_group_limited_routing(T: int, E: int, k: int, num_groups: int, seed: int = 0):
    """Group-limited routing: scores |N(0,1)| + 1; experts are split into
    ``num_groups`` equal groups (one per node); each token keeps the
    ``min(num_groups, 4)`` groups with the largest per-group max score, zeroes
    the scores of the other groups, then takes the top-k experts.

    This is the routing of the bandwidth-accounting script on the "MORI-EP
    Benchmark" page (random-data block of print_bw_values.py). Weights are the
    softmax of the selected scores.
    """
    if E % num_groups:
        raise ValueError("E must divide into num_groups")
    rng = _rng(seed, _STREAM_ROUTE)
    scores = np.abs(rng.standard_normal((T, E), dtype=np.float32)) + np.float32(1)
    g = scores.reshape(T, num_groups, E // num_groups)
    gmax = g.max(axis=2)
    keep = min(num_groups, 4)
    top_groups = np.argpartition(-gmax, keep - 1, axis=1)[:, :keep]
    mask = np.zeros((T, num_groups), dtype=bool)
    np.put_along_axis(mask, top_groups, True, axis=1)
    masked = (g * mask[:, :, None]).reshape(T, E)
    idx, val = _topk_from_logits(masked, k)
    return idx, _softmax(val)


def make_uniform_weights(T: int, k: int, seed: int = 0, lo: float = 0.0, hi: float = 2.0) -> np.ndarray:
    """Unnormalised weights U(lo, hi) (so that a combine that drops or reuses a
    weight cannot pass by accident, as it could with weights summing to 1)."""
    rng = _rng(seed, _STREAM_W)
    return rng.uniform(lo, hi, size=(T, k)).astype(np.float32)


def make_random_rows(rows: int, H: int, seed: int = 0, chunk_rows: int = 4096) -> np.ndarray:
    """Stand-in expert outputs: rows of N(0,1) rounded to bf16 (uint16 bits)."""
    rng = _rng(seed, _STREAM_Y)
    out = np.empty((rows, H), dtype=np.uint16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = bf16_bits_from_f32(rng.standard_normal((r1 - r0, H), dtype=np.float32))
    return out


def make_workload_routing(w: Workload):
    """(topk_idx int64 [T,k], topk_weights float32 [T,k]) of a workload."""
    if w.routing == "group_limited":
        return make_group_limited_routing(w.tokens, w.experts, w.topk, w.nodes, seed=w.seed)
    return make_routing(w.tokens, w.experts, w.topk, seed=w.seed, zipf_s=w.zipf_s)


def make_workload_inputs(w: Workload):
    """(x uint16 [T,H], topk_idx int64 [T,k], topk_weights float32 [T,k])."""
    x = make_tokens(w.tokens, w.hidden, seed=w.seed)
    idx, wt = make_workload_routing(w)
    return x, idx, wt
