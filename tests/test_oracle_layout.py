"""Pins for the oracle's dispatch layout, slots and RDMA token counts.

What pins it (none of it re-runs the oracle's own loops):
  * a worked example done by hand (tests/golden/layout_worked_example.json);
  * the two formulations of the "algo" RDMA count that the "MORI-EP
    Benchmark" page proves equal (per-row dedupe of topk_idx // experts_per_node
    then a count of non-empty entries; a [T, nodes] presence matrix then its
    sum), each written here independently with numpy;
  * set-based counts of unique (token, rank) pairs;
  * slot invariants that determine slots uniquely (a bijection onto
    0..count-1 that increases with the token index);
  * closed-form expectations for uniformly random k-subsets, checked against
    the oracle on seeded inputs and against the numbers the page prints.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_05_gb300 import inputs


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# worked example
# --------------------------------------------------------------------------

def test_worked_example(golden_dir):
    g = _golden(golden_dir, "layout_worked_example.json")
    idx = np.array(g["topk_idx"], np.int64)
    R, G, E = g["num_ranks"], g["gpus_per_node"], g["num_experts"]
    lay, st = oracle.layout(idx, E, R, G)
    assert st == 0
    for key in ("is_token_in_rank", "tokens_per_rank", "recv_tokens_per_rank", "tokens_per_node",
                "tokens_per_expert", "rank_slot", "token_major_offset", "expert_slot", "node_slot"):
        assert np.array_equal(lay[key], np.array(g[key])), key
    algo, phys, st = oracle.rdma_token_count(idx, E, R, G)
    assert st == 0
    assert algo.tolist() == g["algo_per_rank"]
    assert phys.tolist() == g["physical_exact_per_rank"]
    N = R // G
    assert [oracle.rdma_physical_formula(a, N) for a in algo] == g["physical_formula_per_rank"]


def test_worked_example_dispatch_rows(golden_dir):
    g = _golden(golden_dir, "layout_worked_example.json")
    idx = np.array(g["topk_idx"], np.int64)
    R, G, E = g["num_ranks"], g["gpus_per_node"], g["num_experts"]
    T, H = idx.shape[0], 8
    x = np.array([[0x3F80 + t] * H for t in range(T)], np.uint16)
    lay, _ = oracle.layout(idx, E, R, G)
    for name, key, nrows in (("rank_major", "rank_major_rows", R * R * 2),
                             ("expert_major", "expert_major_rows", E * R * 2)):
        recv, _, st = oracle.dispatch(x, idx, lay, E, R, G, layout_name=name)
        assert st == 0 and recv.shape == (nrows, H)
        live = {}
        for t, m in g[key].items():
            for _, row in m.items():
                live[row] = int(t)
        for row in range(nrows):
            if row in live:
                assert np.all(recv[row] == x[live[row]]), (name, row)
            else:
                assert np.all(recv[row] == 0xFFFF), (name, row)   # untouched


def test_worked_example_combine(golden_dir):
    # y[row, h] = row + h (exact in bf16 for these sizes); weights are
    # dyadic so every product and sum is exact in fp64.
    g = _golden(golden_dir, "layout_worked_example.json")
    idx = np.array(g["topk_idx"], np.int64)
    R, G, E = g["num_ranks"], g["gpus_per_node"], g["num_experts"]
    T, k, H = idx.shape[0], idx.shape[1], 8
    w = np.array([[0.5, 0.25, 0.125]] * T, np.float32)
    lay, _ = oracle.layout(idx, E, R, G)
    for name, key in (("rank_major", "rank_major_rows"), ("expert_major", "expert_major_rows")):
        nrows = (R if name == "rank_major" else E) * R * 2
        yv = np.arange(nrows)[:, None] + np.arange(H)[None, :]
        y = inputs.bf16_bits_from_f32(yv.astype(np.float32))
        out, out64, st = oracle.combine(y, idx, w, lay, E, R, G, layout_name=name, want_f64=True)
        assert st == 0
        for t in range(T):
            exp = np.zeros(H)
            for j in range(k):
                e = int(idx[t, j])
                if e < 0:
                    continue
                d = str(e // (E // R)) if name == "rank_major" else str(e)
                exp += w[t, j] * (g[key][str(t)][d] + np.arange(H))
            assert np.array_equal(out64[t], exp), (name, t)
            # exp is exact in float32, so torch's float32 -> bf16 rounds it once
            ref = torch.from_numpy(exp.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
            assert np.array_equal(out[t], ref.view(np.uint16)), (name, t)


# --------------------------------------------------------------------------
# the page's two formulations of the algo RDMA count
# --------------------------------------------------------------------------

def _algo_dedupe_rows(idx, E, N):
    """Per-row dedupe of topk_idx // (E // N), then count of entries != -1."""
    node = np.where(idx >= 0, idx // (E // N), -1)
    cnt = 0
    for row in node:
        seen = []
        for v in row:
            if v != -1 and v not in seen:
                seen.append(v)
        cnt += len(seen)
    return cnt


def _algo_presence_matrix(idx, E, R, G):
    """[T, N] presence matrix scattered from topk_idx // (experts_per_rank * G)."""
    T = idx.shape[0]
    N = R // G
    pres = np.zeros((T, N + 1), bool)
    node = np.where(idx >= 0, idx // ((E // R) * G), N)   # -1 -> a spare column
    np.put_along_axis(pres, node, True, axis=1)
    return int(pres[:, :N].sum())


@pytest.mark.parametrize("R,G,E,k,Tr,seed", [(16, 8, 256, 8, 64, 0), (8, 2, 64, 6, 33, 1),
                                             (6, 3, 36, 4, 17, 2), (4, 1, 8, 3, 9, 3)])
def test_algo_count_two_formulations(R, G, E, k, Tr, seed):
    T = R * Tr
    idx, _ = inputs.make_routing(T, E, k, seed=seed)
    rng = np.random.default_rng(seed)
    idx[rng.random(idx.shape) < 0.1] = -1          # some empty entries
    algo, phys, st = oracle.rdma_token_count(idx, E, R, G)
    assert st == 0
    N = R // G
    for src in range(R):
        part = idx[src * Tr:(src + 1) * Tr]
        a1 = _algo_dedupe_rows(part, E, N)
        a2 = _algo_presence_matrix(part, E, R, G)
        assert a1 == a2 == algo[src]
        node = np.where(part >= 0, part // (E // N), -1)
        mine = src // G
        p = sum(len({int(v) for v in row if v >= 0 and v != mine}) for row in node)
        assert p == phys[src]
    lay, _ = oracle.layout(idx, E, R, G)
    assert np.array_equal(lay["tokens_per_node"].sum(axis=1), algo)


# --------------------------------------------------------------------------
# invariants on random and exhaustive tiny inputs
# --------------------------------------------------------------------------

def _check_invariants(idx, E, R, G):
    T, k = idx.shape
    Tr, N, Er, En = T // R, R // G, E // R, E // (R // G)
    lay, st = oracle.layout(idx, E, R, G)
    assert st == 0
    pairs = set()
    for t in range(T):
        for e in idx[t]:
            if e >= 0:
                pairs.add((t, int(e) // Er))
    # sum of receive counts = number of unique (token, rank) pairs
    assert lay["recv_tokens_per_rank"].sum() == len(pairs)
    assert np.array_equal(lay["recv_tokens_per_rank"], lay["tokens_per_rank"].sum(axis=0))
    itr = np.zeros((T, R), np.uint8)
    for t, r in pairs:
        itr[t, r] = 1
    assert np.array_equal(lay["is_token_in_rank"], itr)
    # per-expert counts sum to the number of valid entries
    assert lay["tokens_per_expert"].sum() == int((idx >= 0).sum())
    # node sets are the unique values of topk_idx // experts_per_node
    for src in range(R):
        for n in range(N):
            c = sum(1 for t in range(src * Tr, (src + 1) * Tr)
                    if n in set(np.unique(idx[t][idx[t] >= 0] // En).tolist()))
            assert lay["tokens_per_node"][src, n] == c
    # rank slots: in every (src, dst) segment, a bijection onto 0..count-1
    # that increases with the token index
    for src in range(R):
        for r in range(R):
            toks = [t for t in range(src * Tr, (src + 1) * Tr) if (t, r) in pairs]
            assert [int(lay["rank_slot"][t, r]) for t in toks] == list(range(len(toks)))
            assert lay["tokens_per_rank"][src, r] == len(toks)
    assert np.all((lay["rank_slot"] >= 0) == (itr == 1))
    # token-major offsets: per destination rank a bijection onto
    # 0..recv-1 in global token order
    for r in range(R):
        toks = [t for t in range(T) if (t, r) in pairs]
        assert [int(lay["token_major_offset"][t, r]) for t in toks] == list(range(len(toks)))
    # expert slots: per (src, expert) a bijection increasing with the token
    for src in range(R):
        for e in range(E):
            occ = [(t, j) for t in range(src * Tr, (src + 1) * Tr) for j in range(k) if idx[t, j] == e]
            assert [int(lay["expert_slot"][t, j]) for t, j in occ] == list(range(len(occ)))
            assert lay["tokens_per_expert"][src, e] == len(occ)
    assert np.all((lay["expert_slot"] >= 0) == (idx >= 0))
    # node slots: per (src, node) a bijection increasing with the token
    for src in range(R):
        for n in range(N):
            toks = [t for t in range(src * Tr, (src + 1) * Tr)
                    if n in set((idx[t][idx[t] >= 0] // En).tolist())]
            assert [int(lay["node_slot"][t, n]) for t in toks] == list(range(len(toks)))
            assert lay["tokens_per_node"][src, n] == len(toks)
    assert int((lay["node_slot"] >= 0).sum()) == int(lay["tokens_per_node"].sum())
    return lay


def test_invariants_exhaustive_tiny():
    # R=2 ranks, E=4 experts, k=2, one token per rank: every pair of rows
    # drawn from all ordered pairs of distinct experts or -1.
    rows = [r for r in itertools.product(range(-1, 4), repeat=2) if r[0] != r[1] or r[0] == -1]
    for G in (1, 2):
        for a, b in itertools.product(rows, rows):
            _check_invariants(np.array([a, b], np.int64), 4, 2, G)


@pytest.mark.parametrize("R,G,E,k,Tr", [(3, 1, 6, 2, 5), (4, 2, 8, 3, 4), (5, 5, 10, 4, 3),
                                        (2, 1, 16, 5, 7), (1, 1, 4, 2, 6)])
def test_invariants_random_small(R, G, E, k, Tr):
    rng = np.random.default_rng(R * 100 + E)
    for trial in range(30):
        T = R * Tr
        idx = np.full((T, k), -1, np.int64)
        for t in range(T):
            m = rng.integers(0, k + 1)
            idx[t, :m] = rng.choice(E, size=m, replace=False)
            idx[t] = idx[t][rng.permutation(k)]
        _check_invariants(idx, E, R, G)


def test_empty_and_all_minus_one():
    lay, st = oracle.layout(np.zeros((0, 8), np.int64), 256, 8, 8)
    assert st == 0 and lay["recv_tokens_per_rank"].sum() == 0
    idx = np.full((16, 4), -1, np.int64)
    lay, st = oracle.layout(idx, 16, 4, 2)
    assert st == 0
    assert lay["tokens_per_rank"].sum() == 0 and np.all(lay["rank_slot"] == -1)
    assert np.all(lay["expert_slot"] == -1)
    algo, phys, _ = oracle.rdma_token_count(idx, 16, 4, 2)
    assert algo.sum() == 0 and phys.sum() == 0


def test_invalid_and_duplicate_ids_flagged():
    idx = np.array([[0, 0, 1], [5, -2, 99], [2, 3, 2], [-1, 7, 6]], np.int64)
    lay, st = oracle.layout(idx, 8, 2, 1)
    assert st == (oracle.BAD_EXPERT | oracle.DUP_EXPERT)
    # flagged entries are ignored: first occurrence kept
    assert lay["expert_slot"][0].tolist() == [0, -1, 0]
    assert lay["expert_slot"][1].tolist() == [0, -1, -1]
    assert lay["expert_slot"][2].tolist() == [0, 0, -1]
    assert lay["tokens_per_expert"].sum() == 2 + 1 + 2 + 2
    _, _, st2 = oracle.rdma_token_count(idx, 8, 2, 1)
    assert st2 == st


def test_bad_arguments_rejected():
    idx = np.zeros((8, 2), np.int64)
    with pytest.raises(ValueError):
        oracle.layout(idx, 10, 4, 1)       # E % R != 0
    with pytest.raises(ValueError):
        oracle.layout(idx, 8, 4, 3)        # R % G != 0
    with pytest.raises(ValueError):
        oracle.layout(np.zeros((7, 2), np.int64), 8, 4, 1)   # T % R != 0


# --------------------------------------------------------------------------
# closed forms for uniform routing, and the page's printed figures
# --------------------------------------------------------------------------

def _hit_dist(E, per_group, k):
    """Distribution of the number of groups (of size per_group) hit by a
    uniformly random k-subset of E items: by inclusion-exclusion."""
    G = E // per_group
    probs = []
    for m in range(0, G + 1):
        # P(exactly m groups hit) = C(G, m) * sum_i (-1)^i C(m, i) C((m-i)*pg, k) / C(E, k)
        s = sum((-1) ** i * math.comb(m, i) * math.comb((m - i) * per_group, k) for i in range(m + 1))
        probs.append(math.comb(G, m) * s / math.comb(E, k))
    return np.array(probs)


def _mean_sd_groups_hit(E, per_group, k):
    p = _hit_dist(E, per_group, k)
    m = np.arange(len(p))
    mu = float((m * p).sum())
    return mu, float(np.sqrt((m * m * p).sum() - mu * mu))


def test_hit_distribution_closed_form():
    # the inclusion-exclusion distribution sums to 1 and its mean matches
    # G * (1 - C(E - pg, k) / C(E, k))
    for E, pg, k in [(256, 128, 8), (256, 16, 8), (256, 32, 8), (128, 16, 8), (12, 3, 4)]:
        p = _hit_dist(E, pg, k)
        assert abs(p.sum() - 1) < 1e-12
        mu, _ = _mean_sd_groups_hit(E, pg, k)
        G = E // pg
        assert abs(mu - G * (1 - math.comb(E - pg, k) / math.comb(E, k))) < 1e-9


def test_pages_printed_counts_match_reading(golden_dir):
    """The page's 8166 algo tokens (4096 tokens, 2 nodes, 256 experts, top-8)
    and 26757 tokens received by one of 16 ranks are single draws; under the
    reading "algo counts unique (token, node) pairs including the local node"
    they sit within 3 sigma of the closed form, and a reading that drops the
    local node (about half) or counts (token, expert) pairs does not."""
    g = _golden(golden_dir, "pages_rdma_counts.json")
    T, E, k = g["num_tokens_per_rank"], g["num_experts"], g["num_topk"]
    N, Gp = g["num_nodes"], g["gpu_per_node"]
    R = N * Gp
    mu, sd = _mean_sd_groups_hit(E, E // N, k)
    algo_mu, algo_sd = T * mu, math.sqrt(T) * sd
    assert abs(g["algo_rdma_tokens_one_rank"] - algo_mu) < 3 * algo_sd
    assert abs(g["algo_rdma_tokens_one_rank"] - algo_mu * (N - 1) / N) > 50 * algo_sd
    assert abs(g["algo_rdma_tokens_one_rank"] - T * k) > 50 * algo_sd
    # receive count of one rank: every source rank sends each token to it
    # with probability 1 - C(E - E/R, k) / C(E, k)
    p = 1 - math.comb(E - E // R, k) / math.comb(E, k)
    n = R * T
    assert abs(g["recv_tokens_rank8"] - n * p) < 3 * math.sqrt(n * p * (1 - p))


@pytest.mark.parametrize("gen", ["uniform", "group_limited"])
def test_oracle_counts_match_closed_form(golden_dir, gen):
    g = _golden(golden_dir, "pages_rdma_counts.json")
    Tr, E, k = g["num_tokens_per_rank"], g["num_experts"], g["num_topk"]
    N, Gp = g["num_nodes"], g["gpu_per_node"]
    R = N * Gp
    T = R * Tr
    if gen == "uniform":
        idx, _ = inputs.make_routing(T, E, k, seed=5)
    else:
        idx, _ = inputs.make_group_limited_routing(T, E, k, N, seed=5)
    algo, phys, st = oracle.rdma_token_count(idx, E, R, Gp)
    assert st == 0
    mu, sd = _mean_sd_groups_hit(E, E // N, k)
    # total over all R source ranks: R*Tr independent tokens
    assert abs(algo.sum() - T * mu) < 4 * math.sqrt(T) * sd
    # physical exact vs the page's formula: equal in expectation
    formula = sum(oracle.rdma_physical_formula(a, N) for a in algo)
    assert abs(phys.sum() - formula) < 4 * math.sqrt(T) * sd
    lay, _ = oracle.layout(idx, E, R, Gp)
    mu_r, sd_r = _mean_sd_groups_hit(E, E // R, k)
    assert abs(lay["recv_tokens_per_rank"].sum() - T * mu_r) < 4 * math.sqrt(T) * sd_r


def test_expected_dispatch_rows_per_token():
    # D/T for the prefill workload shape: R (1 - C(E - E/R, k) / C(E, k)) = 5.295
    mu, sd = _mean_sd_groups_hit(256, 32, 8)
    assert abs(mu - 5.295) < 1e-3
    T = 8 * 4096
    idx, _ = inputs.make_routing(T, 256, 8, seed=0)
    lay, _ = oracle.layout(idx, 256, 8, 8)
    assert abs(lay["recv_tokens_per_rank"].sum() - T * mu) < 4 * math.sqrt(T) * sd
