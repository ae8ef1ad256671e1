"""Pins for the oracle's two-level (node-forwarding) dispatch and combine.

One copy per (token, node) crosses between nodes - the pages' "algo" count
("MORI-EP Benchmark", "Bandwidth Computation") - and is then forwarded to the
token's ranks inside the node; combine reduces inside each node first, then
across nodes.  References: the single-level dispatch (the forwarded result
must equal it bit for bit), the algo count (live staging rows), the
one-node special case (two-level combine = single-level combine), and a
closed form with identity experts and dyadic weights.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_05_gb300 import inputs


@pytest.mark.parametrize("R,G,Tr,H,E,k", [(4, 2, 6, 64, 16, 4), (8, 4, 5, 32, 64, 8), (6, 3, 7, 16, 12, 3),
                                          (4, 1, 3, 16, 8, 2)])
def test_two_level_dispatch_equals_direct(R, G, Tr, H, E, k):
    T = R * Tr
    x = inputs.make_tokens(T, H, seed=R + G)
    idx, _ = inputs.make_routing(T, E, k, seed=R + G)
    idx[::4, 0] = -1
    lay, _ = oracle.layout(idx, E, R, G)
    stage, recv = oracle.dispatch_two_level(x, lay, E, R, G, k)
    direct, _, _ = oracle.dispatch(x, idx, lay, E, R, G)
    assert np.array_equal(recv, direct)
    # live staging rows: one per (token, node) = the algo count, each a copy of its token
    live = np.any(stage != 0xFFFF, axis=1)
    algo, _, _ = oracle.rdma_token_count(idx, E, R, G)
    assert live.sum() == algo.sum()
    N = R // G
    seg = stage.reshape(N, R, Tr, H)
    for src in range(R):
        for n in range(N):
            toks = [t for t in range(src * Tr, (src + 1) * Tr) if lay["node_slot"][t, n] >= 0]
            for i, t in enumerate(toks):
                assert np.array_equal(seg[n, src, i], x[t])


def test_two_level_group_limited_routing():
    # 8 nodes x 2 GPUs, group-limited routing: each token reaches at most 4
    # nodes, so at most 4 staging rows per token; the forwarded buffer still
    # equals the direct dispatch and the combine stays within the partials'
    # rounding of the single-level fp64 combine
    R, G, Tr, H, E, k = 16, 2, 3, 32, 64, 8
    T = R * Tr
    x = inputs.make_tokens(T, H, seed=9)
    idx, w = inputs.make_group_limited_routing(T, E, k, R // G, seed=9)
    lay, _ = oracle.layout(idx, E, R, G)
    assert int((lay["node_slot"] >= 0).sum(axis=1).max()) <= 4
    stage, recv = oracle.dispatch_two_level(x, lay, E, R, G, k)
    direct, _, _ = oracle.dispatch(x, idx, lay, E, R, G)
    assert np.array_equal(recv, direct)
    algo, _, _ = oracle.rdma_token_count(idx, E, R, G)
    assert np.any(stage != 0xFFFF, axis=1).sum() == algo.sum()
    out_bf16, out64, _, st = oracle.combine_two_level(direct, idx, w, lay, E, R, G, want_f64=True)
    assert st == 0
    _, ref64, _ = oracle.combine(direct, idx, w, lay, E, R, G, want_f64=True)
    # each of <= 4 partials is rounded to bf16 once (relative 2^-9), then the sum once
    scale = np.abs(ref64) + 1e-30
    err = np.abs(inputs.f32_from_bf16_bits(out_bf16).astype(np.float64) - ref64)
    assert np.all(err <= 5 * 2.0 ** -8 * np.maximum(scale, np.abs(out64)) + 1e-30)


def test_two_level_combine_one_node_equals_single_level():
    R, G, Tr, H, E, k = 4, 4, 6, 64, 16, 4
    T = R * Tr
    idx, _ = inputs.make_routing(T, E, k, seed=2)
    w = inputs.make_uniform_weights(T, k, seed=2)
    lay, _ = oracle.layout(idx, E, R, G)
    y = inputs.make_random_rows(R * R * Tr, H, seed=2)
    one, _, _ = oracle.combine(y, idx, w, lay, E, R, G)
    two, _, stage, st = oracle.combine_two_level(y, idx, w, lay, E, R, G)
    assert st == 0 and np.array_equal(one, two)


def test_two_level_combine_closed_form():
    # identity experts, dyadic weights: partial_n = bf16(x * W_n) with W_n
    # the weights of node n's experts; out = bf16(sum_n partial_n)
    R, G, Tr, H, E, k = 4, 2, 5, 32, 16, 4
    T = R * Tr
    x = inputs.make_tokens(T, H, seed=3)
    idx, _ = inputs.make_routing(T, E, k, seed=3)
    w = (np.random.default_rng(3).integers(1, 64, (T, k)) / 32).astype(np.float32)
    lay, _ = oracle.layout(idx, E, R, G)
    _, y = oracle.dispatch_two_level(x, lay, E, R, G, k)
    out, _, _, st = oracle.combine_two_level(y, idx, w, lay, E, R, G)
    assert st == 0
    N, En = R // G, E // (R // G)
    xf = torch.from_numpy(inputs.f32_from_bf16_bits(x).copy())
    for t in range(T):
        tot = torch.zeros(H, dtype=torch.float64)
        for n in range(N):
            Wn = sum(float(w[t, j]) for j in range(k) if idx[t, j] // En == n)
            if any(idx[t, j] // En == n for j in range(k)):
                # x * Wn is exact in float32 (8 + 11 bits); torch rounds it to bf16 once
                tot += (xf[t] * Wn).to(torch.bfloat16).double()
        ref = tot.float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out[t], ref), t
