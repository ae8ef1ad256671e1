"""ep_layout_noalloc, the layout entry point for callers that cannot
allocate device memory (for example code inside a framework whose allocator
owns the GPU, or latency-critical paths that cannot afford a cudaMalloc).

It keeps its scratch in a static device array instead of a caller-provided
workspace.  This file is collected last, so a failure here comes after every
other test has run; it also passes on its own in a fresh process.  The test
calls the entry point through the C ABI and compares every output with
ep_layout's (integers: bit-exact, the tolerance the layout tests use) on two
calls in a row with different problems, so stale scratch contents from the
first call cannot leak into the second.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_ep_layout_05_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
KEYS = ("is_token_in_rank", "tokens_per_rank", "tokens_per_expert", "tokens_per_node", "recv_tokens_per_rank",
        "rank_slot", "token_major_offset", "expert_slot", "node_slot", "algo_per_rank", "physical_exact_per_rank")


@pytest.fixture(scope="module")
def ep():
    from combine_ep_layout_05_gb300 import build
    build.build()
    from combine_ep_layout_05_gb300 import ep as m
    return m


def _outputs(p, dev=DEV):
    T, k, E, R, N = p.num_tokens, p.num_topk, p.num_experts, p.num_ranks, p.N
    i32 = dict(dtype=torch.int32, device=dev)
    return {"is_token_in_rank": torch.full((T, R), 7, dtype=torch.uint8, device=dev),
            "tokens_per_rank": torch.full((R, R), -7, **i32), "tokens_per_expert": torch.full((R, E), -7, **i32),
            "tokens_per_node": torch.full((R, N), -7, **i32), "recv_tokens_per_rank": torch.full((R,), -7, **i32),
            "rank_slot": torch.full((T, R), -7, **i32), "token_major_offset": torch.full((T, R), -7, **i32),
            "expert_slot": torch.full((T, k), -7, **i32),
            "node_slot": torch.full((T, N), -7, **i32),
            "algo_per_rank": torch.full((R,), -7, dtype=torch.int64, device=dev),
            "physical_exact_per_rank": torch.full((R,), -7, dtype=torch.int64, device=dev)}


def _noalloc(ep, p, idx, out, status):
    lib = ep.lib()
    rc = lib.ep_layout_noalloc(ctypes.byref(p), idx.data_ptr(), *[out[key].data_ptr() for key in KEYS],
                               status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc


def _reference(ep, p, idx, status):
    out = _outputs(p)
    ws = torch.empty(ep.ep_layout_workspace_bytes(p), dtype=torch.uint8, device=DEV)
    ep.ep_layout(p, idx, *[out[key] for key in KEYS[:8]], ws, status, algo_per_rank=out["algo_per_rank"],
                 physical_exact_per_rank=out["physical_exact_per_rank"], node_slot=out["node_slot"])
    return out


# prefill-sized (two layout kernels using the scratch), a 4 x 300 problem, and
# the decode shape (one small-problem kernel that needs no scratch)
@pytest.mark.parametrize("R,Tr,E,k,G,seed", [(8, 4096, 256, 8, 8, 0), (4, 300, 64, 6, 2, 1), (4, 8, 256, 8, 4, 2)])
def test_noalloc_matches_layout_two_calls_in_a_row(ep, R, Tr, E, k, G, seed):
    # first problem: prefill-sized; second: a different, smaller one
    problems = [(R, Tr, E, k, G, seed), (5, 700, 40, 4, 5, seed + 10)]
    for (r, tr, e, kk, g, sd) in problems:
        T = r * tr
        idx_h, _ = inputs.make_routing(T, e, kk, seed=sd)
        idx = torch.from_numpy(idx_h).to(DEV)
        p = ep.problem(T, 7168, kk, e, r, g)
        st_ref = torch.zeros(1, dtype=torch.int32, device=DEV)
        ref = _reference(ep, p, idx, st_ref)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = _outputs(p)
        assert _noalloc(ep, p, idx, out, st) == ep.EP_OK, ep.ep_last_error_string()
        torch.cuda.synchronize()
        for key in KEYS:
            assert torch.equal(out[key], ref[key]), key
        assert int(st.item()) == int(st_ref.item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch(ep):
    # 64 ranks x 8192 tokens/rank x 1024 experts needs ~9.4 MB of scratch
    p = ep.problem(64 * 8192, 7168, 8, 1024, 64, 8)
    assert ep.ep_layout_workspace_bytes(p) > 4 << 20
    lib = ep.lib()
    rc = lib.ep_layout_noalloc(ctypes.byref(p), None, *[None] * 11, None, None)
    assert rc == ep.EP_ERR_INVALID_ARG
    assert "static scratch" in ep.ep_last_error_string()
