"""The C-ABI library without a GPU: it loads, exports every symbol that
include/ep.h declares, its host-only helpers compute the right sizes, and
bad arguments are rejected on the host before anything reaches the GPU."""
import ctypes
import os
import re

import pytest
import torch

from combine_ep_layout_05_gb300 import build as epbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    epbuild.build()
    from combine_ep_layout_05_gb300 import ep as epmod
    return epmod


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "ep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ \*]*?\b(ep_[a-z0-9_]+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(ep):
    names = _declared_functions()
    assert len(names) >= 9
    lib = ctypes.CDLL(ep.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(ep.EXPORTS) == names


def test_recv_rows_and_workspace(ep):
    p = ep.problem(32768, 7168, 8, 256, 8)
    assert ep.ep_recv_rows(p, "rank_major") == 8 * 8 * 4096
    assert ep.ep_recv_rows(p, "expert_major") == 256 * 8 * 4096
    # 8 ranks x 16 chunks of 256 tokens x (R + E + N) int32 columns
    assert ep.ep_layout_workspace_bytes(p) == (8 * 16 * (8 + 256 + 1) * 4 + 255) // 256 * 256
    bad = ep.problem(100, 7168, 8, 256, 8)            # T % R != 0
    with pytest.raises(ep.EpError):
        ep.ep_recv_rows(bad)
    assert ep.ep_layout_workspace_bytes(bad) == 0


def test_physical_formula(ep):
    assert ep.ep_rdma_physical_formula(8166, 2) == 4083.0
    assert ep.ep_rdma_physical_formula(3, 2) == 1.5
    assert ep.ep_rdma_physical_formula(5, 1) == 0.0


@pytest.mark.parametrize("T,H,k,E,R,G,why", [
    (32, 7168, 8, 250, 4, 4, "num_experts"),     # E % R
    (32, 7168, 8, 256, 4, 3, "gpus_per_node"),   # R % G
    (30, 7168, 8, 256, 4, 4, "num_tokens"),      # T % R
    (32, 7164, 8, 256, 4, 4, "out of range"),    # H % 8
    (32, 7168, 33, 256, 4, 4, "out of range"),   # k > 32
    (32, 7168, 8, 2048, 4, 4, "out of range"),   # E > 1024
    (65 * 2, 7168, 8, 130, 65, 65, "out of range"),   # R > 64
])
def test_invalid_sizes_rejected_on_host(ep, T, H, k, E, R, G, why):
    p = ep.problem(T, H, k, E, R, G)
    lib = ep.lib()
    rc = lib.ep_layout(ctypes.byref(p), None, *[None] * 11, None, 0, None, None)
    assert rc == ep.EP_ERR_INVALID_ARG
    assert why in ep.ep_last_error_string()
    assert lib.ep_dispatch(ctypes.byref(p), 0, 0, None, None, None, None, None, None, None, None) == 1
    assert lib.ep_combine(ctypes.byref(p), 0, None, None, None, None, None, None, None, None) == 1
    assert lib.ep_rdma_token_count(ctypes.byref(p), None, None, None, None, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; fake pointers stay off GPUs")
def test_bad_pointers_rejected_on_host(ep):
    p = ep.problem(32, 7168, 8, 256, 4)
    lib = ep.lib()
    ok16 = 1 << 20     # aligned fake addresses, never dereferenced: validation fails first
    # layout: NULL topk_idx, misaligned topk_idx, missing or small workspace
    assert lib.ep_layout(ctypes.byref(p), None, *[None] * 11, ok16, 1 << 20, None, None) == 1
    assert lib.ep_layout(ctypes.byref(p), ok16 + 4, *[None] * 11, ok16, 1 << 20, None, None) == 1
    assert lib.ep_layout(ctypes.byref(p), ok16, *[None] * 11, None, 1 << 20, None, None) == 1
    assert lib.ep_layout(ctypes.byref(p), ok16, *[None] * 11, ok16, 16, None, None) == 1
    assert "workspace too small" in ep.ep_last_error_string()
    assert lib.ep_layout(ctypes.byref(p), ok16, *[None] * 9, ok16 + 4, None, ok16, 1 << 20, None, None) == 1
    # dispatch: FP8 with H % 128, unknown layout / dtype, misaligned x, missing slots
    p2 = ep.problem(32, 7176, 8, 256, 4)
    assert lib.ep_dispatch(ctypes.byref(p2), 0, 1, ok16, ok16, ok16, ok16, ok16, ok16, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(p), 7, 0, ok16, ok16, ok16, ok16, ok16, ok16, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(p), 0, 9, ok16, ok16, ok16, ok16, ok16, ok16, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(p), 0, 0, ok16 + 8, ok16, ok16, ok16, ok16, None, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(p), 0, 0, ok16, ok16, None, ok16, ok16, None, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(p), 1, 0, ok16, None, ok16, ok16, ok16, None, None, None) == 1
    assert lib.ep_dispatch(ctypes.byref(p), 0, 1, ok16, ok16, ok16, ok16, ok16, None, None, None) == 1
    # combine: missing weights, misaligned out
    assert lib.ep_combine(ctypes.byref(p), 0, ok16, ok16, None, ok16, ok16, ok16, None, None) == 1
    assert lib.ep_combine(ctypes.byref(p), 0, ok16, ok16, ok16, ok16, ok16, ok16 + 2, None, None) == 1
    # dequant: H % 128
    assert lib.ep_dequant_fp8(ctypes.byref(p2), 0, ok16, ok16, ok16, ok16, ok16, ok16, None) == 1
    assert lib.ep_dequant_fp8(ctypes.byref(p), 1, None, ok16, None, ok16, ok16, ok16, None) == 1


def test_get_status_rejects_bad_pointers_on_host(ep):
    lib = ep.lib()
    assert lib.ep_get_status(None, None, None) == ep.EP_ERR_INVALID_ARG
    assert lib.ep_get_status((1 << 20) + 2, None, None) == ep.EP_ERR_INVALID_ARG
    assert "dev_status" in ep.ep_last_error_string()


def test_python_binding_refuses_host_tensors(ep):
    p = ep.problem(8, 64, 2, 8, 2)
    with pytest.raises(ValueError):
        ep.ep_layout(p, torch.zeros((8, 2), dtype=torch.int64))
