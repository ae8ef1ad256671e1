"""Parity at the full sizes of the benchmark workloads, in the launch
configuration the benchmark times (same library calls, same sizes).

Layout, counts, slots and RDMA counts are compared in full; dispatched rows
are compared in full (every live row bit-exact, every other row untouched);
FP8 payloads and scales in full where the oracle's cast finishes in seconds;
combine against the oracle on token ranges at the start, middle and end of
the token range, and on every token through the identity-expert property
out[t] = x[t] * sum of weights (within one bf16 ulp).
"""
import pytest

from combine_ep_layout_05_gb300 import inputs
from gpu_helpers import ep, full_path_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return ep()


def _ranges(T, n=256):
    if T <= 2048:
        return None
    mid = (T // 2) // n * n
    return [(0, n), (mid - n // 2, mid + n // 2), (T - n, T)]


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_full_size(m, name):
    w = inputs.WORKLOADS[name]
    small = w.tokens <= 64
    idx, wts = inputs.make_workload_routing(w)
    full_path_check(m, w.ranks, w.tokens_per_rank, w.hidden, w.experts, w.topk, w.gpus_per_node, w.layout,
                    w.dtype, seed=w.seed, idx=idx, w=wts, random_y=small, combine_ranges=_ranges(w.tokens))


SWEEP = ([("bf16", 7168, 256, tr) for tr in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096, 8192)] +
         [("fp8_e4m3", 7168, 256, tr) for tr in (1, 8, 64, 512, 1024)] +
         [("bf16", 4096, 128, tr) for tr in (1, 16, 256, 4096, 8192)] +
         [("fp8_e4m3", 4096, 128, tr) for tr in (2, 128, 1024)])


@pytest.mark.parametrize("dtype,H,E,tr", SWEEP)
def test_sweep_point(m, dtype, H, E, tr):
    full_path_check(m, 8, tr, H, E, 8, 8, "rank_major", dtype, seed=0, random_y=tr <= 16,
                    combine_ranges=_ranges(8 * tr))


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_wire_prefill_full_size(m, fmt):
    # the benchmark's low-precision combine (--combine-fmt) at the prefill
    # workload, where the staged wire kernel runs; unnormalised weights as in
    # the small wire cases
    w = inputs.WORKLOADS["prefill_r8_t4096"]
    idx, _ = inputs.make_routing(w.tokens, w.experts, w.topk, seed=w.seed)
    wts = inputs.make_uniform_weights(w.tokens, w.topk, seed=w.seed)
    full_path_check(m, w.ranks, w.tokens_per_rank, w.hidden, w.experts, w.topk, w.gpus_per_node, w.layout,
                    w.dtype, seed=w.seed, idx=idx, w=wts, random_y=False, combine_ranges=_ranges(w.tokens),
                    wire=fmt)
