"""Parity at the full sizes of the benchmark workloads, in the launch
configuration the benchmark times (same library calls, same sizes).

Layout, counts, slots and RDMA counts are compared in full; dispatched rows
are compared in full (every live row bit-exact, every other row untouched);
FP8 payloads and scales in full; the FP8 identity expert in full below 2^26
x elements and on the rows the combine check reads above; combine against
the oracle on token ranges (the first and last tokens and the middle of
every source rank's segment), and on every token through the
identity-expert property out[t] = x[t] * sum of weights (within one bf16
ulp).
"""
import pytest

from combine_ep_layout_05_gb300 import inputs
from gpu_helpers import combine_ranges, ep, full_path_check, two_level_check_full_size

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return ep()


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_full_size(m, name):
    w = inputs.WORKLOADS[name]
    small = w.tokens <= 64
    idx, wts = inputs.make_workload_routing(w)
    full_path_check(m, w.ranks, w.tokens_per_rank, w.hidden, w.experts, w.topk, w.gpus_per_node, w.layout,
                    w.dtype, seed=w.seed, idx=idx, w=wts, random_y=small,
                    combine_ranges=combine_ranges(w.tokens, w.ranks))


# every point of the tokens-per-rank sweep: powers of two 1..8192 at
# hidden 7168 / 256 experts and hidden 4096 / 128 experts, bf16 and FP8
SWEEP_TOKENS = [1 << i for i in range(14)]
SWEEP = [(dtype, H, E, tr) for H, E in ((7168, 256), (4096, 128)) for dtype in ("bf16", "fp8_e4m3")
         for tr in SWEEP_TOKENS]


@pytest.mark.parametrize("dtype,H,E,tr", SWEEP)
def test_sweep_point(m, dtype, H, E, tr):
    full_path_check(m, 8, tr, H, E, 8, 8, "rank_major", dtype, seed=0, random_y=tr <= 16,
                    combine_ranges=combine_ranges(8 * tr, 8))


@pytest.mark.parametrize("weights", ["softmax", "uniform"])
@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_wire_prefill_full_size(m, fmt, weights):
    # the benchmark's low-precision combine (--combine-fmt) at the prefill
    # workload, where the staged wire kernel runs: with the routing's softmax
    # weights (what the benchmark times) and with unnormalised U(0,2) weights
    w = inputs.WORKLOADS["prefill_r8_t4096"]
    idx, wts = inputs.make_routing(w.tokens, w.experts, w.topk, seed=w.seed)
    if weights == "uniform":
        wts = inputs.make_uniform_weights(w.tokens, w.topk, seed=w.seed)
    full_path_check(m, w.ranks, w.tokens_per_rank, w.hidden, w.experts, w.topk, w.gpus_per_node, w.layout,
                    w.dtype, seed=w.seed, idx=idx, w=wts, random_y=False,
                    combine_ranges=combine_ranges(w.tokens, w.ranks), wire=fmt)


@pytest.mark.parametrize("name", ["twolevel_n2g8_t4096_zipf", "grouped_n8g2_t4096"])
def test_two_level_full_size(m, name):
    # the node-forwarding path at the sizes the benchmark times it: 16 ranks
    # x 4096 tokens, 2 nodes x 8 GPUs with Zipf(1) routing, and 8 nodes x 2
    # GPUs with group-limited routing
    w = inputs.WORKLOADS[name]
    two_level_check_full_size(m, w, combine_ranges(w.tokens, w.ranks))
