"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: layout, counts, slots, RDMA counts and dispatched bf16 rows bit-exact;
FP8 payloads and scales bit-exact; combine within one bf16 ulp per element of
the fp64 oracle (plus room for fp32 accumulation under cancellation, used by
at most 0.1% of the elements), and a relative L2 distance to the fp64 sum at
most 1e-3 above that of the oracle's own bf16-rounded output.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_05_gb300 import inputs
from gpu_helpers import DEV, bf16_dev, ep, full_path_check, run_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    return ep()


# --------------------------------------------------------------------------
# small and medium problems: several layout chunks, ragged tails, odd R
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout_name,dtype", [("rank_major", "bf16"), ("expert_major", "bf16"),
                                               ("rank_major", "fp8_e4m3"), ("expert_major", "fp8_e4m3")])
@pytest.mark.parametrize("R,Tr,H,E,k,G", [
    (3, 700, 1024, 48, 6, 1),     # 3 chunks per rank, ragged last chunk, 3 nodes
    (4, 257, 7168, 256, 8, 2),    # 2 chunks per rank (256 + 1), 2 nodes
    (5, 40, 2048, 40, 4, 5),      # R not a power of two, one node
    (8, 128, 7168, 256, 8, 8),
])
def test_parity_small(m, layout_name, dtype, R, Tr, H, E, k, G):
    full_path_check(m, R, Tr, H, E, k, G, layout_name, dtype, seed=R * 7 + Tr)


def test_parity_edge_one_token_per_rank(m):
    full_path_check(m, 8, 1, 7168, 256, 8, 8, "rank_major", "bf16")
    full_path_check(m, 8, 1, 7168, 256, 8, 8, "expert_major", "fp8_e4m3")


def test_parity_single_rank(m):
    full_path_check(m, 1, 300, 512, 16, 4, 1, "rank_major", "bf16")
    full_path_check(m, 1, 300, 512, 16, 4, 1, "expert_major", "fp8_e4m3")


def test_parity_max_ranks_and_topk(m):
    # R = 64 (two ballot rounds in dispatch), k = 32, E = 128
    full_path_check(m, 64, 6, 256, 128, 32, 8, "rank_major", "bf16")
    full_path_check(m, 48, 5, 256, 96, 20, 6, "expert_major", "bf16")


def test_parity_max_experts(m):
    full_path_check(m, 4, 300, 256, 1024, 16, 2, "rank_major", "bf16")
    full_path_check(m, 4, 300, 256, 1024, 16, 2, "expert_major", "fp8_e4m3")


@pytest.mark.parametrize("Tr", [64, 16])   # the small-problem layout (a CTA per rank), the tiny one (a warp)
def test_parity_empty_entries_and_bad_ids(m, Tr):
    R, H, E, k = 4, 256, 32, 6
    T = R * Tr
    idx, w = inputs.make_routing(T, E, k, seed=3)
    rng = np.random.default_rng(3)
    idx[rng.random(idx.shape) < 0.15] = -1
    idx[5] = -1                       # token with no expert: combine gives zeros
    idx[7, 2] = idx[7, 0]             # repeated expert
    idx[9, 1] = E + 3                 # out of range
    idx[11, 4] = -5                   # negative, not -1
    for layout_name in ("rank_major", "expert_major"):
        full_path_check(m, R, Tr, H, E, k, 2, layout_name, "bf16", idx=idx, w=w)


def test_parity_unnormalised_weights(m):
    R, Tr, H, E, k = 4, 100, 512, 64, 8
    w = inputs.make_uniform_weights(R * Tr, k, seed=1)
    idx, _ = inputs.make_routing(R * Tr, E, k, seed=1)
    for layout_name in ("rank_major", "expert_major"):
        full_path_check(m, R, Tr, H, E, k, R, layout_name, "bf16", idx=idx, w=w)


def test_empty_problem(m):
    p = m.problem(0, 7168, 8, 256, 8)
    lb = m.LayoutBuffers(p, DEV)
    lb.tokens_per_rank.fill_(7)
    lb.run(p, torch.empty((0, 8), dtype=torch.int64, device=DEV))
    assert int(lb.tokens_per_rank.abs().sum()) == 0
    algo = torch.full((8,), 5, dtype=torch.int64, device=DEV)
    m.ep_rdma_token_count(p, torch.empty((0, 8), dtype=torch.int64, device=DEV), algo)
    assert int(algo.abs().sum()) == 0
    # every other entry point accepts the empty problem and launches nothing
    e16 = torch.empty((0, 7168), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((0, 8), dtype=torch.int64, device=DEV)
    w = torch.empty((0, 8), dtype=torch.float32, device=DEV)
    i32 = torch.empty((0,), dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for layout_name in ("rank_major", "expert_major"):
        m.ep_dispatch(p, layout_name, "bf16", e16, idx, i32, i32, e16, None, st)
        m.ep_combine(p, layout_name, e16, idx, w, i32, i32, e16, st)
        m.ep_layout_dispatch(p, layout_name, "bf16", e16, idx, lb, e16, None, st)
        for fmt in ("mxfp8", "nvfp4"):
            qs, ss, sdt = m.wire_shapes(p, layout_name, fmt)
            wq = torch.empty(qs, dtype=torch.uint8, device=DEV)
            ws = torch.empty(ss, dtype=sdt, device=DEV)
            m.ep_combine_quantize(p, layout_name, fmt, e16, idx, i32, i32, wq, ws)
            m.ep_combine_wire(p, layout_name, fmt, wq, ws, idx, w, i32, i32, e16, st)
    stage = torch.empty((0, 7168), dtype=torch.bfloat16, device=DEV)
    m.ep_dispatch_two_level(p, e16, i32, i32, stage, e16, st)
    m.ep_combine_two_level(p, e16, idx, w, i32, i32, stage, e16, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_fp8_every_bf16_value(m):
    # one 448 per 128-channel block makes inv = 1, so every bf16 value with
    # |v| <= 448 goes through the device's e4m3 conversion unchanged
    allb = np.arange(65536, dtype=np.uint16)
    v = inputs.f32_from_bf16_bits(allb)
    keep = allb[np.isfinite(v) & (np.abs(v) <= 448)]
    per = 127
    H = 7168
    nblk_row = H // 128
    nblk = -(-keep.size // per)
    T = -(-nblk // nblk_row)
    x = np.zeros((T * nblk_row, 128), np.uint16)
    for b in range(nblk):
        part = keep[b * per:(b + 1) * per]
        x[b, 0] = 0x43E0   # 448.0
        x[b, 1:1 + part.size] = part
    x = x.reshape(T, H)
    idx = np.tile(np.array([[0]], np.int64), (T, 1))
    w = np.ones((T, 1), np.float32)
    full_path_check(m, 1, T, H, 1, 1, 1, "rank_major", "fp8_e4m3", idx=idx, w=w, x=x)


def test_repeat_calls_identical(m):
    # fixed order everywhere: two runs give identical bits
    R, Tr, H, E, k = 8, 256, 7168, 256, 8
    T = R * Tr
    x = bf16_dev(inputs.make_tokens(T, H, seed=2))
    idx, w = inputs.make_routing(T, E, k, seed=2)
    p = m.problem(T, H, k, E, R)
    idx_d, w_d = torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV)
    outs = []
    for _ in range(2):
        lb = run_layout(m, p, idx_d, None)
        recv = torch.zeros((m.ep_recv_rows(p), H), dtype=torch.bfloat16, device=DEV)
        m.ep_dispatch(p, "rank_major", "bf16", x, idx_d, lb.rank_slot, None, recv)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        m.ep_combine(p, "rank_major", recv, idx_d, w_d, lb.rank_slot, None, out)
        outs.append((lb.rank_slot.clone(), recv, out))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))
    assert torch.equal(outs[0][2].view(torch.int16), outs[1][2].view(torch.int16))


# --------------------------------------------------------------------------
# bf16 dispatch from 2048 tokens on runs on the bulk-copy engine
# --------------------------------------------------------------------------

def test_bulk_dispatch_max_ranks(m):
    # 64 ranks x 40 tokens = 2560 tokens: two ballot rounds per token
    full_path_check(m, 64, 40, 256, 128, 32, 8, "rank_major", "bf16", random_y=False)
    full_path_check(m, 64, 40, 256, 128, 32, 8, "expert_major", "bf16", random_y=False)


def test_bulk_dispatch_max_experts(m):
    full_path_check(m, 4, 600, 512, 1024, 16, 2, "rank_major", "bf16", random_y=False)
    full_path_check(m, 4, 600, 512, 1024, 16, 2, "expert_major", "bf16", random_y=False)


def test_bulk_dispatch_split_rows(m):
    # 8200 channels = 16400 bytes per row: two staged pieces of unequal size
    full_path_check(m, 2, 1100, 8200, 16, 4, 1, "rank_major", "bf16", random_y=False)
    full_path_check(m, 2, 1100, 8200, 16, 4, 2, "expert_major", "bf16", random_y=False)


def test_combine_whole_rows_both_lane_widths(m):
    # 5200 tokens: whole rows per combine unit; hidden 1000 (not a multiple
    # of 16 channels) takes the 16-byte lanes, hidden 1024 the 32-byte lanes
    full_path_check(m, 2, 2600, 1000, 16, 4, 1, "rank_major", "bf16", combine_ranges=[(0, 256), (4944, 5200)])
    full_path_check(m, 2, 2600, 1024, 16, 4, 1, "expert_major", "bf16", combine_ranges=[(0, 256), (4944, 5200)])


@pytest.mark.parametrize("Tr,H", [(400, 1536), (1280, 4096), (1280, 4352)])
def test_combine_wide_lanes_few_and_many_rows(m, Tr, H):
    # the 32-byte-lane combine with tokens of 0 to 8 source rows: at most 4
    # rows load two 512-channel steps per batch, more load one.  400 x 8
    # tokens, hidden 1536 = 3 steps: whole rows, and a two-step batch ends
    # half outside the row; 1280 x 8 tokens, hidden 4096: rows in two
    # halves of 2048 channels; hidden 4352: halves of 2304 and 2048
    R, E, k = 8, 64, 8
    T = R * Tr
    idx, w = inputs.make_routing(T, E, k, seed=11)
    rng = np.random.default_rng(11)
    per_rank = E // R
    for t in range(0, T, 3):                    # every third token: 1-4 ranks only
        ranks = rng.choice(R, size=int(rng.integers(1, 5)), replace=False)
        pool = (ranks[:, None] * per_rank + np.arange(per_rank)[None, :]).ravel()
        idx[t] = rng.choice(pool, size=k, replace=False)
    idx[1::17] = -1                             # tokens without experts: zeros
    idx[2::13, 3:] = -1                         # tokens with 3 experts
    for layout_name in ("rank_major", "expert_major"):
        full_path_check(m, R, Tr, H, E, k, R, layout_name, "bf16", idx=idx, w=w,
                        combine_ranges=[(0, 512), (T // 2 - 256, T // 2 + 256), (T - 512, T)])


def test_dispatch_both_kernels_agree_at_threshold(m):
    # 2040 tokens (register copies) and 2048 tokens (bulk copies) of the same
    # stream of routing: the rows both write must be identical
    for R, Tr in ((8, 255), (8, 256)):
        full_path_check(m, R, Tr, 7168, 256, 8, 8, "rank_major", "bf16", seed=5, random_y=False)


def test_cuda_graph_replay_matches_eager(m):
    # the whole step captured once and replayed gives the eager step's bits
    from combine_ep_layout_05_gb300.pipeline import EpPipeline
    for R, Tr, layout, dtype in ((4, 8, "rank_major", "bf16"), (8, 128, "expert_major", "fp8_e4m3"),
                                 (8, 512, "rank_major", "bf16")):
        T, H, E, k = R * Tr, 7168, 256, 8
        x = bf16_dev(inputs.make_tokens(T, H, seed=4))
        idx_h, w_h = inputs.make_routing(T, E, k, seed=4)
        idx, w = torch.from_numpy(idx_h).to(DEV), torch.from_numpy(w_h).to(DEV)
        pipe = EpPipeline(T, H, k, E, R, R, layout, dtype, DEV)
        eager = pipe.step(x, idx, w).clone()
        torch.cuda.synchronize()
        pipe.out.zero_()
        g = pipe.capture(x, idx, w)
        pipe.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(pipe.out.view(torch.int16), eager.view(torch.int16)), (R, Tr, layout, dtype)
        assert int(pipe.status.item()) == 0


# --------------------------------------------------------------------------
# layout + dispatch fused into one cooperative launch
# --------------------------------------------------------------------------

FUSED_CASES = [
    # R, Tr, H, E, k, G, layout, payload
    (8, 4096, 7168, 256, 8, 8, "rank_major", "bf16"),       # the prefill workload: bulk copies, 128 chunks
    (8, 512, 7168, 256, 8, 8, "rank_major", "fp8_e4m3"),
    (8, 128, 7168, 256, 8, 8, "expert_major", "fp8_e4m3"),  # the low-latency workload
    (8, 128, 7168, 256, 8, 8, "expert_major", "bf16"),
    (3, 700, 1024, 48, 6, 1, "rank_major", "bf16"),         # ragged chunks; bulk from 2048 tokens
    (3, 700, 1024, 48, 6, 1, "expert_major", "bf16"),
    (3, 700, 1024, 48, 6, 1, "expert_major", "fp8_e4m3"),
    (4, 200, 2048, 64, 8, 2, "rank_major", "bf16"),         # register copies: 800 tokens
    (4, 200, 2048, 64, 8, 2, "rank_major", "fp8_e4m3"),
    (8, 1, 7168, 256, 8, 8, "rank_major", "bf16"),          # one token per rank
    (8, 1, 7168, 256, 8, 8, "expert_major", "fp8_e4m3"),
    # the one-launch small-problem kernel (a CTA group per source rank, no
    # grid barrier): 64 ranks and top-32, 256 tokens per rank (8 bitmap
    # words), 1024 experts with an FP8 payload
    (64, 4, 256, 128, 32, 8, "rank_major", "bf16"),
    (64, 4, 256, 128, 32, 8, "expert_major", "bf16"),
    (4, 256, 1024, 64, 8, 2, "rank_major", "bf16"),
    (4, 200, 512, 1024, 16, 2, "expert_major", "fp8_e4m3"),
    (4, 8, 7168, 256, 8, 4, "rank_major", "bf16"),          # the decode workload's shape
    (16, 16, 1024, 512, 10, 4, "expert_major", "fp8_e4m3"),  # tiny layout: k > 8, 4 nodes
    (40, 6, 512, 80, 8, 8, "rank_major", "bf16"),           # tiny layout: ranks 32..39
]


@pytest.mark.parametrize("R,Tr,H,E,k,G,layout_name,dtype", FUSED_CASES)
def test_fused_layout_dispatch(m, R, Tr, H, E, k, G, layout_name, dtype):
    full_path_check(m, R, Tr, H, E, k, G, layout_name, dtype, seed=R + Tr, random_y=False, fused=True,
                    combine_ranges=[(0, min(R * Tr, 512))])


def test_fused_more_chunks_than_ctas(m):
    # 16 ranks x 8192 tokens = 512 layout chunks on at most 152 resident CTAs
    full_path_check(m, 16, 8192, 1024, 256, 8, 8, "rank_major", "bf16", random_y=False, fused=True,
                    combine_ranges=[(0, 256), (131072 - 256, 131072)])


def test_fused_max_experts_and_ranks(m):
    # 1024 experts: the slot phase needs more than 48 KB of shared memory
    full_path_check(m, 4, 600, 512, 1024, 16, 2, "expert_major", "bf16", random_y=False, fused=True)
    full_path_check(m, 64, 40, 256, 128, 32, 8, "rank_major", "bf16", random_y=False, fused=True)


@pytest.mark.parametrize("Tr", [600, 64, 16])   # the cooperative kernel, the one-launch kernel (CTA / warp layout)
def test_fused_bad_ids(m, Tr):
    R, H, E, k = 4, 256, 32, 6
    T = R * Tr
    idx, w = inputs.make_routing(T, E, k, seed=3)
    idx[np.random.default_rng(3).random(idx.shape) < 0.15] = -1
    idx[7, 2] = idx[7, 0]
    idx[9, 1] = E + 3
    idx[T - 3, 4] = -9
    for layout_name in ("rank_major", "expert_major"):
        full_path_check(m, R, Tr, H, E, k, 2, layout_name, "bf16", idx=idx, w=w, random_y=False, fused=True)


@pytest.mark.parametrize("Tr", [512, 16])
def test_fused_graph_replay(m, Tr):
    from combine_ep_layout_05_gb300.pipeline import EpPipeline
    R, H, E, k = 8, 7168, 256, 8
    T = R * Tr
    x = bf16_dev(inputs.make_tokens(T, H, seed=6))
    idx_h, w_h = inputs.make_routing(T, E, k, seed=6)
    idx, w = torch.from_numpy(idx_h).to(DEV), torch.from_numpy(w_h).to(DEV)
    ref = EpPipeline(T, H, k, E, R, R, "rank_major", "bf16", DEV, fused=False).step(x, idx, w).clone()
    pipe = EpPipeline(T, H, k, E, R, R, "rank_major", "bf16", DEV, fused=True)
    g = pipe.capture(x, idx, w)
    pipe.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(pipe.out.view(torch.int16), ref.view(torch.int16))
    assert int(pipe.status.item()) == 0


def test_get_status_reads_the_kernels_bits(m):
    # ep_get_status waits for the stream and returns the status word: 0 after
    # a clean layout, the bad-expert and repeated-expert bits after one fed
    # such ids (the C call then returns EP_ERR_DEVICE)
    import ctypes
    R, Tr, E, k = 2, 40, 16, 4
    idx, _ = inputs.make_routing(R * Tr, E, k, seed=9)
    p = m.problem(R * Tr, 256, k, E, R)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_layout(m, p, torch.from_numpy(idx).to(DEV), st)
    assert m.ep_get_status(st) == 0
    idx[3, 1] = idx[3, 0]
    idx[5, 2] = E + 1
    run_layout(m, p, torch.from_numpy(idx).to(DEV), st)
    assert m.ep_get_status(st) == m.EP_STATUS_BAD_EXPERT | m.EP_STATUS_DUP_EXPERT
    word = ctypes.c_int32(0)
    rc = m.lib().ep_get_status(st.data_ptr(), ctypes.byref(word), torch.cuda.current_stream().cuda_stream)
    assert rc == m.EP_ERR_DEVICE and word.value == m.EP_STATUS_BAD_EXPERT | m.EP_STATUS_DUP_EXPERT


def test_bounded_waits_run_out_and_report(m):
    # a counter nothing increments and an mbarrier whose bytes never arrive:
    # both bounded waits give up, raise EP_STATUS_TIMEOUT, and the context
    # keeps working
    words = torch.full((2,), 77, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.ep_selftest_wait_timeout(words, 1000, st)
    torch.cuda.synchronize()
    assert int(words[0].item()) == 3
    assert int(st.item()) == m.EP_STATUS_TIMEOUT
    full_path_check(m, 2, 16, 256, 8, 2, 2, "rank_major", "bf16")


# --------------------------------------------------------------------------
# low-precision combine wire formats
# --------------------------------------------------------------------------

WIRE_CASES = [
    # R, Tr, H, E, k, G, layout, dispatch payload
    (4, 257, 7168, 256, 8, 2, "rank_major", "bf16"),
    (8, 128, 7168, 256, 8, 8, "expert_major", "fp8_e4m3"),   # the low-latency workload
    (3, 700, 1024, 48, 6, 1, "rank_major", "bf16"),
    (5, 40, 2048, 40, 4, 5, "expert_major", "bf16"),
    (8, 1, 7168, 256, 8, 8, "rank_major", "bf16"),
    # more than 8 rows per token: several row groups per channel step
    (2, 300, 1024, 64, 12, 2, "expert_major", "bf16"),
    (16, 40, 512, 64, 12, 8, "rank_major", "bf16"),
    # hidden not a multiple of 128: mxfp8 takes the unstaged kernel
    (4, 33, 160, 32, 4, 2, "rank_major", "bf16"),
]


def _wire_weights(weights, T, k, seed, w_softmax):
    return w_softmax if weights == "softmax" else inputs.make_uniform_weights(T, k, seed=seed)


@pytest.mark.parametrize("weights", ["softmax", "uniform"])
@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("R,Tr,H,E,k,G,layout_name,dtype", WIRE_CASES)
def test_wire_combine(m, fmt, weights, R, Tr, H, E, k, G, layout_name, dtype):
    # The routing's softmax weights (what the benchmark runs) and
    # unnormalised U(0,2) weights (a combine that drops or reuses a weight
    # cannot pass).  With softmax weights (sum 1 +- 2^-24) and identity
    # experts, out = v * sum(w) where a decoded nvfp4 value v is often exactly
    # a bf16 midpoint: the last bits of the weight sum pick the rounding
    # direction, so the GPU's fp32 sum and the oracle's fp64 sum round many
    # such elements to neighbouring bf16 values.  Both are within one ulp of
    # the fp64 sum, and the rel-L2 gate is measured against the fp64 sum.
    T = R * Tr
    seed = R * 3 + Tr
    idx, w_sm = inputs.make_routing(T, E, k, seed=seed)
    w = _wire_weights(weights, T, k, seed, w_sm)
    full_path_check(m, R, Tr, H, E, k, G, layout_name, dtype, seed=seed, idx=idx, w=w, random_y=False,
                    wire=fmt)


# enough tokens for the staged wire kernel (it takes over from about 8192
# tokens at hidden 7168); k = 12 gives up to 12 rows per token, so a channel
# step has two row groups
STAGED_WIRE_CASES = [
    (16, 2048, 1024, 64, 12, 8, "rank_major"),
    (4, 8192, 512, 64, 12, 2, "expert_major"),
]


@pytest.mark.parametrize("weights", ["softmax", "uniform"])
@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("R,Tr,H,E,k,G,layout_name", STAGED_WIRE_CASES)
def test_wire_combine_staged(m, fmt, weights, R, Tr, H, E, k, G, layout_name):
    T = R * Tr
    idx, w_sm = inputs.make_routing(T, E, k, seed=T + k)
    w = _wire_weights(weights, T, k, T + k, w_sm)
    full_path_check(m, R, Tr, H, E, k, G, layout_name, "bf16", seed=T + k, idx=idx, w=w, random_y=False,
                    combine_ranges=[(0, 512), (T // 2 - 256, T // 2 + 256), (T - 512, T)], wire=fmt)


@pytest.mark.parametrize("R,Tr,H,E,k,G,layout_name", [(3, 21, 48, 12, 3, 3, "rank_major"),
                                                      (2, 17, 208, 8, 5, 1, "expert_major")])
def test_wire_combine_nvfp4_unstaged(m, R, Tr, H, E, k, G, layout_name):
    # hidden not a multiple of 32: nvfp4 takes the unstaged kernel
    T = R * Tr
    idx, w_sm = inputs.make_routing(T, E, k, seed=T)
    for weights in ("softmax", "uniform"):
        w = _wire_weights(weights, T, k, T, w_sm)
        full_path_check(m, R, Tr, H, E, k, G, layout_name, "bf16", seed=T, idx=idx, w=w, random_y=False,
                        wire="nvfp4")


def _every_block_max_rows(blk, H, seed):
    """Rows whose blocks of `blk` channels take every positive finite bf16
    value as their maximum magnitude (one block each, in order); the other
    elements are nonzero bf16 values no larger in magnitude, random signs."""
    rng = np.random.default_rng(seed)
    maxima = np.arange(1, 0x7F80, dtype=np.uint32)
    nb = H // blk
    rows = -(-len(maxima) // nb)
    amax = np.ones(rows * nb, dtype=np.uint32) * 0x3F80        # pad blocks: max 1.0
    amax[:len(maxima)] = maxima
    a = (amax << 16).view(np.float32)[:, None]
    v = (a * rng.uniform(0.0, 1.0, (len(amax), blk)).astype(np.float32)).astype(np.float32)
    bits = inputs.bf16_bits_from_f32(v).astype(np.uint32)
    mag = np.minimum(bits & 0x7FFF, amax[:, None])             # rounding never exceeds the maximum
    mag = np.where(mag == 0, amax[:, None], mag)                # no zero elements
    mag[:, 0] = amax                                            # the maximum itself
    sign = rng.integers(0, 2, mag.shape).astype(np.uint32) << 15
    return (mag | sign).astype(np.uint16).reshape(rows, H)


def test_fp8_cast_every_block_max(m):
    # the FP8 dispatch's block scale and inverse over every positive finite
    # bf16 block maximum, bit-exact against the oracle (one rank, one expert:
    # expert-major row t holds token t)
    H = 1024
    x = _every_block_max_rows(128, H, seed=22)
    T = x.shape[0]
    idx_h = np.zeros((T, 1), np.int64)
    p = m.problem(T, H, 1, 1, 1, 1)
    idx = torch.from_numpy(idx_h).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lb = run_layout(m, p, idx, st)
    rows = m.ep_recv_rows(p, "expert_major")
    q = torch.full((rows, H), 0xFF, dtype=torch.uint8, device=DEV)
    s = torch.full((rows, H // 128), float("nan"), dtype=torch.float32, device=DEV)
    m.ep_dispatch(p, "expert_major", "fp8_e4m3", bf16_dev(x), idx, lb.rank_slot, lb.expert_slot, q, s, st)
    lay_o, _ = oracle.layout(idx_h, 1, 1, 1)
    q_o, s_o, _ = oracle.dispatch(x, idx_h, lay_o, 1, 1, 1, layout_name="expert_major", dtype="fp8_e4m3")
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_o.view(np.uint32)), "FP8 scales differ"
    assert np.array_equal(q.cpu().numpy(), q_o), "FP8 codes differ"
    assert int(st.item()) == 0


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_wire_cast_every_block_max(m, fmt):
    # the casts' scale arithmetic over every positive finite bf16 block
    # maximum, bit-exact against the oracle: one token per row on one rank and
    # one expert, so receive row t holds token t
    H = 512
    y = _every_block_max_rows(32 if fmt == "mxfp8" else 16, H, seed=21)
    T = y.shape[0]
    p = m.problem(T, H, 1, 1, 1, 1)
    idx = torch.zeros((T, 1), dtype=torch.int64, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lb = run_layout(m, p, idx, st)
    qs, ss, sdt = m.wire_shapes(p, "rank_major", fmt)
    wq = torch.full(qs, 0xAB, dtype=torch.uint8, device=DEV)
    ws = torch.zeros(ss, dtype=sdt, device=DEV)
    m.ep_combine_quantize(p, "rank_major", fmt, bf16_dev(y), idx, lb.rank_slot, lb.expert_slot, wq, ws)
    q_o, s_o = oracle.quant_wire_rows(y, range(T), fmt)
    s_h = ws.view(torch.int16).cpu().numpy().view(np.uint16) if fmt == "nvfp4" else ws.cpu().numpy()
    assert np.array_equal(s_h, s_o), f"{fmt} scales differ"
    assert np.array_equal(wq.cpu().numpy(), q_o), f"{fmt} codes differ"
    assert int(st.item()) == 0


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_wire_pipeline_graph(m, fmt):
    from combine_ep_layout_05_gb300.pipeline import EpPipeline
    R, Tr, H, E, k = 8, 512, 7168, 256, 8
    T = R * Tr
    x = bf16_dev(inputs.make_tokens(T, H, seed=8))
    idx_h, w_h = inputs.make_routing(T, E, k, seed=8)
    idx, w = torch.from_numpy(idx_h).to(DEV), torch.from_numpy(w_h).to(DEV)
    ref = EpPipeline(T, H, k, E, R, R, "rank_major", "bf16", DEV).step(x, idx, w).float()
    pipe = EpPipeline(T, H, k, E, R, R, "rank_major", "bf16", DEV, combine_fmt=fmt)
    eager = pipe.step(x, idx, w).clone()
    g = pipe.capture(x, idx, w)
    pipe.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(pipe.out.view(torch.int16), eager.view(torch.int16))
    # accuracy against the bf16 combine (rel-L2): the formats' cost
    rel = float((eager.float() - ref).norm() / ref.norm())
    assert rel < (0.06 if fmt == "mxfp8" else 0.2), rel


def test_group_limited_routing_two_nodes(m):
    # the pages' bandwidth-accounting routing: |N(0,1)|+1 scores, top
    # min(N, 4) node groups by group max, then top-8; 2 nodes x 8 GPUs
    R, Tr, H, E, k, G = 16, 512, 2048, 256, 8, 8
    T = R * Tr
    idx, w = inputs.make_group_limited_routing(T, E, k, R // G, seed=11)
    for layout_name in ("rank_major", "expert_major"):
        full_path_check(m, R, Tr, H, E, k, G, layout_name, "bf16", idx=idx, w=w, random_y=False,
                        combine_ranges=[(0, 256), (T - 256, T)])
    # 4 nodes x 4 GPUs: top-4 of 4 groups, then top-8
    idx4, w4 = inputs.make_group_limited_routing(T, E, k, 4, seed=12)
    full_path_check(m, R, Tr, H, E, k, 4, "rank_major", "bf16", idx=idx4, w=w4, random_y=False,
                    combine_ranges=[(0, 256)])


# --------------------------------------------------------------------------
# two-level (node-forwarding) dispatch and combine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("R,G,Tr,H,E,k", [
    (16, 8, 256, 2048, 256, 8),   # 2 nodes x 8 GPUs, 4096 tokens: bulk-copy first hop
    (8, 2, 40, 512, 64, 6),       # 4 nodes, register-copy first hop
    (6, 3, 100, 256, 24, 4),      # 2 nodes, odd sizes
    (4, 1, 33, 256, 16, 4),       # one GPU per node
    (8, 8, 64, 256, 32, 4),       # one node: hop 2 fans out inside it
    (6, 3, 50, 1000, 24, 4),      # 125 16-byte chunks per row: a ragged last chunk pair
])
def test_two_level(m, R, G, Tr, H, E, k):
    from gpu_helpers import two_level_check
    two_level_check(m, R, G, Tr, H, E, k, seed=R + G + Tr, combine_ranges=[(0, min(R * Tr, 256))])


def test_two_level_identity_zipf(m):
    from gpu_helpers import two_level_check
    two_level_check(m, 16, 8, 512, 1024, 256, 8, seed=2, zipf=1.0, random_y=False,
                    combine_ranges=[(0, 128), (16 * 512 - 128, 16 * 512)])


def test_two_level_group_limited(m):
    # the pages' node-group-limited routing with 8 nodes x 2 GPUs: each token
    # reaches at most 4 nodes
    from gpu_helpers import two_level_check
    R, G, Tr, H, E, k = 16, 2, 256, 1024, 256, 8
    routing = inputs.make_group_limited_routing(R * Tr, E, k, R // G, seed=5)
    assert int(max(len(set((row // (E // (R // G))).tolist())) for row in routing[0])) <= 4
    two_level_check(m, R, G, Tr, H, E, k, seed=5, routing=routing, combine_ranges=[(0, 256), (R * Tr - 256, R * Tr)])
