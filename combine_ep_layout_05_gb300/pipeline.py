"""One pass of the hot path through the C ABI, with its device buffers.

``EpPipeline`` allocates (with torch) every device buffer one problem needs
and runs layout (with the RDMA token counts) -> dispatch -> identity expert
-> combine on one stream, every step in the library's kernels.  The identity
expert is free for a bf16 payload (combine reads the receive buffer itself)
and ``ep_dequant_fp8`` for an FP8 payload.
"""
from __future__ import annotations

import torch

from . import ep


def one_launch_layout_dispatch(T: int, R: int, dtype: str) -> bool:
    """True where layout and dispatch are faster as one ep_layout_dispatch
    launch than as ep_layout followed by ep_dispatch: problems the library's
    single small-problem kernel covers (every source rank in one 256-token
    chunk, at most 4096 tokens before the last source rank, a register-copy
    or FP8 dispatch) with at most 32 tokens per rank.  Measured on GB300
    (8 ranks, hidden 7168, steps replayed from a CUDA graph): one launch is
    2 us shorter at 1-8 tokens/rank (bf16 12.8 against 14.8 us at 1 token/rank,
    FP8 18.9 against 21.0), equal at 32, and 2-10% longer from 64 tokens/rank
    (bf16 at 128: 45.6 against 43.6 us; FP8 at 128: 66.0 against 59.9), where
    each source rank's CTAs rebuild that rank's layout; eager steps gain
    2-4 us up to 32 tokens/rank."""
    Tr = T // R
    return Tr <= 32 and (R - 1) * Tr <= 4096 and (dtype != "bf16" or T < 2048)


class EpPipeline:
    def __init__(self, T: int, H: int, k: int, E: int, R: int, G: int | None = None,
                 layout: str = "rank_major", dtype: str = "bf16", device="cuda", fused: bool | None = None,
                 combine_fmt: str = "bf16", two_level: bool = False):
        """fused: layout and dispatch in one ep_layout_dispatch launch (True),
        as two calls (False), or where the one launch is the faster (None)."""
        if fused is None:
            fused = one_launch_layout_dispatch(T, R, dtype) and not two_level
        self.p = ep.problem(T, H, k, E, R, G)
        # node-forwarding dispatch and combine (rank-major bf16 only)
        self.two_level = two_level
        if two_level and (layout != "rank_major" or dtype != "bf16" or combine_fmt != "bf16" or fused):
            raise ValueError("the two-level path is rank-major bf16 with a bf16 combine")
        self.fused = fused   # layout + dispatch in one launch (ep_layout_dispatch)
        self.combine_fmt = combine_fmt   # "bf16", or a low-precision wire format: "mxfp8", "nvfp4"
        self.layout, self.dtype = layout, dtype
        self.T, self.H, self.k, self.E, self.R = T, H, k, E, R
        self.rows = ep.ep_recv_rows(self.p, layout)
        self.buf = ep.LayoutBuffers(self.p, device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.algo = torch.zeros(R, dtype=torch.int64, device=device)
        self.phys = torch.zeros(R, dtype=torch.int64, device=device)
        if dtype == "bf16":
            self.recv = torch.empty((self.rows, H), dtype=torch.bfloat16, device=device)
            self.recv_scales = None
            self.y = self.recv
        else:
            self.recv = torch.empty((self.rows, H), dtype=torch.uint8, device=device)
            self.recv_scales = torch.empty((self.rows, H // 128), dtype=torch.float32, device=device)
            self.y = torch.empty((self.rows, H), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        if two_level:
            self.stage = torch.empty((ep.ep_stage_rows(self.p), H), dtype=torch.bfloat16, device=device)
        if combine_fmt != "bf16":
            qs, ss, sdt = ep.wire_shapes(self.p, layout, combine_fmt)
            self.wq = torch.empty(qs, dtype=torch.uint8, device=device)
            self.ws = torch.empty(ss, dtype=sdt, device=device)
        self._calls = {}   # bound library calls, see _run

    def _run(self, name, tensors, stream, make):
        """Issues library call `name`: the first time for these input tensors
        and this stream its arguments are checked and marshalled (`make`
        under ep.binding()); later steps replay the bound call, which keeps the
        host cost of a step to a few microseconds per launch."""
        key = (name, ep._stream(stream)) + tuple(
            None if t is None else (t.data_ptr(), t.numel(), t.dtype) for t in tensors)
        b = self._calls.get(key)
        if b is None:
            if len(self._calls) > 256:
                self._calls.clear()
            with ep.binding():
                b = make()
            self._calls[key] = b
        b()

    # individual steps (each enqueues on `stream`)
    def layout_step(self, topk_idx, stream=None):
        b = self.buf
        self._run("layout", (topk_idx,), stream, lambda: ep.ep_layout(
            self.p, topk_idx, b.is_token_in_rank, b.tokens_per_rank, b.tokens_per_expert, b.tokens_per_node,
            b.recv_tokens_per_rank, b.rank_slot, b.token_major_offset, b.expert_slot, b.workspace, self.status,
            stream, b.algo_per_rank, b.physical_exact_per_rank, b.node_slot))

    def rdma_step(self, topk_idx, stream=None):
        self._run("rdma", (topk_idx,), stream, lambda: ep.ep_rdma_token_count(
            self.p, topk_idx, self.algo, self.phys, self.status, stream))

    def dispatch_step(self, x, topk_idx, stream=None):
        if self.two_level:
            self._run("dispatch2", (x,), stream, lambda: ep.ep_dispatch_two_level(
                self.p, x, self.buf.rank_slot, self.buf.node_slot, self.stage, self.recv, self.status, stream))
            return
        self._run("dispatch", (x, topk_idx), stream, lambda: ep.ep_dispatch(
            self.p, self.layout, self.dtype, x, topk_idx, self.buf.rank_slot, self.buf.expert_slot, self.recv,
            self.recv_scales, self.status, stream))

    def expert_step(self, topk_idx=None, stream=None):
        if self.dtype != "bf16":
            self._run("expert", (topk_idx,), stream, lambda: ep.ep_dequant_fp8(
                self.p, self.layout, topk_idx, self.buf.rank_slot, self.buf.expert_slot, self.recv,
                self.recv_scales, self.y, stream))

    def wire_step(self, topk_idx, stream=None):
        """Expert-side cast of the expert outputs to the combine wire format."""
        if self.combine_fmt != "bf16":
            self._run("wire", (topk_idx,), stream, lambda: ep.ep_combine_quantize(
                self.p, self.layout, self.combine_fmt, self.y, topk_idx, self.buf.rank_slot, self.buf.expert_slot,
                self.wq, self.ws, stream))

    def combine_step(self, topk_idx, topk_weights, stream=None, out=None):
        out = self.out if out is None else out
        if self.two_level:
            self._run("combine2", (topk_idx, topk_weights, out), stream, lambda: ep.ep_combine_two_level(
                self.p, self.y, topk_idx, topk_weights, self.buf.rank_slot, self.buf.node_slot, self.stage, out,
                self.status, stream))
        elif self.combine_fmt == "bf16":
            self._run("combine", (topk_idx, topk_weights, out), stream, lambda: ep.ep_combine(
                self.p, self.layout, self.y, topk_idx, topk_weights, self.buf.rank_slot, self.buf.expert_slot, out,
                self.status, stream))
        else:
            self._run("combine_wire", (topk_idx, topk_weights, out), stream, lambda: ep.ep_combine_wire(
                self.p, self.layout, self.combine_fmt, self.wq, self.ws, topk_idx, topk_weights,
                self.buf.rank_slot, self.buf.expert_slot, out, self.status, stream))
        return out

    def layout_dispatch_step(self, x, topk_idx, stream=None):
        self._run("layout_dispatch", (x, topk_idx), stream, lambda: ep.ep_layout_dispatch(
            self.p, self.layout, self.dtype, x, topk_idx, self.buf, self.recv, self.recv_scales, self.status,
            stream))

    def step(self, x, topk_idx, topk_weights, stream=None, out=None):
        # the layout also yields the RDMA token counts (buf.algo_per_rank,
        # buf.physical_exact_per_rank); rdma_step is the standalone call
        if self.fused:
            self.layout_dispatch_step(x, topk_idx, stream)
        else:
            self.layout_step(topk_idx, stream)
            self.dispatch_step(x, topk_idx, stream)
        self.expert_step(topk_idx, stream)
        self.wire_step(topk_idx, stream)
        return self.combine_step(topk_idx, topk_weights, stream, out)

    def capture(self, x, topk_idx, topk_weights, warmup: int = 2, steps: int = 1):
        """Records `steps` steps into one CUDA graph (after `warmup` eager steps
        on a side stream) and returns it; graph.replay() re-runs them on the
        same buffers.  Launch latency, not bandwidth, bounds small batches,
        and one graph launch replaces the steps' kernel launches."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(warmup):
                self.step(x, topk_idx, topk_weights, s)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(steps):
                self.step(x, topk_idx, topk_weights, torch.cuda.current_stream())
        return g

    def kernels_per_step(self) -> int:
        """Library kernels one step launches (layout 2 — RDMA counts
        included —, dispatch 1, or the two fused into 1; FP8 identity expert
        1; wire-format cast 1; combine 1)."""
        return ((3 if self.fused else 4) + (1 if self.dtype != "bf16" else 0) +
                (1 if self.combine_fmt != "bf16" else 0) + (2 if self.two_level else 0))


class HostBatchRunner:
    """Runs the hot path over batches held in (pinned) host memory.

    Each batch's inputs are copied host -> device on one stream, its kernels
    run on a second, and its combined output is copied device -> host on a
    third; with two device slots for inputs and outputs, the copies of batch
    i+1 and of batch i-1 overlap the kernels of batch i.  The kernels of
    consecutive batches stay ordered on the compute stream (they share the
    pipeline's layout and receive buffers).
    """

    def __init__(self, pipe: EpPipeline, slots: int = 2, device="cuda"):
        self.pipe = pipe
        self.slots = slots
        T, H, k = pipe.T, pipe.H, pipe.k
        self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(device) for _ in range(3))
        self.x = [torch.empty((T, H), dtype=torch.bfloat16, device=device) for _ in range(slots)]
        self.idx = [torch.empty((T, k), dtype=torch.int64, device=device) for _ in range(slots)]
        self.w = [torch.empty((T, k), dtype=torch.float32, device=device) for _ in range(slots)]
        self.out = [torch.empty((T, H), dtype=torch.bfloat16, device=device) for _ in range(slots)]
        ev = lambda: [torch.cuda.Event() for _ in range(slots)]
        self.in_ready, self.comp_done, self.out_done = ev(), ev(), ev()
        self.used = [False] * slots

    def run(self, batches):
        """batches: iterable of (x, topk_idx, topk_weights, out) host tensors
        (x / out viewed as int16 or bfloat16).  Returns after enqueueing;
        synchronize (or wait on self.s_out) before reading the outputs."""
        for i, (xh, ih, wh, oh) in enumerate(batches):
            s = i % self.slots
            if self.used[s]:
                self.s_in.wait_event(self.comp_done[s])      # slot's inputs no longer read
            with torch.cuda.stream(self.s_in):
                self.x[s].view(xh.dtype).copy_(xh, non_blocking=True)
                self.idx[s].copy_(ih, non_blocking=True)
                self.w[s].copy_(wh, non_blocking=True)
                self.in_ready[s].record(self.s_in)
            self.s_comp.wait_event(self.in_ready[s])
            if self.used[s]:
                self.s_comp.wait_event(self.out_done[s])     # slot's output copied out
            self.pipe.step(self.x[s], self.idx[s], self.w[s], self.s_comp, out=self.out[s])
            self.comp_done[s].record(self.s_comp)
            self.s_out.wait_event(self.comp_done[s])
            with torch.cuda.stream(self.s_out):
                oh.copy_(self.out[s].view(oh.dtype), non_blocking=True)
                self.out_done[s].record(self.s_out)
            self.used[s] = True
