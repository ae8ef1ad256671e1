"""One pass of the hot path through the C ABI, with its device buffers.

``EpPipeline`` allocates (with torch) every device buffer one problem needs
and runs layout -> RDMA token count -> dispatch -> identity expert ->
combine on one stream, every step in the library's kernels.  The identity
expert is free for a bf16 payload (combine reads the receive buffer itself)
and ``ep_dequant_fp8`` for an FP8 payload.
"""
from __future__ import annotations

import torch

from . import ep


class EpPipeline:
    def __init__(self, T: int, H: int, k: int, E: int, R: int, G: int | None = None,
                 layout: str = "rank_major", dtype: str = "bf16", device="cuda"):
        self.p = ep.problem(T, H, k, E, R, G)
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

    # individual steps (each enqueues on `stream`)
    def layout_step(self, topk_idx, stream=None):
        self.buf.run(self.p, topk_idx, self.status, stream)

    def rdma_step(self, topk_idx, stream=None):
        ep.ep_rdma_token_count(self.p, topk_idx, self.algo, self.phys, self.status, stream)

    def dispatch_step(self, x, topk_idx, stream=None):
        ep.ep_dispatch(self.p, self.layout, self.dtype, x, topk_idx, self.buf.rank_slot, self.buf.expert_slot,
                       self.recv, self.recv_scales, self.status, stream)

    def expert_step(self, stream=None):
        if self.dtype != "bf16":
            counts = self.buf.tokens_per_rank if self.layout == "rank_major" else self.buf.tokens_per_expert
            ep.ep_dequant_fp8(self.p, self.layout, counts, self.recv, self.recv_scales, self.y, stream)

    def combine_step(self, topk_idx, topk_weights, stream=None):
        ep.ep_combine(self.p, self.layout, self.y, topk_idx, topk_weights, self.buf.rank_slot,
                      self.buf.expert_slot, self.out, self.status, stream)

    def step(self, x, topk_idx, topk_weights, stream=None):
        self.layout_step(topk_idx, stream)
        self.rdma_step(topk_idx, stream)
        self.dispatch_step(x, topk_idx, stream)
        self.expert_step(stream)
        self.combine_step(topk_idx, topk_weights, stream)
        return self.out

    def kernels_per_step(self) -> int:
        """Library kernels one step launches (layout 2, RDMA count 1,
        dispatch 1, FP8 identity expert 1, combine 1)."""
        return 5 + (1 if self.dtype != "bf16" else 0)
