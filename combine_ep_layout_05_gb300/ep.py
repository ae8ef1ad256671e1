"""Python binding of the C ABI in include/ep.h (libep.so).

Argument marshalling only: every function here checks the tensors it is
given (device, dtype, contiguity, shape), passes their device pointers and
the current CUDA stream to the function of the same name in libep.so, and
raises ``EpError`` on a non-zero return code.  All computation happens in
the library's CUDA kernels; there is no fallback of any kind.  Importing this
module raises if libep.so has not been built
(``python -m combine_ep_layout_05_gb300.build``).
"""
from __future__ import annotations

import ctypes
import threading
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libep.so")

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_CUDA, EP_ERR_DEVICE = 0, 1, 2, 3
EP_STATUS_BAD_EXPERT, EP_STATUS_DUP_EXPERT, EP_STATUS_BAD_SLOT, EP_STATUS_TIMEOUT = 1, 2, 4, 8
EP_RANK_MAJOR, EP_EXPERT_MAJOR = 0, 1
EP_BF16, EP_FP8_E4M3 = 0, 1
EP_WIRE_MXFP8, EP_WIRE_NVFP4 = 1, 2
WIRES = {"mxfp8": EP_WIRE_MXFP8, "nvfp4": EP_WIRE_NVFP4}

LAYOUTS = {"rank_major": EP_RANK_MAJOR, "expert_major": EP_EXPERT_MAJOR}
DTYPES = {"bf16": EP_BF16, "fp8_e4m3": EP_FP8_E4M3}

# every symbol include/ep.h declares
EXPORTS = ("ep_last_error_string", "ep_get_status", "ep_recv_rows", "ep_layout_workspace_bytes", "ep_layout",
           "ep_rdma_token_count", "ep_rdma_physical_formula", "ep_dispatch", "ep_combine",
           "ep_dequant_fp8", "ep_layout_noalloc", "ep_layout_dispatch_workspace_bytes", "ep_layout_dispatch",
           "ep_selftest_wait_timeout", "ep_combine_quantize", "ep_combine_wire", "ep_stage_rows",
           "ep_dispatch_two_level", "ep_combine_two_level")


class EpError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with code {code}: {msg}")
        self.code = code


class ep_problem(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int64), ("hidden", ctypes.c_int64), ("num_topk", ctypes.c_int64),
                ("num_experts", ctypes.c_int64), ("num_ranks", ctypes.c_int64),
                ("gpus_per_node", ctypes.c_int64)]

    @property
    def T(self):
        return self.num_tokens

    @property
    def N(self):
        return self.num_ranks // self.gpus_per_node


def problem(T: int, H: int, k: int, E: int, R: int, G: int | None = None) -> ep_problem:
    return ep_problem(T, H, k, E, R, R if G is None else G)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m combine_ep_layout_05_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    pp = ctypes.POINTER(ep_problem)
    lib.ep_last_error_string.argtypes = []
    lib.ep_last_error_string.restype = ctypes.c_char_p
    lib.ep_get_status.argtypes = [P, P, P]
    lib.ep_get_status.restype = i
    lib.ep_recv_rows.argtypes = [pp, i]
    lib.ep_recv_rows.restype = i64
    lib.ep_layout_workspace_bytes.argtypes = [pp]
    lib.ep_layout_workspace_bytes.restype = sz
    lib.ep_layout.argtypes = [pp, P, P, P, P, P, P, P, P, P, P, P, P, P, sz, P, P]
    lib.ep_layout.restype = i
    lib.ep_rdma_token_count.argtypes = [pp, P, P, P, P, P]
    lib.ep_rdma_token_count.restype = i
    lib.ep_rdma_physical_formula.argtypes = [i64, i64]
    lib.ep_rdma_physical_formula.restype = ctypes.c_double
    lib.ep_dispatch.argtypes = [pp, i, i, P, P, P, P, P, P, P, P]
    lib.ep_dispatch.restype = i
    lib.ep_combine.argtypes = [pp, i, P, P, P, P, P, P, P, P]
    lib.ep_combine.restype = i
    lib.ep_dequant_fp8.argtypes = [pp, i, P, P, P, P, P, P, P]
    lib.ep_dequant_fp8.restype = i
    lib.ep_layout_noalloc.argtypes = [pp, P, P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.ep_layout_noalloc.restype = i
    lib.ep_layout_dispatch_workspace_bytes.argtypes = [pp]
    lib.ep_layout_dispatch_workspace_bytes.restype = sz
    lib.ep_layout_dispatch.argtypes = [pp, i, i] + [P] * 16 + [sz, P, P]
    lib.ep_layout_dispatch.restype = i
    lib.ep_selftest_wait_timeout.argtypes = [P, ctypes.c_uint32, P, P]
    lib.ep_selftest_wait_timeout.restype = i
    lib.ep_combine_quantize.argtypes = [pp, i, i, P, P, P, P, P, P, P]
    lib.ep_combine_quantize.restype = i
    lib.ep_combine_wire.argtypes = [pp, i, i, P, P, P, P, P, P, P, P, P]
    lib.ep_combine_wire.restype = i
    lib.ep_stage_rows.argtypes = [pp]
    lib.ep_stage_rows.restype = i64
    lib.ep_dispatch_two_level.argtypes = [pp, P, P, P, P, P, P, P]
    lib.ep_dispatch_two_level.restype = i
    lib.ep_combine_two_level.argtypes = [pp, P, P, P, P, P, P, P, P, P]
    lib.ep_combine_two_level.restype = i
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    """The loaded libep.so (argtypes set), for callers that pass raw pointers."""
    return _lib


def ep_last_error_string() -> str:
    return _lib.ep_last_error_string().decode()


def _check(fn, code):
    if code != EP_OK:
        raise EpError(fn, code, ep_last_error_string())


class Bound:
    """One library call with its arguments checked and marshalled once; calling
    it re-issues the call (the same buffers, the same stream).  Steps that
    repeat on fixed buffers replay these instead of re-marshalling ~15
    arguments per call in Python."""

    __slots__ = ("name", "fn", "args")

    def __init__(self, name, fn, args):
        self.name, self.fn, self.args = name, fn, args

    def __call__(self):
        code = self.fn(*self.args)
        if code != EP_OK:
            raise EpError(self.name, code, ep_last_error_string())


_bind = threading.local()


class binding:
    """Inside `with binding():` the wrappers below return a `Bound` instead of
    calling the library."""

    def __enter__(self):
        _bind.on = True
        return self

    def __exit__(self, *exc):
        _bind.on = False
        return False


def _call(name, fn, args):
    if getattr(_bind, "on", False):
        return Bound(name, fn, args)
    _check(name, fn(*args))


def _ptr(t, dtype=None, name="tensor", numel=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def ep_get_status(dev_status, stream=None) -> int:
    """Waits for `stream` and returns the EP_STATUS_* bits in `dev_status`
    (0 when the kernels found no error).  Raises EpError if the wait or the
    read fails."""
    word = ctypes.c_int32(0)
    code = _lib.ep_get_status(_ptr(dev_status, torch.int32, "dev_status", 1), ctypes.byref(word), _stream(stream))
    if code not in (EP_OK, EP_ERR_DEVICE):
        raise EpError("ep_get_status", code, ep_last_error_string())
    return int(word.value)


def ep_recv_rows(p: ep_problem, layout: str = "rank_major") -> int:
    r = _lib.ep_recv_rows(ctypes.byref(p), LAYOUTS[layout])
    if r < 0:
        raise EpError("ep_recv_rows", EP_ERR_INVALID_ARG, ep_last_error_string())
    return r


def ep_layout_workspace_bytes(p: ep_problem) -> int:
    return _lib.ep_layout_workspace_bytes(ctypes.byref(p))


def ep_rdma_physical_formula(algo_tokens: int, num_nodes: int) -> float:
    return _lib.ep_rdma_physical_formula(int(algo_tokens), int(num_nodes))


def ep_layout(p: ep_problem, topk_idx, is_token_in_rank=None, tokens_per_rank=None, tokens_per_expert=None,
              tokens_per_node=None, recv_tokens_per_rank=None, rank_slot=None, token_major_offset=None,
              expert_slot=None, workspace=None, dev_status=None, stream=None, algo_per_rank=None,
              physical_exact_per_rank=None, node_slot=None) -> None:
    T, k, E, R, N = p.num_tokens, p.num_topk, p.num_experts, p.num_ranks, p.N
    i32 = torch.int32
    return _call("ep_layout", _lib.ep_layout, (
        ctypes.byref(p), _ptr(topk_idx, torch.int64, "topk_idx", T * k),
        _ptr(is_token_in_rank, torch.uint8, "is_token_in_rank", T * R),
        _ptr(tokens_per_rank, i32, "tokens_per_rank", R * R),
        _ptr(tokens_per_expert, i32, "tokens_per_expert", R * E),
        _ptr(tokens_per_node, i32, "tokens_per_node", R * N),
        _ptr(recv_tokens_per_rank, i32, "recv_tokens_per_rank", R),
        _ptr(rank_slot, i32, "rank_slot", T * R),
        _ptr(token_major_offset, i32, "token_major_offset", T * R),
        _ptr(expert_slot, i32, "expert_slot", T * k),
        _ptr(node_slot, i32, "node_slot", T * N),
        _ptr(algo_per_rank, torch.int64, "algo_per_rank", R),
        _ptr(physical_exact_per_rank, torch.int64, "physical_exact_per_rank", R),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size() if workspace is not None else 0,
        _ptr(dev_status, i32, "dev_status", 1), _stream(stream)))


def ep_rdma_token_count(p: ep_problem, topk_idx, algo_per_rank, physical_exact_per_rank=None, dev_status=None,
                        stream=None) -> None:
    R = p.num_ranks
    return _call("ep_rdma_token_count", _lib.ep_rdma_token_count, (
        ctypes.byref(p), _ptr(topk_idx, torch.int64, "topk_idx", p.num_tokens * p.num_topk),
        _ptr(algo_per_rank, torch.int64, "algo_per_rank", R),
        _ptr(physical_exact_per_rank, torch.int64, "physical_exact_per_rank", R),
        _ptr(dev_status, torch.int32, "dev_status", 1), _stream(stream)))


def ep_dispatch(p: ep_problem, layout: str, dtype: str, x, topk_idx, rank_slot, expert_slot, recv,
                recv_scales=None, dev_status=None, stream=None) -> None:
    rows, H = ep_recv_rows(p, layout), p.hidden
    rdt = torch.bfloat16 if dtype == "bf16" else torch.uint8
    return _call("ep_dispatch", _lib.ep_dispatch, (
        ctypes.byref(p), LAYOUTS[layout], DTYPES[dtype], _ptr(x, torch.bfloat16, "x", p.num_tokens * H),
        _ptr(topk_idx, torch.int64, "topk_idx", p.num_tokens * p.num_topk),
        _ptr(rank_slot, torch.int32, "rank_slot", p.num_tokens * p.num_ranks),
        _ptr(expert_slot, torch.int32, "expert_slot", p.num_tokens * p.num_topk),
        _ptr(recv, rdt, "recv", rows * H),
        _ptr(recv_scales, torch.float32, "recv_scales", rows * (H // 128)),
        _ptr(dev_status, torch.int32, "dev_status", 1), _stream(stream)))


def ep_combine(p: ep_problem, layout: str, y, topk_idx, topk_weights, rank_slot, expert_slot, out,
               dev_status=None, stream=None) -> None:
    rows, H, T, k = ep_recv_rows(p, layout), p.hidden, p.num_tokens, p.num_topk
    return _call("ep_combine", _lib.ep_combine, (
        ctypes.byref(p), LAYOUTS[layout], _ptr(y, torch.bfloat16, "y", rows * H),
        _ptr(topk_idx, torch.int64, "topk_idx", T * k), _ptr(topk_weights, torch.float32, "topk_weights", T * k),
        _ptr(rank_slot, torch.int32, "rank_slot", T * p.num_ranks),
        _ptr(expert_slot, torch.int32, "expert_slot", T * k),
        _ptr(out, torch.bfloat16, "out", T * H), _ptr(dev_status, torch.int32, "dev_status", 1),
        _stream(stream)))


def ep_dequant_fp8(p: ep_problem, layout: str, topk_idx, rank_slot, expert_slot, recv, recv_scales, y,
                   stream=None) -> None:
    rows, H, T, k = ep_recv_rows(p, layout), p.hidden, p.num_tokens, p.num_topk
    return _call("ep_dequant_fp8", _lib.ep_dequant_fp8, (
        ctypes.byref(p), LAYOUTS[layout], _ptr(topk_idx, torch.int64, "topk_idx", T * k),
        _ptr(rank_slot, torch.int32, "rank_slot", T * p.num_ranks),
        _ptr(expert_slot, torch.int32, "expert_slot", T * k),
        _ptr(recv, torch.uint8, "recv", rows * H), _ptr(recv_scales, torch.float32, "recv_scales", rows * (H // 128)),
        _ptr(y, torch.bfloat16, "y", rows * H), _stream(stream)))


def ep_layout_dispatch_workspace_bytes(p: ep_problem) -> int:
    return _lib.ep_layout_dispatch_workspace_bytes(ctypes.byref(p))


def ep_layout_dispatch(p: ep_problem, layout: str, dtype: str, x, topk_idx, buf, recv, recv_scales=None,
                       dev_status=None, stream=None) -> None:
    """ep_layout + ep_dispatch in one launch; `buf` is a LayoutBuffers whose
    workspace holds at least ep_layout_dispatch_workspace_bytes(p) bytes."""
    T, k, E, R, N, H = p.num_tokens, p.num_topk, p.num_experts, p.num_ranks, p.N, p.hidden
    rows = ep_recv_rows(p, layout)
    i32 = torch.int32
    rdt = torch.bfloat16 if dtype == "bf16" else torch.uint8
    return _call("ep_layout_dispatch", _lib.ep_layout_dispatch, (
        ctypes.byref(p), LAYOUTS[layout], DTYPES[dtype], _ptr(x, torch.bfloat16, "x", T * H),
        _ptr(topk_idx, torch.int64, "topk_idx", T * k),
        _ptr(buf.is_token_in_rank, torch.uint8, "is_token_in_rank", T * R),
        _ptr(buf.tokens_per_rank, i32, "tokens_per_rank", R * R),
        _ptr(buf.tokens_per_expert, i32, "tokens_per_expert", R * E),
        _ptr(buf.tokens_per_node, i32, "tokens_per_node", R * N),
        _ptr(buf.recv_tokens_per_rank, i32, "recv_tokens_per_rank", R),
        _ptr(buf.rank_slot, i32, "rank_slot", T * R),
        _ptr(buf.token_major_offset, i32, "token_major_offset", T * R),
        _ptr(buf.expert_slot, i32, "expert_slot", T * k),
        _ptr(buf.node_slot, i32, "node_slot", T * N),
        _ptr(buf.algo_per_rank, torch.int64, "algo_per_rank", R),
        _ptr(buf.physical_exact_per_rank, torch.int64, "physical_exact_per_rank", R),
        _ptr(recv, rdt, "recv", rows * H), _ptr(recv_scales, torch.float32, "recv_scales", rows * (H // 128)),
        _ptr(buf.workspace, None, "workspace"), buf.workspace.numel(),
        _ptr(dev_status, i32, "dev_status", 1), _stream(stream)))


def wire_shapes(p: ep_problem, layout: str, fmt: str):
    """((rows, payload bytes per row), (rows, scales per row), scale dtype) of a wire buffer."""
    rows, H = ep_recv_rows(p, layout), p.hidden
    if fmt == "mxfp8":
        return (rows, H), (rows, H // 32), torch.uint8
    return (rows, H // 2), (rows, H // 16), torch.bfloat16


def ep_combine_quantize(p: ep_problem, layout: str, fmt: str, y, topk_idx, rank_slot, expert_slot, wq, wscales,
                        stream=None) -> None:
    (qr, qb), (sr, sn), sdt = wire_shapes(p, layout, fmt)
    T, k = p.num_tokens, p.num_topk
    return _call("ep_combine_quantize", _lib.ep_combine_quantize, (
        ctypes.byref(p), LAYOUTS[layout], WIRES[fmt], _ptr(y, torch.bfloat16, "y", qr * p.hidden),
        _ptr(topk_idx, torch.int64, "topk_idx", T * k), _ptr(rank_slot, torch.int32, "rank_slot", T * p.num_ranks),
        _ptr(expert_slot, torch.int32, "expert_slot", T * k), _ptr(wq, torch.uint8, "wq", qr * qb),
        _ptr(wscales, sdt, "wscales", sr * sn), _stream(stream)))


def ep_combine_wire(p: ep_problem, layout: str, fmt: str, wq, wscales, topk_idx, topk_weights, rank_slot,
                    expert_slot, out, dev_status=None, stream=None) -> None:
    (qr, qb), (sr, sn), sdt = wire_shapes(p, layout, fmt)
    T, k, H = p.num_tokens, p.num_topk, p.hidden
    return _call("ep_combine_wire", _lib.ep_combine_wire, (
        ctypes.byref(p), LAYOUTS[layout], WIRES[fmt], _ptr(wq, torch.uint8, "wq", qr * qb),
        _ptr(wscales, sdt, "wscales", sr * sn), _ptr(topk_idx, torch.int64, "topk_idx", T * k),
        _ptr(topk_weights, torch.float32, "topk_weights", T * k),
        _ptr(rank_slot, torch.int32, "rank_slot", T * p.num_ranks),
        _ptr(expert_slot, torch.int32, "expert_slot", T * k), _ptr(out, torch.bfloat16, "out", T * H),
        _ptr(dev_status, torch.int32, "dev_status", 1), _stream(stream)))


def ep_stage_rows(p: ep_problem) -> int:
    r = _lib.ep_stage_rows(ctypes.byref(p))
    if r < 0:
        raise EpError("ep_stage_rows", EP_ERR_INVALID_ARG, ep_last_error_string())
    return r


def ep_dispatch_two_level(p: ep_problem, x, rank_slot, node_slot, stage, recv, dev_status=None,
                          stream=None) -> None:
    T, H, R, N = p.num_tokens, p.hidden, p.num_ranks, p.N
    return _call("ep_dispatch_two_level", _lib.ep_dispatch_two_level, (
        ctypes.byref(p), _ptr(x, torch.bfloat16, "x", T * H), _ptr(rank_slot, torch.int32, "rank_slot", T * R),
        _ptr(node_slot, torch.int32, "node_slot", T * N), _ptr(stage, torch.bfloat16, "stage", ep_stage_rows(p) * H),
        _ptr(recv, torch.bfloat16, "recv", ep_recv_rows(p) * H), _ptr(dev_status, torch.int32, "dev_status", 1),
        _stream(stream)))


def ep_combine_two_level(p: ep_problem, y, topk_idx, topk_weights, rank_slot, node_slot, stage, out,
                         dev_status=None, stream=None) -> None:
    T, H, R, N, k = p.num_tokens, p.hidden, p.num_ranks, p.N, p.num_topk
    return _call("ep_combine_two_level", _lib.ep_combine_two_level, (
        ctypes.byref(p), _ptr(y, torch.bfloat16, "y", ep_recv_rows(p) * H),
        _ptr(topk_idx, torch.int64, "topk_idx", T * k), _ptr(topk_weights, torch.float32, "topk_weights", T * k),
        _ptr(rank_slot, torch.int32, "rank_slot", T * R), _ptr(node_slot, torch.int32, "node_slot", T * N),
        _ptr(stage, torch.bfloat16, "stage", ep_stage_rows(p) * H), _ptr(out, torch.bfloat16, "out", T * H),
        _ptr(dev_status, torch.int32, "dev_status", 1), _stream(stream)))


def ep_selftest_wait_timeout(words, polls: int, dev_status, stream=None) -> None:
    return _call("ep_selftest_wait_timeout", _lib.ep_selftest_wait_timeout,
                 (_ptr(words, torch.int32, "words", 2), int(polls), _ptr(dev_status, torch.int32, "dev_status", 1),
                  _stream(stream)))


class LayoutBuffers:
    """Device buffers for one ep_layout call (allocated with torch)."""

    def __init__(self, p: ep_problem, device="cuda", token_major_offset: bool = True):
        T, k, E, R, N = p.num_tokens, p.num_topk, p.num_experts, p.num_ranks, p.N
        i32 = dict(dtype=torch.int32, device=device)
        self.is_token_in_rank = torch.empty((T, R), dtype=torch.uint8, device=device)
        self.tokens_per_rank = torch.empty((R, R), **i32)
        self.tokens_per_expert = torch.empty((R, E), **i32)
        self.tokens_per_node = torch.empty((R, N), **i32)
        self.recv_tokens_per_rank = torch.empty((R,), **i32)
        self.rank_slot = torch.empty((T, R), **i32)
        self.token_major_offset = torch.empty((T, R), **i32) if token_major_offset else None
        self.expert_slot = torch.empty((T, k), **i32)
        self.node_slot = torch.empty((T, N), **i32)
        self.algo_per_rank = torch.empty((R,), dtype=torch.int64, device=device)
        self.physical_exact_per_rank = torch.empty((R,), dtype=torch.int64, device=device)
        # sized for ep_layout_dispatch too (the layout scratch plus a barrier word)
        self.workspace = torch.empty((max(16, ep_layout_dispatch_workspace_bytes(p)),), dtype=torch.uint8,
                                     device=device)

    def run(self, p: ep_problem, topk_idx, dev_status=None, stream=None):
        ep_layout(p, topk_idx, self.is_token_in_rank, self.tokens_per_rank, self.tokens_per_expert,
                  self.tokens_per_node, self.recv_tokens_per_rank, self.rank_slot, self.token_major_offset,
                  self.expert_slot, self.workspace, dev_status, stream, self.algo_per_rank,
                  self.physical_exact_per_rank, self.node_slot)
        return self
