"""CPU oracle for MoE expert-parallel dispatch layout, dispatch and combine.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg load this module; the CUDA library never does, and the two
share no code.  The arithmetic lives in ``ep_oracle.c`` (plain sequential C,
compiled with gcc); this module only marshals numpy arrays into it.

bf16 arrays are uint16 bit patterns; FP8 payloads are uint8 e4m3 codes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_LIB = os.path.join(_HERE, "libep_oracle.so")
_lock = threading.Lock()
_lib = None

RANK_MAJOR, EXPERT_MAJOR = 0, 1
BF16, FP8 = 0, 1
WIRE_MXFP8, WIRE_NVFP4 = 1, 2
_WIRES = {"mxfp8": WIRE_MXFP8, "nvfp4": WIRE_NVFP4}
BAD_EXPERT, DUP_EXPERT, BAD_SLOT = 1, 2, 4

_LAYOUTS = {"rank_major": RANK_MAJOR, "expert_major": EXPERT_MAJOR}
_DTYPES = {"bf16": BF16, "fp8_e4m3": FP8}


def build(force: bool = False) -> str:
    """Compile ep_oracle.c into libep_oracle.so (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_layout.argtypes = [i64] * 5 + [p] * 10
            lib.oracle_layout.restype = i32
            lib.oracle_rdma_token_count.argtypes = [i64] * 5 + [p] * 3
            lib.oracle_rdma_token_count.restype = i32
            lib.oracle_rdma_physical_formula.argtypes = [i64, i64]
            lib.oracle_rdma_physical_formula.restype = ctypes.c_double
            lib.oracle_dispatch.argtypes = [i64] * 6 + [i32, i32] + [p] * 6 + [i64, i64]
            lib.oracle_dispatch.restype = i32
            lib.oracle_dequant_fp8.argtypes = [i64] * 4 + [i32] + [p] * 4
            lib.oracle_dequant_fp8.restype = i32
            lib.oracle_combine.argtypes = [i64] * 6 + [i32] + [p] * 7 + [i64, i64]
            lib.oracle_combine.restype = i32
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
            lib.oracle_bf16_from_double.restype = ctypes.c_uint16
            lib.oracle_quant_fp8_row.argtypes = [i64, p, p, p]
            lib.oracle_quant_fp8_row.restype = None
            lib.oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_decode.restype = ctypes.c_double
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_decode.restype = ctypes.c_double
            lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_quant_mxfp8_row.argtypes = [i64, p, p, p]
            lib.oracle_quant_mxfp8_row.restype = None
            lib.oracle_quant_nvfp4_row.argtypes = [i64, p, p, p]
            lib.oracle_quant_nvfp4_row.restype = None
            lib.oracle_combine_wire.argtypes = [i64] * 6 + [i32, i32] + [p] * 8 + [i64, i64]
            lib.oracle_combine_wire.restype = i32
            lib.oracle_quant_wire_rows.argtypes = [i32, i64, i64, p, p, p, p]
            lib.oracle_quant_wire_rows.restype = i32
            lib.oracle_dispatch_two_level.argtypes = [i64] * 6 + [p] * 5
            lib.oracle_dispatch_two_level.restype = i32
            lib.oracle_combine_two_level.argtypes = [i64] * 6 + [p] * 8 + [i64, i64]
            lib.oracle_combine_two_level.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _check(st):
    if st < 0:
        raise ValueError("oracle: arguments do not describe a problem")
    return st


def layout(topk_idx: np.ndarray, E: int, R: int, G: int, want_offsets: bool = True):
    """Dispatch layout of all source ranks. Returns (dict of arrays, status bits)."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, k = topk_idx.shape
    N = R // G if G and R % G == 0 else 1
    out = {
        "is_token_in_rank": np.zeros((T, R), np.uint8),
        "tokens_per_rank": np.zeros((R, R), np.int32),
        "tokens_per_expert": np.zeros((R, E), np.int32),
        "tokens_per_node": np.zeros((R, N), np.int32),
        "recv_tokens_per_rank": np.zeros((R,), np.int32),
        "rank_slot": np.zeros((T, R), np.int32),
        "token_major_offset": np.zeros((T, R), np.int32) if want_offsets else None,
        "expert_slot": np.zeros((T, k), np.int32),
        "node_slot": np.zeros((T, N), np.int32),
    }
    st = _load().oracle_layout(T, k, E, R, G, _ptr(topk_idx),
                               *[_ptr(out[n]) for n in ("is_token_in_rank", "tokens_per_rank",
                                                        "tokens_per_expert", "tokens_per_node",
                                                        "recv_tokens_per_rank", "rank_slot",
                                                        "token_major_offset", "expert_slot", "node_slot")])
    return out, _check(st)


def rdma_token_count(topk_idx: np.ndarray, E: int, R: int, G: int):
    """(algo_per_rank int64 [R], physical_exact_per_rank int64 [R], status)."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, k = topk_idx.shape
    algo = np.zeros(R, np.int64)
    phys = np.zeros(R, np.int64)
    st = _load().oracle_rdma_token_count(T, k, E, R, G, _ptr(topk_idx), _ptr(algo), _ptr(phys))
    return algo, phys, _check(st)


def rdma_physical_formula(algo: int, num_nodes: int) -> float:
    return _load().oracle_rdma_physical_formula(int(algo), int(num_nodes))


def recv_rows(T: int, E: int, R: int, layout_name: str) -> int:
    Tr = T // R
    return (R if layout_name == "rank_major" else E) * R * Tr


def dispatch(x, topk_idx, lay, E, R, G, layout_name="rank_major", dtype="bf16", recv=None,
             recv_scales=None, poison=True, t0=0, t1=None):
    """Dispatch tokens [t0, t1) into a fresh (poisoned) buffer, or into `recv`.
    Returns (recv, recv_scales, status)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, H = x.shape
    k = topk_idx.shape[1]
    rows = recv_rows(T, E, R, layout_name)
    if recv is None:
        if dtype == "bf16":
            recv = np.full((rows, H), 0xFFFF, np.uint16) if poison else np.zeros((rows, H), np.uint16)
        else:
            recv = np.full((rows, H), 0xFF, np.uint8) if poison else np.zeros((rows, H), np.uint8)
    if dtype == "fp8_e4m3" and recv_scales is None:
        recv_scales = np.full((rows, H // 128), np.nan, np.float32)
    st = _load().oracle_dispatch(T, H, k, E, R, G, _LAYOUTS[layout_name], _DTYPES[dtype], _ptr(x),
                                 _ptr(topk_idx), _ptr(lay["rank_slot"]), _ptr(lay["expert_slot"]),
                                 _ptr(recv), _ptr(recv_scales), int(t0), int(T if t1 is None else t1))
    return recv, recv_scales, _check(st)


def dequant_fp8(q, s, lay, T, E, R, layout_name="rank_major", y=None):
    """Identity expert for FP8 payloads (live rows only). Returns y uint16."""
    rows, H = q.shape
    if y is None:
        y = np.zeros((rows, H), np.uint16)
    counts = lay["tokens_per_rank"] if layout_name == "rank_major" else lay["tokens_per_expert"]
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    st = _load().oracle_dequant_fp8(T, H, E, R, _LAYOUTS[layout_name], _ptr(counts), _ptr(q),
                                    _ptr(np.ascontiguousarray(s, dtype=np.float32)), _ptr(y))
    _check(st)
    return y


def combine(y, topk_idx, topk_weights, lay, E, R, G, layout_name="rank_major", t0=0, t1=None,
            want_f64=False):
    """Weighted combine of tokens [t0, t1). Returns (out_bf16 [T,H], out_f64 or None, status);
    rows outside [t0, t1) are left zero."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, k = topk_idx.shape
    H = y.shape[1]
    t1 = T if t1 is None else t1
    out = np.zeros((T, H), np.uint16)
    out64 = np.zeros((T, H), np.float64) if want_f64 else None
    st = _load().oracle_combine(T, H, k, E, R, G, _LAYOUTS[layout_name], _ptr(y), _ptr(topk_idx),
                                _ptr(topk_weights), _ptr(lay["rank_slot"]), _ptr(lay["expert_slot"]),
                                _ptr(out), _ptr(out64), t0, t1)
    return out, out64, _check(st)


def quant_fp8_row(x_row: np.ndarray):
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    H = x_row.shape[0]
    q = np.zeros(H, np.uint8)
    s = np.zeros(H // 128, np.float32)
    _load().oracle_quant_fp8_row(H, _ptr(x_row), _ptr(q), _ptr(s))
    return q, s


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e4m3_decode(c: int) -> float:
    return float(_load().oracle_e4m3_decode(int(c)))


def bf16_from_double(v: float) -> int:
    return int(_load().oracle_bf16_from_double(float(v)))


def e8m0_decode(c: int) -> float:
    return float(_load().oracle_e8m0_decode(int(c)))


def e2m1_decode(c: int) -> float:
    return float(_load().oracle_e2m1_decode(int(c)))


def e2m1_encode(v: float) -> int:
    return int(_load().oracle_e2m1_encode(float(v)))


def wire_row_shapes(H: int, fmt: str):
    """(payload bytes, scale count, scale numpy dtype) of one wire row."""
    if fmt == "mxfp8":
        return H, H // 32, np.uint8
    return H // 2, H // 16, np.uint16


def quant_wire_row(y_row: np.ndarray, fmt: str):
    """Cast one bf16 row (uint16 bits) to a wire format: (codes, scales)."""
    y_row = np.ascontiguousarray(y_row, dtype=np.uint16)
    H = y_row.shape[0]
    qb, ns, sdt = wire_row_shapes(H, fmt)
    q = np.zeros(qb, np.uint8)
    s = np.zeros(ns, sdt)
    fn = _load().oracle_quant_mxfp8_row if fmt == "mxfp8" else _load().oracle_quant_nvfp4_row
    fn(H, _ptr(y_row), _ptr(q), _ptr(s))
    return q, s


def quant_wire_rows(y: np.ndarray, rows, fmt: str, q=None, s=None):
    """Cast the listed rows of y [nrows, H] into (q [nrows, qb], s [nrows, ns])."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    nrows, H = y.shape
    qb, ns, sdt = wire_row_shapes(H, fmt)
    if q is None:
        q = np.zeros((nrows, qb), np.uint8)
    if s is None:
        s = np.zeros((nrows, ns), sdt)
    rows = np.ascontiguousarray(np.asarray(list(rows) if not isinstance(rows, np.ndarray) else rows, np.int64))
    _check(_load().oracle_quant_wire_rows(_WIRES[fmt], H, rows.size, _ptr(rows), _ptr(y), _ptr(q), _ptr(s)))
    return q, s


def combine_wire(q, s, topk_idx, topk_weights, lay, E, R, G, fmt, H, layout_name="rank_major", t0=0, t1=None,
                 want_f64=False):
    """Weighted combine from a wire-format buffer, tokens [t0, t1)."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, k = topk_idx.shape
    t1 = T if t1 is None else t1
    out = np.zeros((T, H), np.uint16)
    out64 = np.zeros((T, H), np.float64) if want_f64 else None
    st = _load().oracle_combine_wire(T, H, k, E, R, G, _LAYOUTS[layout_name], _WIRES[fmt],
                                     _ptr(np.ascontiguousarray(q)), _ptr(np.ascontiguousarray(s)),
                                     _ptr(topk_idx), _ptr(topk_weights), _ptr(lay["rank_slot"]),
                                     _ptr(lay["expert_slot"]), _ptr(out), _ptr(out64), t0, t1)
    return out, out64, _check(st)


def stage_rows(T: int, R: int, G: int) -> int:
    """Rows of the node-major staging buffer [N][R src][Tr]."""
    return (R // G) * R * (T // R)


def dispatch_two_level(x, lay, E, R, G, k):
    """Two-hop dispatch. Returns (stage, recv), both poisoned (0xFFFF) where unwritten."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = x.shape
    stage = np.full((stage_rows(T, R, G), H), 0xFFFF, np.uint16)
    recv = np.full((R * R * (T // R), H), 0xFFFF, np.uint16)
    st = _load().oracle_dispatch_two_level(T, H, k, E, R, G, _ptr(x), _ptr(lay["rank_slot"]),
                                           _ptr(lay["node_slot"]), _ptr(stage), _ptr(recv))
    _check(st)
    return stage, recv


def combine_two_level(y, topk_idx, topk_weights, lay, E, R, G, t0=0, t1=None, want_f64=False, stage=None):
    """Two-hop combine of tokens [t0, t1). Returns (out_bf16, out_f64 or None, stage, status).
    stage: the staging buffer to write the node partials into (only the rows
    of tokens [t0, t1) are written); by default a fresh one filled with 0xFFFF."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    topk_weights = np.ascontiguousarray(topk_weights, dtype=np.float32)
    T, k = topk_idx.shape
    H = y.shape[1]
    t1 = T if t1 is None else t1
    if stage is None:
        stage = np.full((stage_rows(T, R, G), H), 0xFFFF, np.uint16)
    assert stage.shape == (stage_rows(T, R, G), H) and stage.dtype == np.uint16
    out = np.zeros((T, H), np.uint16)
    out64 = np.zeros((T, H), np.float64) if want_f64 else None
    st = _load().oracle_combine_two_level(T, H, k, E, R, G, _ptr(y), _ptr(topk_idx), _ptr(topk_weights),
                                          _ptr(lay["rank_slot"]), _ptr(lay["node_slot"]), _ptr(stage),
                                          _ptr(out), _ptr(out64), t0, t1)
    return out, out64, stage, _check(st)
