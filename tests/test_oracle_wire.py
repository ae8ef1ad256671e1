"""Pins for the oracle's low-precision combine wire formats.

mxfp8: 32 e4m3 values sharing one e8m0 (power-of-two) scale; nvfp4: 16 e2m1
values with one bf16 scale ("MoE-EP Benchmark", environment reference,
MEGA_COMBINE_DTYPE).  References: the OCP MX formats' value tables, torch's
float8_e8m0fnu / float8_e4m3fn conversions, brute-force nearest-value search,
and exact closed forms of the combine.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_05_gb300 import inputs

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # OCP MX FP4 (E2M1) table


def test_e2m1_table():
    for c in range(8):
        assert oracle.e2m1_decode(c) == E2M1_MAGNITUDES[c]
        assert oracle.e2m1_decode(c | 8) == -E2M1_MAGNITUDES[c]
        assert oracle.e2m1_encode(E2M1_MAGNITUDES[c]) == c
        assert oracle.e2m1_encode(-E2M1_MAGNITUDES[c]) == c | 8


def _nearest_e2m1(v):
    """Brute force: nearest magnitude, ties to the even code (even mantissa),
    saturating at 6."""
    a = min(abs(v), 6.0)
    d = [abs(a - m) for m in E2M1_MAGNITUDES]
    best = min(d)
    cands = [c for c in range(8) if d[c] == best]
    c = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
    return c | (8 if np.signbit(v) else 0)


def test_e2m1_encode_matches_brute_force():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.uniform(-8, 8, 20000), np.arange(-7, 7.01, 0.125),
                           [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, 6.0, 1e9]]).astype(np.float32)
    for v in vals:
        assert oracle.e2m1_encode(float(v)) == _nearest_e2m1(float(v)), v


def test_e8m0_matches_torch():
    codes = torch.arange(255, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    mine = np.array([oracle.e8m0_decode(c) for c in range(255)])
    assert np.array_equal(ref, mine)
    assert np.isnan(oracle.e8m0_decode(255))


def _frexp_exp(a):
    return np.frexp(a)[1] - 1          # floor(log2 a) for a > 0


def test_mxfp8_row_matches_torch_steps():
    rng = np.random.default_rng(1)
    H = 1024
    for scale in (1e-6, 1.0, 3e4):
        y = inputs.bf16_bits_from_f32((rng.standard_normal(H) * scale).astype(np.float32))
        y[64:96] = 0                                           # an all-zero block
        q, s = oracle.quant_wire_row(y, "mxfp8")
        v = inputs.f32_from_bf16_bits(y).astype(np.float64).reshape(-1, 32)
        amax = np.abs(v).max(axis=1)
        X = np.where(amax > 0, np.clip(_frexp_exp(np.where(amax > 0, amax, 1)) - 8, -127, 127), -127)
        assert np.array_equal(s, (X + 127).astype(np.uint8))
        scaled = torch.from_numpy(np.ldexp(v, -X[:, None]).astype(np.float32)).clamp(-448, 448)
        ref = scaled.to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1).numpy()
        assert np.array_equal(q, ref)
        assert np.all(q[64:96] == 0) and s[2] == 0


def test_mxfp8_reconstruction_bound():
    rng = np.random.default_rng(2)
    y = inputs.bf16_bits_from_f32(rng.standard_normal(4096).astype(np.float32))
    q, s = oracle.quant_wire_row(y, "mxfp8")
    v = inputs.f32_from_bf16_bits(y).astype(np.float64)
    X = np.repeat([oracle.e8m0_decode(c) for c in s], 32)
    d = np.array([oracle.e4m3_decode(c) for c in q]) * X
    # half an e4m3 step of the scaled value (relative 2^-4 for normals,
    # 2^-10 absolute below), plus saturation of the block maximum at 448/512
    err = np.abs(v - d)
    assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(v), 2.0 ** -10 * X) + (64 / 512) * np.abs(v) * (np.abs(v) >= 448 * X))


def test_nvfp4_row_matches_brute_force_steps():
    rng = np.random.default_rng(3)
    H = 512
    for scale in (1e-3, 1.0, 100.0):
        y = inputs.bf16_bits_from_f32((rng.standard_normal(H) * scale).astype(np.float32))
        y[32:48] = 0
        q, s = oracle.quant_wire_row(y, "nvfp4")
        v = inputs.f32_from_bf16_bits(y).reshape(-1, 16)
        amax = torch.from_numpy(np.abs(v).max(axis=1).astype(np.float32))
        sb = torch.div(amax, torch.full_like(amax, 6.0)).to(torch.bfloat16)
        assert np.array_equal(s, sb.view(torch.int16).numpy().view(np.uint16))
        sf = sb.to(torch.float32)
        inv = torch.where(sf > 0, torch.div(torch.ones_like(sf), sf), torch.zeros_like(sf))
        p = (torch.from_numpy(v) * inv[:, None]).reshape(-1).numpy()
        codes = np.array([_nearest_e2m1(float(x)) for x in p], np.uint8)
        packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
        assert np.array_equal(q, packed)
        assert np.all(q[16:24] == 0) and s[2] == 0


def _layout(R, Tr, E, k, seed):
    idx, w = inputs.make_routing(R * Tr, E, k, seed=seed)
    lay, _ = oracle.layout(idx, E, R, R)
    return idx, w, lay


@pytest.mark.parametrize("fmt,H", [("mxfp8", 64), ("nvfp4", 64), ("nvfp4", 48)])
def test_combine_wire_closed_form(fmt, H):
    # every wire element decodes to 1.0 * 2^(row % 3): combine = sum of w * that
    # (nvfp4 rows need whole blocks of 16 only: H = 48 is a valid row)
    R, Tr, E, k = 2, 4, 8, 3
    idx, _, lay = _layout(R, Tr, E, k, 5)
    rows = R * R * Tr
    qb, ns, sdt = oracle.wire_row_shapes(H, fmt)
    q = np.zeros((rows, qb), np.uint8)
    s = np.zeros((rows, ns), sdt)
    for r in range(rows):
        if fmt == "mxfp8":
            q[r] = 0x38                     # e4m3 1.0
            s[r] = 127 + (r % 3)            # 2^(r % 3)
        else:
            q[r] = 0x22                     # two e2m1 1.0 codes
            s[r] = inputs.bf16_bits_from_f32(np.array([2.0 ** (r % 3)], np.float32))[0]
    w = (np.random.default_rng(0).integers(0, 64, (R * Tr, k)) / 32).astype(np.float32)
    _, out64, st = oracle.combine_wire(q, s, idx, w, lay, E, R, R, fmt, H, want_f64=True)
    assert st == 0
    for t in range(R * Tr):
        src = t // Tr
        exp = 0.0
        for j in range(k):
            r = int(idx[t, j]) // (E // R)
            row = (r * R + src) * Tr + lay["rank_slot"][t, r]
            exp += float(w[t, j]) * 2.0 ** (row % 3)
        assert np.all(out64[t] == exp)


@pytest.mark.parametrize("fmt,tol", [("mxfp8", 0.06), ("nvfp4", 0.2)])
def test_combine_wire_tracks_bf16_combine(fmt, tol):
    # the wire combine of quantised expert rows stays within the formats'
    # quantisation error of the bf16 combine (rel-L2, the pages' accuracy gate)
    R, Tr, H, E, k = 4, 16, 256, 32, 6
    idx, w, lay = _layout(R, Tr, E, k, 7)
    rows = R * R * Tr
    y = inputs.make_random_rows(rows, H, seed=7)
    _, ref64, _ = oracle.combine(y, idx, w, lay, E, R, R, want_f64=True)
    q, s = oracle.quant_wire_rows(y, range(rows), fmt)
    _, out64, st = oracle.combine_wire(q, s, idx, w, lay, E, R, R, fmt, H, want_f64=True)
    assert st == 0
    rel = np.linalg.norm(out64 - ref64) / np.linalg.norm(ref64)
    assert 0 < rel < tol, rel
