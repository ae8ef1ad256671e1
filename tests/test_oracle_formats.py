"""Pins for the oracle's number formats: OCP E4M3 and bf16 rounding.

The references here are the format definitions themselves (OCP 8-bit
floating point E4M3: bias 7, largest finite 448, S.1111.111 = NaN,
subnormals m/8 * 2^-6; bf16: the upper half of an IEEE binary32) and
torch's CPU conversions, which are independent library routines.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_05_gb300.inputs import bf16_bits_from_f32, f32_from_bf16_bits


def test_e4m3_decode_spot_values():
    # values read off the format definition
    assert oracle.e4m3_decode(0x7E) == 448.0          # S.1111.110, largest finite
    assert oracle.e4m3_decode(0xFE) == -448.0
    assert oracle.e4m3_decode(0x38) == 1.0            # E=7, M=0
    assert oracle.e4m3_decode(0x40) == 2.0
    assert oracle.e4m3_decode(0x77) == 240.0          # (1 + 7/8) * 2^7
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_decode(0x00) == 0.0
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_decode(c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(mine)
    assert np.all(both_nan | (ref == mine))


def test_e4m3_encode_roundtrips_every_finite_code():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        v = oracle.e4m3_decode(c)
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_e4m3_ties_go_to_even():
    # midpoint between consecutive codes c and c+1 (same sign, below 448)
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2
        want = c if (c & 1) == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want, (hex(c), mid)
        assert oracle.e4m3_encode(-mid) == want | 0x80


def test_e4m3_saturates():
    for v in [448.0, 449.0, 463.99, 464.0, 470.0, 480.0, 1e6, 3.0e38, float("inf")]:
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE


def test_e4m3_encode_matches_torch_in_range():
    # torch's float32 -> float8_e4m3fn is round-to-nearest-even and agrees
    # with a saturating conversion below the 448/480 midpoint.
    rng = np.random.default_rng(7)
    mags = np.exp2(rng.uniform(-14, np.log2(463.9), 20000)).astype(np.float32)
    vals = mags * rng.choice([-1, 1], mags.shape).astype(np.float32)
    # every bf16 pattern whose value lies below 464 in magnitude
    allb = f32_from_bf16_bits(np.arange(65536, dtype=np.uint16))
    allb = allb[np.isfinite(allb) & (np.abs(allb) < 464)]
    vals = np.concatenate([vals, allb]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_encode(v) for v in vals], dtype=np.uint8)
    bad = np.nonzero(ref != mine)[0]
    assert bad.size == 0, [(float(vals[i]), int(ref[i]), int(mine[i])) for i in bad[:5]]


def test_bf16_from_double_matches_torch_on_float32_values():
    # For doubles that are exact float32 values torch's float32 -> bf16 is a
    # single round-to-nearest-even.
    rng = np.random.default_rng(3)
    u = rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([oracle.bf16_from_double(float(v)) for v in f], dtype=np.uint16)
    bad = np.nonzero(ref != mine)[0]
    assert bad.size == 0, [(float(f[i]), hex(ref[i]), hex(mine[i])) for i in bad[:5]]


def test_bf16_from_double_rounds_once():
    # 1 + 2^-8 + 2^-30 lies just above the midpoint of 1.0 and 1 + 2^-7: one
    # rounding gives 0x3F81; going through float32 first would land on the
    # midpoint and round to even, 0x3F80.
    assert oracle.bf16_from_double(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert oracle.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80       # exact tie -> even
    assert oracle.bf16_from_double(1.0 + 3 * 2.0 ** -8) == 0x3F82   # tie -> even (up)
    assert oracle.bf16_from_double(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == 0xBF81
    # largest finite and overflow
    assert oracle.bf16_from_double((2 - 2.0 ** -7) * 2.0 ** 127) == 0x7F7F
    assert oracle.bf16_from_double((2 - 2.0 ** -8) * 2.0 ** 127) == 0x7F80
    # subnormals: smallest, half of smallest (tie -> 0), min normal
    assert oracle.bf16_from_double(2.0 ** -133) == 0x0001
    assert oracle.bf16_from_double(2.0 ** -134) == 0x0000
    assert oracle.bf16_from_double(1.5 * 2.0 ** -133) == 0x0002
    assert oracle.bf16_from_double(2.0 ** -126) == 0x0080
    assert oracle.bf16_from_double(0.0) == 0 and oracle.bf16_from_double(-0.0) == 0x8000


def test_generator_bf16_cast_matches_torch():
    rng = np.random.default_rng(11)
    f = rng.standard_normal(100000, dtype=np.float32) * np.float32(3.0)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_bits_from_f32(f), ref)
