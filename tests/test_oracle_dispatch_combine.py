"""Pins for the oracle's dispatch (bf16 and FP8) and weighted combine.

References: the inverse-map property of dispatch (every live receive row is a
copy of its source token, every other row untouched), the FP8 format's error
bound and saturation, torch's float8 conversion, exact closed forms of the
combine with identity experts and dyadic weights, and a dense-matrix
restatement of the combine evaluated with a numpy matmul.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_ep_layout_05_gb300 import inputs


def _problem(R, Tr, H, E, k, seed=0, G=None, zipf=None):
    T = R * Tr
    x = inputs.make_tokens(T, H, seed=seed)
    idx, w = inputs.make_routing(T, E, k, seed=seed, zipf_s=zipf)
    return x, idx, w, (G or R)


# --------------------------------------------------------------------------
# dispatch
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout_name", ["rank_major", "expert_major"])
@pytest.mark.parametrize("R,Tr,H,E,k", [(4, 8, 256, 32, 4), (3, 5, 64, 12, 3), (8, 16, 128, 64, 8)])
def test_dispatch_inverse_map(layout_name, R, Tr, H, E, k):
    x, idx, _, G = _problem(R, Tr, H, E, k, seed=R + k)
    idx[::5, 0] = -1
    T = R * Tr
    lay, _ = oracle.layout(idx, E, R, G)
    recv, _, st = oracle.dispatch(x, idx, lay, E, R, G, layout_name=layout_name)
    assert st == 0
    nd = R if layout_name == "rank_major" else E
    seg = recv.reshape(nd, R, Tr, H)
    live = np.zeros((nd, R, Tr), bool)
    for src in range(R):
        toks = range(src * Tr, (src + 1) * Tr)
        for d in range(nd):
            if layout_name == "rank_major":
                want = [t for t in toks if any(e >= 0 and e // (E // R) == d for e in idx[t])]
            else:
                want = [t for t in toks if d in idx[t].tolist()]
            # the segment holds exactly these tokens, in token order, compacted
            for i, t in enumerate(want):
                assert np.array_equal(seg[d, src, i], x[t])
            live[d, src, :len(want)] = True
    assert np.all(seg[~live] == 0xFFFF)


def test_dispatch_fp8_payload_is_the_row_cast():
    R, Tr, H, E, k = 4, 4, 512, 16, 4
    x, idx, _, G = _problem(R, Tr, H, E, k, seed=9)
    lay, _ = oracle.layout(idx, E, R, G)
    for layout_name in ("rank_major", "expert_major"):
        q, s, st = oracle.dispatch(x, idx, lay, E, R, G, layout_name=layout_name, dtype="fp8_e4m3")
        assert st == 0
        b, _, _ = oracle.dispatch(x, idx, lay, E, R, G, layout_name=layout_name)
        live = np.any(b != 0xFFFF, axis=1)
        for row in np.nonzero(live)[0]:
            t = int(np.nonzero(np.all(x == b[row], axis=1))[0][0])
            qr, sr = oracle.quant_fp8_row(x[t])
            assert np.array_equal(q[row], qr) and np.array_equal(s[row], sr)
        assert np.all(q[~live] == 0xFF) and np.all(np.isnan(s[~live]))


# --------------------------------------------------------------------------
# FP8 cast
# --------------------------------------------------------------------------

def _dec(q):
    return np.array([oracle.e4m3_decode(c) for c in q])


def test_fp8_block_properties():
    rng = np.random.default_rng(1)
    H = 1024
    for scale in (1e-3, 1.0, 300.0):
        x = inputs.bf16_bits_from_f32((rng.standard_normal(H) * scale).astype(np.float32))
        q, s = oracle.quant_fp8_row(x)
        xf = inputs.f32_from_bf16_bits(x).astype(np.float64)
        d = _dec(q)
        for b in range(H // 128):
            blk = slice(b * 128, (b + 1) * 128)
            amax = np.abs(xf[blk]).max()
            assert s[b] == np.float32(np.float32(amax) / np.float32(448))
            # the largest element of each block lands on +-448
            assert np.abs(d[blk]).max() == 448.0
            # half an e4m3 step, relative 2^-4 for normals, 2^-10 * s below
            err = np.abs(xf[blk] - d[blk] * s[b])
            bound = np.maximum(2.0 ** -4 * np.abs(xf[blk]), 2.0 ** -10 * float(s[b])) * (1 + 2.0 ** -20) \
                + 2.0 ** -21 * np.abs(xf[blk])
            assert np.all(err <= bound)


def test_fp8_special_blocks():
    H = 256
    x = np.zeros(H, np.uint16)                        # zero block -> s = 0, q = 0
    x[128:] = inputs.bf16_bits_from_f32(np.full(128, 3.0, np.float32))   # constant block
    q, s = oracle.quant_fp8_row(x)
    assert s[0] == 0.0 and np.all(q[:128] == 0)
    assert s[1] == np.float32(3.0) / np.float32(448) and np.all(q[128:] == 0x7E)
    # negative zero keeps its sign bit
    x[:128] = 0x8000
    q, _ = oracle.quant_fp8_row(x)
    assert np.all(q[:128] == 0x80)


def test_fp8_cast_matches_torch_pipeline():
    # the same fp32 steps done with torch ops; the e4m3 conversion is torch's
    rng = np.random.default_rng(4)
    H = 7168
    x = inputs.bf16_bits_from_f32(rng.standard_normal(H).astype(np.float32))
    q, s = oracle.quant_fp8_row(x)
    xt = torch.from_numpy(inputs.f32_from_bf16_bits(x).copy()).view(-1, 128)
    amax = xt.abs().amax(dim=1)
    # tensor / tensor is a correctly rounded division (a Python scalar over
    # a tensor goes through a reciprocal and rounds twice)
    c448 = torch.full_like(amax, 448.0)
    st = torch.div(amax, c448)
    inv = torch.div(c448, amax)
    qt = (xt * inv[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(-1).numpy()
    assert np.array_equal(s, st.numpy())
    assert np.array_equal(q, qt)


def test_fp8_every_bf16_value_converts_like_torch():
    # one 448 per block makes inv = 1 exactly, so q is the plain e4m3 cast of
    # each bf16 value; all bf16 patterns with |v| <= 448 go through the row cast
    allb = np.arange(65536, dtype=np.uint16)
    v = inputs.f32_from_bf16_bits(allb)
    keep = allb[np.isfinite(v) & (np.abs(v) <= 448)]
    per = 127
    nblk = -(-keep.size // per)
    x = np.zeros(nblk * 128, np.uint16)
    for b in range(nblk):
        part = keep[b * per:(b + 1) * per]
        x[b * 128] = inputs.bf16_bits_from_f32(np.array([448.0], np.float32))[0]
        x[b * 128 + 1:b * 128 + 1 + part.size] = part
    q, s = oracle.quant_fp8_row(x)
    assert np.all(s == np.float32(1.0))
    ref = torch.from_numpy(inputs.f32_from_bf16_bits(x).copy()).to(torch.float8_e4m3fn)
    assert np.array_equal(q, ref.view(torch.uint8).numpy())


def test_fp8_dequant_identity_expert():
    R, Tr, H, E, k = 2, 4, 256, 8, 2
    x, idx, _, G = _problem(R, Tr, H, E, k, seed=2)
    lay, _ = oracle.layout(idx, E, R, G)
    q, s, _ = oracle.dispatch(x, idx, lay, E, R, G, layout_name="expert_major", dtype="fp8_e4m3")
    y = oracle.dequant_fp8(q, s, lay, R * Tr, E, R, layout_name="expert_major")
    # decode(q) has at most 4 significant bits and s 24: the fp64 product is
    # exact; y must be the bf16 value nearest to it (ties to an even code)
    rows = np.nonzero(np.any(q != 0xFF, axis=1))[0]
    assert rows.size == lay["tokens_per_expert"].sum()
    for row in rows[:8]:
        p = _dec(q[row]) * np.repeat(s[row].astype(np.float64), 128)
        yv = inputs.f32_from_bf16_bits(y[row]).astype(np.float64)
        up = inputs.f32_from_bf16_bits((y[row].astype(np.int64) + 1).astype(np.uint16)).astype(np.float64)
        dn = inputs.f32_from_bf16_bits((y[row].astype(np.int64) - 1).astype(np.uint16)).astype(np.float64)
        nz = p != 0
        err = np.abs(p - yv)
        assert np.all(err[nz] <= np.abs(p - up)[nz]) and np.all(err[nz] <= np.abs(p - dn)[nz])
        tie = nz & ((err == np.abs(p - up)) | (err == np.abs(p - dn)))
        assert np.all(y[row][tie] % 2 == 0)
        assert np.all(y[row][~nz] & 0x7FFF == 0)


# --------------------------------------------------------------------------
# combine
# --------------------------------------------------------------------------

def _dyadic_weights(T, k, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, 128, size=(T, k)) / 64.0).astype(np.float32)


@pytest.mark.parametrize("layout_name", ["rank_major", "expert_major"])
def test_combine_identity_closed_form(layout_name):
    R, Tr, H, E, k = 4, 6, 128, 32, 4
    x, idx, _, G = _problem(R, Tr, H, E, k, seed=3)
    idx[::7] = -1
    w = _dyadic_weights(R * Tr, k, 3)
    lay, _ = oracle.layout(idx, E, R, G)
    y, _, _ = oracle.dispatch(x, idx, lay, E, R, G, layout_name=layout_name)
    out, out64, st = oracle.combine(y, idx, w, lay, E, R, G, layout_name=layout_name, want_f64=True)
    assert st == 0
    wsum = np.where(idx >= 0, w, 0).astype(np.float64).sum(axis=1)
    exact = inputs.f32_from_bf16_bits(x).astype(np.float64) * wsum[:, None]
    assert np.array_equal(out64, exact)
    # x * sum(w) has at most 16 significant bits, so torch's float32 -> bf16
    # rounds it once
    # (compared as values: an empty or all-zero-weight sum is +0, x * 0 may be -0)
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(inputs.f32_from_bf16_bits(out), ref)
    assert np.all(out[::7] == 0)


def test_combine_dense_matmul_restatement():
    # out = M @ Y with M[t, row] the summed weight of t's entries that read
    # that row: a matrix product over the whole receive buffer
    R, Tr, H, E, k = 3, 5, 64, 12, 4
    x, idx, _, G = _problem(R, Tr, H, E, k, seed=8)
    w = inputs.make_uniform_weights(R * Tr, k, seed=8)
    lay, _ = oracle.layout(idx, E, R, G)
    for layout_name in ("rank_major", "expert_major"):
        nrows = (R if layout_name == "rank_major" else E) * R * Tr
        y = inputs.make_random_rows(nrows, H, seed=8)
        out, out64, st = oracle.combine(y, idx, w, lay, E, R, G, layout_name=layout_name, want_f64=True)
        assert st == 0
        T = R * Tr
        M = np.zeros((T, nrows))
        for t in range(T):
            src = t // Tr
            for j in range(k):
                e = int(idx[t, j])
                if layout_name == "rank_major":
                    r = e // (E // R)
                    row = (r * R + src) * Tr + lay["rank_slot"][t, r]
                else:
                    row = (e * R + src) * Tr + lay["expert_slot"][t, j]
                M[t, row] += float(w[t, j])
        ref = M @ inputs.f32_from_bf16_bits(y).astype(np.float64)
        np.testing.assert_allclose(out64, ref, rtol=1e-13, atol=1e-13)


def test_combine_linear_and_permutation_invariant():
    R, Tr, H, E, k = 2, 8, 64, 16, 4
    x, idx, _, G = _problem(R, Tr, H, E, k, seed=6)
    lay, _ = oracle.layout(idx, E, R, G)
    y = inputs.make_random_rows(E * R * Tr, H, seed=6)
    w1, w2 = _dyadic_weights(R * Tr, k, 1), _dyadic_weights(R * Tr, k, 2)
    f = lambda w, i=idx, l=lay: oracle.combine(y, i, w, l, E, R, G, layout_name="expert_major",
                                               want_f64=True)[1]
    assert np.array_equal(f(w1 + w2), f(w1) + f(w2))
    perm = np.random.default_rng(0).permutation(k)
    idx_p = np.ascontiguousarray(idx[:, perm])
    lay_p, _ = oracle.layout(idx_p, E, R, G)
    assert np.array_equal(f(w1), f(np.ascontiguousarray(w1[:, perm]), idx_p, lay_p))


def test_combine_rank_major_reads_one_row_per_rank():
    # two experts of a token on the same rank read the same row
    R, Tr, H, E, k = 2, 1, 16, 8, 2
    idx = np.array([[0, 1], [5, 2]], np.int64)       # t0: experts 0,1 both on rank 0
    lay, _ = oracle.layout(idx, E, R, R)
    y = np.zeros((R * R * Tr, H), np.uint16)
    y[0] = inputs.bf16_bits_from_f32(np.full(H, 2.0, np.float32))    # (r0, src0)
    y[2] = inputs.bf16_bits_from_f32(np.full(H, 4.0, np.float32))    # (r1, src0)
    y[1] = inputs.bf16_bits_from_f32(np.full(H, 8.0, np.float32))    # (r0, src1)
    y[3] = inputs.bf16_bits_from_f32(np.full(H, 16.0, np.float32))   # (r1, src1)
    w = np.array([[0.5, 0.25], [1.0, 2.0]], np.float32)
    _, out64, _ = oracle.combine(y, idx, w, lay, E, R, R, want_f64=True)
    assert np.all(out64[0] == 0.75 * 2.0)
    assert np.all(out64[1] == 1.0 * 16.0 + 2.0 * 8.0)


def test_combine_token_range():
    R, Tr, H, E, k = 2, 4, 32, 8, 2
    x, idx, w, G = _problem(R, Tr, H, E, k, seed=1)
    lay, _ = oracle.layout(idx, E, R, G)
    y, _, _ = oracle.dispatch(x, idx, lay, E, R, G)
    full, _, _ = oracle.combine(y, idx, w, lay, E, R, G)
    part, _, _ = oracle.combine(y, idx, w, lay, E, R, G, t0=3, t1=6)
    assert np.array_equal(part[3:6], full[3:6]) and np.all(part[:3] == 0) and np.all(part[6:] == 0)


def test_fp8_byte_factor(golden_dir):
    import json
    import os
    g = json.load(open(os.path.join(golden_dir, "fp8_byte_factor.json")))
    H = g["hidden"]
    q, s = oracle.quant_fp8_row(np.zeros(H, np.uint16))
    assert q.nbytes + s.nbytes == g["fp8_row_bytes"]
    assert (q.nbytes + s.nbytes) / (2 * H) == g["fp8_factor"]
