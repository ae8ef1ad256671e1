"""Shared plumbing for the GPU parity tests: moving seeded inputs to the
device, running the library's path, and comparing with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_ep_layout_05_gb300 import inputs

DEV = "cuda"


def ep():
    from combine_ep_layout_05_gb300 import build
    build.build()
    from combine_ep_layout_05_gb300 import ep as m
    return m


def bf16_dev(a_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).to(DEV).view(torch.bfloat16)


def u16_host(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_layout(m, p, idx_dev, status):
    lb = m.LayoutBuffers(p, DEV)
    lb.run(p, idx_dev, dev_status=status)
    return lb


def compare_layout(lb, lay_o):
    for key in ("is_token_in_rank", "tokens_per_rank", "tokens_per_expert", "tokens_per_node",
                "recv_tokens_per_rank", "rank_slot", "token_major_offset", "expert_slot", "node_slot"):
        got = getattr(lb, key).cpu().numpy()
        want = lay_o[key]
        assert got.shape == want.shape, key
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{key}: {bad.shape[0]} mismatches, first at {bad[0].tolist()}: " \
                              f"got {got[tuple(bad[0])]} want {want[tuple(bad[0])]}"


def row_token_map(idx, lay_o, E, R, G, layout_name):
    """Receive row -> source token (-1 for rows the layout leaves empty),
    obtained from the oracle's own dispatch of an 8-channel token-id tensor."""
    T = idx.shape[0]
    ids = np.zeros((T, 8), np.uint16)
    ids[:, 0] = np.arange(T) & 0xFFFF
    ids[:, 1] = np.arange(T) >> 16
    # (status bits for invalid ids are compared by the caller)
    recv, _, _ = oracle.dispatch(ids, idx, lay_o, E, R, G, layout_name=layout_name, poison=True)
    live = recv[:, 2] != 0xFFFF
    tok = np.where(live, recv[:, 0].astype(np.int64) | (recv[:, 1].astype(np.int64) << 16), -1)
    return tok


def check_dispatch_bf16(recv_dev, x_dev, tok):
    """Every live row bit-equals its token's row; every other row still holds
    the 0xFFFF poison."""
    live = torch.from_numpy(np.nonzero(tok >= 0)[0]).to(DEV)
    src = torch.from_numpy(tok[tok >= 0]).to(DEV)
    rv = recv_dev.view(torch.int16)
    xv = x_dev.view(torch.int16)
    for i in range(0, live.numel(), 65536):
        a = rv.index_select(0, live[i:i + 65536])
        b = xv.index_select(0, src[i:i + 65536])
        assert torch.equal(a, b), f"live rows differ near row {int(live[i])}"
    dead = torch.ones(rv.shape[0], dtype=torch.bool, device=DEV)
    dead[live] = False
    assert bool((rv[dead] == -1).all()), "a row the layout leaves empty was written"


def bf16_ulp(b: np.ndarray) -> np.ndarray:
    """Spacing of bf16 at each (finite) bf16 value, magnitude-wise."""
    mag = (b & 0x7FFF).astype(np.int64)
    up = inputs.f32_from_bf16_bits((mag + 1).astype(np.uint16)).astype(np.float64)
    here = inputs.f32_from_bf16_bits(mag.astype(np.uint16)).astype(np.float64)
    return up - here


def check_combine(out_gpu_u16, oracle_f64, oracle_bf16, abs_sum, k, rows=None, max_slack_frac=1e-3):
    """GPU combine vs the oracle (fp64 sum, rounded once to bf16).

    Per element: |gpu - fp64 sum| at most one bf16 ulp of the oracle's rounded
    value plus k * 2^-23 * sum_j |w_j y_j| (room for fp32 accumulation when
    terms cancel).  The elements that needed that room beyond the ulp are
    counted; at most `max_slack_frac` of them may.
    Overall: the relative L2 distance of the GPU output to the fp64 sum may
    exceed that of the oracle's own bf16 output (its rounding error alone,
    1.3e-3 to 1.7e-3 for N(0,1)-like values, so no bf16 output can be within
    1e-3 of the fp64 sum) by at most 1e-3.  That admits the unavoidable
    rounding to bf16 and nothing more: a dropped term or a wrong weight
    moves rel-L2 by far more than 1e-3.
    Returns (rel-L2 of the GPU output, rel-L2 of the oracle's bf16 output,
    elements that used the fp32 room)."""
    if rows is not None:
        out_gpu_u16, oracle_f64, oracle_bf16, abs_sum = (a[rows] for a in
                                                        (out_gpu_u16, oracle_f64, oracle_bf16, abs_sum))
    g = inputs.f32_from_bf16_bits(out_gpu_u16).astype(np.float64)
    err = np.abs(g - oracle_f64)
    ulp = bf16_ulp(oracle_bf16)
    tol = ulp + k * 2.0 ** -23 * abs_sum
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{bad.shape[0]} elements off, first {bad[0].tolist()}: gpu {g[tuple(bad[0])]} " \
                          f"oracle {oracle_f64[tuple(bad[0])]} tol {tol[tuple(bad[0])]}"
    slack = int(np.count_nonzero(err > ulp))
    assert slack <= max(1, max_slack_frac * err.size), \
        f"{slack} of {err.size} elements needed the fp32 accumulation room beyond one bf16 ulp"
    ob = inputs.f32_from_bf16_bits(oracle_bf16).astype(np.float64)
    den = np.linalg.norm(oracle_f64)
    rel = rel_o = 0.0
    if den > 0:
        rel = float(np.linalg.norm(g - oracle_f64) / den)
        rel_o = float(np.linalg.norm(ob - oracle_f64) / den)
        assert rel <= rel_o + 1e-3, f"relative L2 {rel} to the fp64 sum (the oracle's bf16 output: {rel_o})"
    return rel, rel_o, slack


def combine_ranges(T, R, n=128):
    """Token ranges the combine is compared on when the oracle is too slow for
    every token: the first and last n tokens and n tokens from the middle of
    each source rank's segment (all tokens when T <= 2048)."""
    if T <= 2048:
        return None
    Tr = T // R
    rs = [(0, n)]
    for s in range(R):
        mid = s * Tr + Tr // 2
        lo = max(0, min(mid - n // 2, T - n))
        rs.append((lo, lo + n))
    rs.append((T - n, T))
    out = []
    for a, b in sorted(set(rs)):
        if out and a < out[-1][1]:
            out[-1] = (out[-1][0], max(out[-1][1], b))
        else:
            out.append((a, b))
    return out


# problems with at least this many x elements compare the FP8 identity
# expert on the rows the combine check reads rather than on every live row
DEQUANT_FULL_ELEMS = 1 << 26


def combine_ranges_or_all(T, ranges):
    return ranges if ranges else [(0, T)]


def rows_of_tokens(tok, ranges):
    """Receive rows (sorted) whose token lies in one of the ranges."""
    sel = np.zeros(tok.shape[0], dtype=bool)
    for t0, t1 in ranges:
        sel |= (tok >= t0) & (tok < t1)
    return np.nonzero(sel)[0].astype(np.int64)


def dequant_rows(q, s, rows):
    """The oracle's FP8 identity expert on the listed rows only: the rows are
    gathered into a one-rank, one-segment buffer whose every row is live."""
    n = rows.size
    lay1 = {"tokens_per_rank": np.array([[n]], np.int32)}
    return oracle.dequant_fp8(np.ascontiguousarray(q[rows]), np.ascontiguousarray(s[rows]), lay1, n, 1, 1,
                              layout_name="rank_major")


def status_word():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def full_path_check(m, R, Tr, H, E, k, G, layout_name, dtype, seed=0, zipf=None, idx=None, w=None,
                    x=None, random_y=True, combine_ranges=None, fused=False, wire=None):
    """Runs layout -> rdma count -> dispatch -> (dequant) -> combine on the GPU
    and compares every output with the oracle on the same seeded inputs.
    fused: layout and dispatch through the one-launch ep_layout_dispatch.
    wire: also cast the identity experts' rows to a combine wire format
    ("mxfp8" / "nvfp4") and combine from it."""
    T = R * Tr
    if x is None:
        x = inputs.make_tokens(T, H, seed=seed)
    if idx is None:
        idx, w0 = inputs.make_routing(T, E, k, seed=seed, zipf_s=zipf)
        w = w0 if w is None else w
    p = m.problem(T, H, k, E, R, G)
    st = status_word()
    idx_d = torch.from_numpy(idx).to(DEV)
    w_d = torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV)
    x_d = bf16_dev(x)

    rows = m.ep_recv_rows(p, layout_name)
    if dtype == "bf16":
        recv = torch.full((rows, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        scales = None
    else:
        recv = torch.full((rows, H), 0xFF, dtype=torch.uint8, device=DEV)
        scales = torch.full((rows, H // 128), float("nan"), dtype=torch.float32, device=DEV)

    # layout + RDMA counts (and, fused, the dispatch)
    if fused:
        lb = m.LayoutBuffers(p, DEV)
        m.ep_layout_dispatch(p, layout_name, dtype, x_d, idx_d, lb, recv, scales, st)
    else:
        lb = run_layout(m, p, idx_d, st)
    lay_o, st_o = oracle.layout(idx, E, R, G)
    compare_layout(lb, lay_o)
    algo_d = torch.empty(R, dtype=torch.int64, device=DEV)
    phys_d = torch.empty(R, dtype=torch.int64, device=DEV)
    m.ep_rdma_token_count(p, idx_d, algo_d, phys_d, st)
    algo_o, phys_o, _ = oracle.rdma_token_count(idx, E, R, G)
    assert np.array_equal(algo_d.cpu().numpy(), algo_o)
    assert np.array_equal(phys_d.cpu().numpy(), phys_o)
    # the same counts come out of the layout
    assert np.array_equal(lb.algo_per_rank.cpu().numpy(), algo_o)
    assert np.array_equal(lb.physical_exact_per_rank.cpu().numpy(), phys_o)

    # dispatch
    tok = row_token_map(idx, lay_o, E, R, G, layout_name)
    if dtype == "bf16":
        if not fused:
            m.ep_dispatch(p, layout_name, "bf16", x_d, idx_d, lb.rank_slot, lb.expert_slot, recv, None, st)
        check_dispatch_bf16(recv, x_d, tok)
        y_d = recv
        # the oracle's own identity-expert rows (its dispatch of x)
        y_o, _, _ = oracle.dispatch(x, idx, lay_o, E, R, G, layout_name=layout_name, poison=False)
    else:
        q, s = recv, scales
        if not fused:
            m.ep_dispatch(p, layout_name, "fp8_e4m3", x_d, idx_d, lb.rank_slot, lb.expert_slot, q, s, st)
        q_o, s_o, _ = oracle.dispatch(x, idx, lay_o, E, R, G, layout_name=layout_name, dtype="fp8_e4m3",
                                      poison=True)
        q_h, s_h = q.cpu().numpy(), s.cpu().numpy()
        assert np.array_equal(q_h, q_o), f"FP8 payload differs at {np.argwhere(q_h != q_o)[:3].tolist()}"
        assert np.array_equal(s_h.view(np.uint32), s_o.view(np.uint32)), "FP8 scales differ"
        y_d = torch.zeros((rows, H), dtype=torch.bfloat16, device=DEV)
        m.ep_dequant_fp8(p, layout_name, idx_d, lb.rank_slot, lb.expert_slot, q, s, y_d)
        if T * H < DEQUANT_FULL_ELEMS:
            y_o = oracle.dequant_fp8(q_o, s_o, lay_o, T, E, R, layout_name=layout_name)
            live = tok >= 0
            assert np.array_equal(u16_host(y_d)[live], y_o[live]), "identity-expert dequant differs"
        else:
            # the oracle's dequant is slow (tens of ns per element): compare
            # the rows the combine check reads, every one of them bit-exact
            need = rows_of_tokens(tok, combine_ranges_or_all(T, combine_ranges))
            y_o = np.zeros((rows, H), np.uint16)          # pages only touched where written
            y_o[need] = dequant_rows(q_o, s_o, need)
            got = u16_host(y_d.index_select(0, torch.from_numpy(need).to(DEV)))
            assert np.array_equal(got, y_o[need]), "identity-expert dequant differs"

    # combine: identity experts (the GPU combines what its dispatch wrote,
    # the oracle what its own dispatch wrote), then random rows
    ys = [("identity", y_d, y_o)]
    if random_y:
        yr = inputs.make_random_rows(rows, H, seed=seed + 100)
        ys.append(("random", bf16_dev(yr), yr))
    if wire is not None:
        check_wire(m, p, layout_name, wire, y_d, y_o, tok, idx, idx_d, w, w_d, lay_o, lb, E, R, G, k, st,
                   combine_ranges)
    for name, yd, yh in ys:
        out = torch.full((T, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        m.ep_combine(p, layout_name, yd, idx_d, w_d, lb.rank_slot, lb.expert_slot, out, st)
        out_h = u16_host(out)
        for t0, t1 in (combine_ranges or [(0, T)]):
            ob, of, _ = oracle.combine(yh, idx, w, lay_o, E, R, G, layout_name=layout_name, t0=t0, t1=t1,
                                       want_f64=True)
            _, oa, _ = oracle.combine(yh & 0x7FFF, idx, np.abs(w), lay_o, E, R, G, layout_name=layout_name,
                                      t0=t0, t1=t1, want_f64=True)
            check_combine(out_h[t0:t1], of[t0:t1], ob[t0:t1], oa[t0:t1], k)
        if name == "identity" and dtype == "bf16":
            identity_property(out, x_d, idx_d, w_d, E)
    torch.cuda.synchronize()
    assert int(st.item()) == st_o, f"device status {int(st.item())} vs oracle {st_o}"
    return p


def identity_property(out, x_d, idx_d, w_d, E):
    """With identity experts every kept expert returns x[t], so out[t] is
    x[t] * (sum of kept weights) to within one bf16 ulp, on every token."""
    keep = (idx_d >= 0) & (idx_d < E)
    dup = torch.zeros_like(keep)
    for j in range(1, idx_d.shape[1]):
        dup[:, j] = ((idx_d[:, :j] == idx_d[:, j:j + 1]) & keep[:, :j]).any(dim=1)
    wsum = torch.where(keep & ~dup, w_d, torch.zeros_like(w_d)).sum(dim=1, dtype=torch.float64)
    ref = x_d.double() * wsum[:, None]
    refb = ref.to(torch.bfloat16)
    mag = refb.view(torch.int16).to(torch.int32) & 0x7FFF
    up = (mag + 1).to(torch.int16).view(torch.bfloat16).double()
    ulp = up - mag.to(torch.int16).view(torch.bfloat16).double()
    err = (out.double() - ref).abs()
    assert bool((err <= ulp * 1.0001).all()), f"identity property fails on {int((err > ulp).sum())} elements"




def check_wire(m, p, layout_name, fmt, y_d, y_o, tok, idx, idx_d, w, w_d, lay_o, lb, E, R, G, k, st,
               combine_ranges):
    """Wire-format cast of the live rows bit-exact against the oracle's cast
    of its own rows; the wire combine within the combine tolerance."""
    T, H = p.num_tokens, p.hidden
    qs, ss, sdt = m.wire_shapes(p, layout_name, fmt)
    wq = torch.full(qs, 0xAB, dtype=torch.uint8, device=DEV)
    ws = torch.zeros(ss, dtype=sdt, device=DEV)
    m.ep_combine_quantize(p, layout_name, fmt, y_d, idx_d, lb.rank_slot, lb.expert_slot, wq, ws)
    live = np.nonzero(tok >= 0)[0]
    q_o, s_o = oracle.quant_wire_rows(y_o, live, fmt)
    q_h = wq.cpu().numpy()
    s_h = ws.view(torch.int16).cpu().numpy().view(np.uint16) if fmt == "nvfp4" else ws.cpu().numpy()
    assert np.array_equal(q_h[live], q_o[live]), f"{fmt} codes differ"
    assert np.array_equal(s_h[live], s_o[live]), f"{fmt} scales differ"
    assert np.all(q_h[tok < 0] == 0xAB), "a row the layout leaves empty was cast"
    out = torch.full((T, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    m.ep_combine_wire(p, layout_name, fmt, wq, ws, idx_d, w_d, lb.rank_slot, lb.expert_slot, out, st)
    out_h = u16_host(out)
    s_abs = s_o.copy()
    for t0, t1 in (combine_ranges or [(0, T)]):
        ob, of, _ = oracle.combine_wire(q_o, s_o, idx, w, lay_o, E, R, G, fmt, H, layout_name=layout_name,
                                        t0=t0, t1=t1, want_f64=True)
        # sum of |w * value|: the same wire rows with the sign bits cleared
        qa = q_o & (0x7F if fmt == "mxfp8" else 0x77)
        _, oa, _ = oracle.combine_wire(qa, s_abs, idx, np.abs(w), lay_o, E, R, G, fmt, H,
                                       layout_name=layout_name, t0=t0, t1=t1, want_f64=True)
        check_combine(out_h[t0:t1], of[t0:t1], ob[t0:t1], oa[t0:t1], k)


def check_two_level_combine(out_h, cst_h, yh, yh_abs, idx, w, lay_o, E, R, G, k, ranges, stage_bufs=(None, None)):
    """The two-level combine of the tokens in `ranges` against the oracle's:
    every node partial within one bf16 ulp of the oracle's partial plus fp32
    room (k * 2^-22 * sum |w y| of the node); every output element within one
    ulp of the fp64 sum of the oracle's partials plus one ulp of each partial
    (both sides round every partial to bf16 once) plus the fp32 room each
    partial is allowed; and over each range the
    relative L2 distance to that fp64 sum within 1e-3 of the oracle's own
    bf16 output's.  yh_abs: yh with the sign bits cleared (on the rows the
    ranges read).  stage_bufs: two reusable oracle staging buffers (values,
    magnitudes), or None to let the oracle allocate them."""
    T, H = out_h.shape[0], out_h.shape[1]
    N, Tr = R // G, T // R
    ns_all = lay_o["node_slot"]
    for t0, t1 in ranges:
        ob, of, so, _ = oracle.combine_two_level(yh, idx, w, lay_o, E, R, G, t0=t0, t1=t1, want_f64=True,
                                                 stage=stage_bufs[0])
        _, _, sa, _ = oracle.combine_two_level(yh_abs, idx, np.abs(w), lay_o, E, R, G, t0=t0, t1=t1,
                                               stage=stage_bufs[1])
        t = np.arange(t0, t1)
        src = t // Tr
        ulp_sum = np.zeros((t1 - t0, H))     # what the partials may differ by: one ulp + fp32 room each
        for n in range(N):
            ns = ns_all[t0:t1, n]
            has = ns >= 0
            if not has.any():
                continue
            srow = (n * R + src[has]) * Tr + ns[has]
            po = inputs.f32_from_bf16_bits(so[srow]).astype(np.float64)
            pg = inputs.f32_from_bf16_bits(cst_h[srow]).astype(np.float64)
            pa = np.abs(inputs.f32_from_bf16_bits(sa[srow]).astype(np.float64))
            up = bf16_ulp(so[srow])
            room = up + k * 2.0 ** -22 * pa
            bad = np.argwhere(np.abs(pg - po) > room)
            assert bad.size == 0, ("partial", int(t[has][bad[0][0]]), n)
            ulp_sum[has] += room
        g = inputs.f32_from_bf16_bits(out_h[t0:t1]).astype(np.float64)
        ref = of[t0:t1]
        tol = bf16_ulp(ob[t0:t1]) + ulp_sum + 1e-30
        bad = np.argwhere(np.abs(g - ref) > tol)
        assert bad.size == 0, ("out", int(t0 + bad[0][0]), int(bad[0][1]))
        den = np.linalg.norm(ref)
        if den > 0:
            rel = np.linalg.norm(g - ref) / den
            rel_o = np.linalg.norm(inputs.f32_from_bf16_bits(ob[t0:t1]).astype(np.float64) - ref) / den
            assert rel <= rel_o + 1e-3, f"two-level relative L2 {rel} (the oracle's bf16 output: {rel_o})"


def two_level_check(m, R, G, Tr, H, E, k, seed=0, zipf=None, random_y=True, combine_ranges=None, routing=None):
    """Two-level dispatch and combine against the oracle: staging rows and
    the forwarded receive buffer bit-exact; the combine as
    check_two_level_combine states."""
    T = R * Tr
    x = inputs.make_tokens(T, H, seed=seed)
    idx, w = routing if routing is not None else inputs.make_routing(T, E, k, seed=seed, zipf_s=zipf)
    if random_y:
        w = inputs.make_uniform_weights(T, k, seed=seed)
    p = m.problem(T, H, k, E, R, G)
    st = status_word()
    idx_d, w_d, x_d = torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), bf16_dev(x)
    lb = run_layout(m, p, idx_d, st)
    lay_o, _ = oracle.layout(idx, E, R, G)
    compare_layout(lb, lay_o)
    srows, rows = m.ep_stage_rows(p), m.ep_recv_rows(p)
    stage = torch.full((srows, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    recv = torch.full((rows, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    m.ep_dispatch_two_level(p, x_d, lb.rank_slot, lb.node_slot, stage, recv, st)
    stage_o, recv_o = oracle.dispatch_two_level(x, lay_o, E, R, G, k)
    assert np.array_equal(u16_host(stage), stage_o), "staging rows differ"
    tok = row_token_map(idx, lay_o, E, R, G, "rank_major")
    check_dispatch_bf16(recv, x_d, tok)
    del stage_o
    # combine: random expert rows (or the identity rows of the oracle's dispatch)
    yh = inputs.make_random_rows(rows, H, seed=seed + 1) if random_y else recv_o
    y_d = bf16_dev(yh)
    del recv_o
    cstage = torch.full((srows, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    out = torch.full((T, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    m.ep_combine_two_level(p, y_d, idx_d, w_d, lb.rank_slot, lb.node_slot, cstage, out, st)
    check_two_level_combine(u16_host(out), u16_host(cstage), yh, yh & 0x7FFF, idx, w, lay_o, E, R, G, k,
                            combine_ranges or [(0, T)])
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def two_level_row_maps(idx, lay_o, E, R, G, k):
    """(staging row -> token, receive row -> token), -1 for rows the layout
    leaves empty, from the oracle's own two-level dispatch of an 8-channel
    token-id tensor."""
    T = idx.shape[0]
    ids = np.zeros((T, 8), np.uint16)
    ids[:, 0] = np.arange(T) & 0xFFFF
    ids[:, 1] = np.arange(T) >> 16
    st_i, rv_i = oracle.dispatch_two_level(ids, lay_o, E, R, G, k)
    maps = []
    for a in (st_i, rv_i):
        live = a[:, 2] != 0xFFFF
        maps.append(np.where(live, a[:, 0].astype(np.int64) | (a[:, 1].astype(np.int64) << 16), -1))
    return maps


def two_level_check_full_size(m, wl, ranges):
    """The two-level path at a workload's full size.  Staging rows and the
    forwarded receive buffer are compared in full on the GPU against the
    token rows the oracle's own row maps name (every live row bit-exact,
    every other row untouched).  The combine is compared on `ranges`, twice:
    identity experts with the routing's softmax weights, then random expert
    rows with unnormalised U(0,2) weights (written into the rows those
    tokens read, on both sides)."""
    R, G, Tr, H, E, k = wl.ranks, wl.gpus_per_node, wl.tokens_per_rank, wl.hidden, wl.experts, wl.topk
    T = R * Tr
    x = inputs.make_tokens(T, H, seed=wl.seed)
    idx, w = inputs.make_workload_routing(wl)
    p = m.problem(T, H, k, E, R, G)
    st = status_word()
    idx_d, x_d = torch.from_numpy(idx).to(DEV), bf16_dev(x)
    lb = run_layout(m, p, idx_d, st)
    lay_o, _ = oracle.layout(idx, E, R, G)
    compare_layout(lb, lay_o)
    srows, rows = m.ep_stage_rows(p), m.ep_recv_rows(p)
    stage = torch.full((srows, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    recv = torch.full((rows, H), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    m.ep_dispatch_two_level(p, x_d, lb.rank_slot, lb.node_slot, stage, recv, st)
    stage_tok, recv_tok = two_level_row_maps(idx, lay_o, E, R, G, k)
    assert int((stage_tok >= 0).sum()) == int(lay_o["tokens_per_node"].sum())
    check_dispatch_bf16(stage, x_d, stage_tok)
    check_dispatch_bf16(recv, x_d, recv_tok)
    del stage
    need = rows_of_tokens(recv_tok, ranges)
    need_d = torch.from_numpy(need).to(DEV)
    yh = np.zeros((rows, H), np.uint16)                     # pages only touched where written
    yh_abs = np.zeros((rows, H), np.uint16)
    # the oracle writes the staging rows of the tokens it combines only
    stage_bufs = (np.zeros((srows, H), np.uint16), np.zeros((srows, H), np.uint16))
    cstage = torch.empty((srows, H), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    w_rand = inputs.make_uniform_weights(T, k, seed=wl.seed)
    for name, wts in (("identity", w), ("random", w_rand)):
        if name == "identity":
            yh[need] = x[recv_tok[need]]                    # the oracle's identity rows
        else:
            yr = inputs.make_random_rows(need.size, H, seed=wl.seed + 1)
            yh[need] = yr
            recv.view(torch.int16).index_copy_(0, need_d, torch.from_numpy(yr.view(np.int16)).to(DEV))
        yh_abs[need] = yh[need] & 0x7FFF
        w_d = torch.from_numpy(np.ascontiguousarray(wts, np.float32)).to(DEV)
        cstage.view(torch.int16).fill_(-1)
        out.view(torch.int16).fill_(-1)
        m.ep_combine_two_level(p, recv, idx_d, w_d, lb.rank_slot, lb.node_slot, cstage, out, st)
        check_two_level_combine(u16_host(out), u16_host(cstage), yh, yh_abs, idx, wts, lay_o, E, R, G, k, ranges,
                                stage_bufs=stage_bufs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
