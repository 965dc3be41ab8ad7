"""Seeded random shapes through the variant paths on the GPU, checked against
the oracle:
  - one record per (token, rank): receive layout with a drawn expert
    alignment, records and the rank-row combine, bit for bit;
  - fixed-capacity expert-major buffers: positions (including capacity
    overflow), packed payload and scale rows bit for bit, and the top-k
    combine over those positions;
  - backward: gradient rows of the combine and of the dispatch bit for bit;
  - combine + residual + RMSNorm in its three modes: the new residual bit for
    bit, the normed row at most one BF16 step apart (the sum of squares and
    the reciprocal square root round differently from the oracle's fp64 mean).
Each family draws its own cases, so shapes no hand-written case names are
reached: odd k, experts per rank that are not powers of two, more than 32
ranks, ragged hidden sizes."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, assert_combine_close, dev_bf16, dev_f32, dev_i32, dev_u8, host, host_bf16

pytestmark = pytest.mark.gpu

KINDS = {"bf16": oracle.BF16, "fp8": oracle.FP8_E4M3_B128, "ue8m0": oracle.FP8_E4M3_UE8M0,
         "nvfp4": oracle.NVFP4_B16, "raw": oracle.RAW}


def _shape(g, max_cells=6_000_000):
    """Ranks, experts, top-k, tokens and a hidden size for a combine row."""
    r = int(g.choice([1, 2, 3, 4, 6, 8, 16, 33, 64]))
    e = r * int(g.integers(1, max(2, 512 // r) + 1))
    k = int(g.integers(1, 11))
    n = int(g.choice([1, 3, 32, 33, 100, 256, 257, 1000, 2048]))
    h = 8 * int(g.integers(1, 130))
    while n * k * h > max_cells and n > 1:
        n //= 2
    return r, e, k, n, h


def _ids(g, n, k, e):
    distinct = k <= e and g.random() < 0.7
    ids = np.empty((n, k), np.int32)
    for t in range(n):
        ids[t] = g.choice(e, size=k, replace=not distinct)
    pad = float(g.choice([0.0, 0.05, 0.3]))
    if pad > 0:
        ids[g.random((n, k)) < pad] = -1
    return ids


def _payload(g, kind, n):
    """(in kind, out kind, hidden, raw payload bytes, raw scale bytes, host rows,
    host scales, device rows, device scales) for a drawn payload format."""
    if kind == "raw":
        rp, rs = 16 * int(g.integers(1, 100)), 16 * int(g.integers(0, 6))
        x = g.integers(0, 256, size=(n, rp), dtype=np.uint8)
        sc = g.integers(0, 256, size=(n, rs), dtype=np.uint8) if rs else None
        return oracle.RAW, oracle.RAW, 2 * rp, rp, rs, x, sc, dev_u8(x), (dev_u8(sc) if rs else None)
    h = {"bf16": 8 * int(g.integers(1, 130)), "nvfp4": 16 * int(g.integers(1, 70))}.get(
        kind, 128 * int(g.integers(1, 9)))
    x = synth.bf16_normal(g, (n, h))
    return oracle.BF16, KINDS[kind], h, 0, 0, x, None, dev_bf16(x), None


@pytest.mark.parametrize("i", range(32))
def test_rank_path(i):
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(8100 + i)
    r, e, k, n, _ = _shape(g)
    ids = _ids(g, n, k, e)
    w = g.standard_normal((n, k)).astype(np.float32)
    align = int(g.choice([1, 2, 8, 16, 128]))
    ikind, okind, h, rp, rs, x, sc, x_d, sc_d = _payload(g, str(g.choice(list(KINDS))), n)

    ol = oracle.layout(ids, e, r)
    orl = oracle.rank_layout(ol["is_token_in_rank"], ol["tokens_per_expert"], align)
    d = moe.MoeDesc(n, k, e, r, h, ikind, okind, rp, rs)
    ids_d, w_d = dev_i32(ids), dev_f32(w)
    lay = moe.moe_layout(d, ids_d)
    rl = moe.moe_rank_layout(d, lay, align)
    torch.cuda.synchronize()
    for key in ("send_head", "recv_src_idx", "recv_offset", "recv_tokens_per_expert"):
        np.testing.assert_array_equal(host(rl[key]).reshape(orl[key].shape), orl[key],
                                      err_msg=f"case {i}: {key}")

    P = int(orl["recv_offset"][-1])
    rb = moe.moe_record_layout(d)["record_bytes"]
    rec = torch.full((n * r, rb), 0xAB, dtype=torch.uint8, device=DEV)
    moe.moe_dispatch_ranks(d, ids_d, w_d, x_d, sc_d, rl["send_head"], rec)
    torch.cuda.synchronize()
    got = host(rec)
    want = oracle.dispatch_ranks(ids, w, x, sc, orl["send_head"], P, e, ikind, okind, h, rp, rs)
    np.testing.assert_array_equal(got[:P], want, err_msg=f"case {i}: rank records")
    assert np.all(got[P:] == 0xAB), f"case {i}: bytes past the rank records were written"

    hc = 8 * int(g.integers(1, 130))
    y = synth.bf16_normal(g, (max(P, 1), hc))
    dc = moe.MoeDesc(n, k, e, r, hc)
    out = moe.moe_combine_gather_ranks(dc, dev_bf16(y), rl["send_head"])
    torch.cuda.synchronize()
    ref = oracle.combine_gather_ranks(y, orl["send_head"], hc)
    got_c = host_bf16(out)
    assert_combine_close(got_c, ref, f"case {i}: gather ranks")
    np.testing.assert_array_equal(got_c, ref, err_msg=f"case {i}: gather ranks")


@pytest.mark.parametrize("i", range(32))
def test_fixed_capacity_path(i):
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(8200 + i)
    r, e, k, _, _ = _shape(g)
    e = r * int(g.integers(1, max(2, 256 // r) + 1))
    # the buffers have E * R * max_t rows: keep them to 200k rows
    lim = max(1, 200_000 // (e * r))
    tpr = min(int(g.integers(1, 300)), lim)  # tokens per source rank
    n = r * tpr
    sel = g.random()
    if sel < 0.2:
        # capacity exactly N/R, ids crowded onto a few experts: experts overflow
        max_t = tpr
        ids = g.integers(-1, min(e, 3), size=(n, k)).astype(np.int32)
    elif sel < 0.3 and tpr > 1:
        max_t = tpr - 1  # fewer positions than a source rank's tokens: rejected
        ids = _ids(g, n, k, e)
    else:
        max_t = min(tpr + int(g.integers(0, 65)), max(lim, tpr))
        ids = _ids(g, n, k, e)
    w = g.standard_normal((n, k)).astype(np.float32)
    ikind, okind, h, rp, rs, x, sc, x_d, sc_d = _payload(g, str(g.choice(list(KINDS))), n)

    d = moe.MoeDesc(n, k, e, r, h, ikind, okind, rp, rs)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    if n > max_t * r:
        with pytest.raises(RuntimeError):
            moe.moe_ll_layout(d, max_t, ids_d, lay)
        return
    ll = moe.moe_ll_layout(d, max_t, ids_d, lay)
    torch.cuda.synchronize()
    ref = oracle.ll_layout(ids, e, r, max_t)
    for key in ("ll_slot_of", "src_info", "layout_range", "recv_count"):
        np.testing.assert_array_equal(host(ll[key]).reshape(ref[key].shape), ref[key],
                                      err_msg=f"case {i}: {key}")

    cap = ll["capacity"]
    rows = e * cap
    if moe.moe_record_layout(d)["payload_bytes"] % 16:
        # payload rows must be whole 16-byte vectors (NVFP4 with H % 32 != 0)
        with pytest.raises(RuntimeError):
            moe.moe_dispatch_ll(d, x_d, sc_d, ll["ll_slot_of"], cap)
        return
    xo, so = moe.moe_dispatch_ll(d, x_d, sc_d, ll["ll_slot_of"], cap)
    torch.cuda.synchronize()
    so_h = ref["ll_slot_of"]
    pos = so_h[so_h >= 0]
    ref_x, ref_s = oracle.dispatch_ll(x, sc, so_h, rows, ikind, okind, h, rp, rs)
    if pos.size:
        idx = torch.from_numpy(pos.astype(np.int64)).to(DEV)
        np.testing.assert_array_equal(host(xo.index_select(0, idx)), ref_x[pos],
                                      err_msg=f"case {i}: payload rows")
        if ref_s.shape[1]:
            np.testing.assert_array_equal(host(so.index_select(0, idx)), ref_s[pos],
                                          err_msg=f"case {i}: scale rows")

    # top-k combine over the fixed-capacity positions (rows no pair uses are zero)
    hc = 8 * int(g.integers(1, 130))
    used = np.unique(pos)
    y_used = synth.bf16_normal(g, (max(used.size, 1), hc))
    y_d = torch.zeros((rows, hc), dtype=torch.bfloat16, device=DEV)
    if used.size:
        y_d[torch.from_numpy(used.astype(np.int64)).to(DEV)] = dev_bf16(y_used[: used.size])
    compact = np.where(so_h >= 0, np.searchsorted(used, so_h), -1).astype(np.int32)
    dc = moe.MoeDesc(n, k, e, r, hc)
    out = moe.moe_combine(dc, moe.MOE_COMBINE_TOPK, y_d, ids_d, dev_f32(w), ll["ll_slot_of"])
    torch.cuda.synchronize()
    assert_combine_close(host_bf16(out), oracle.combine_topk(y_used, w, compact, hc),
                         f"case {i}: combine over positions")


@pytest.mark.parametrize("i", range(24))
def test_backward(i):
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(8300 + i)
    r, e, k, n, h = _shape(g)
    ids = _ids(g, n, k, e)
    w = g.standard_normal((n, k)).astype(np.float32)
    lay = oracle.layout(ids, e, r)
    so = lay["slot_of"]
    P = lay["num_pairs"]
    rows = P + int(g.integers(0, 4))
    go = synth.bf16_normal(g, (n, h))
    d = moe.MoeDesc(n, k, e, r, h)
    gy_d = torch.zeros((max(rows, 1), h), dtype=torch.bfloat16, device=DEV)
    gy_d, gw_d = moe.moe_combine_backward(d, dev_bf16(go), dev_f32(w), dev_i32(so), None,
                                          max(rows, 1), gy_d)
    torch.cuda.synchronize()
    ref_gy, _ = oracle.combine_backward(go, w, so, None, max(rows, 1), h)
    np.testing.assert_array_equal(host_bf16(gy_d), ref_gy, err_msg=f"case {i}: gradient rows")
    assert gw_d is None

    gi = synth.bf16_normal(g, (max(P, 1), h))
    gx = moe.moe_dispatch_backward(d, dev_bf16(gi), dev_i32(so))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bf16(gx), oracle.dispatch_backward(gi, so, h),
                                  err_msg=f"case {i}: dispatch backward")


@pytest.mark.parametrize("i", range(24))
def test_combine_norm(i):
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(8400 + i)
    r, e, k, n, h = _shape(g, max_cells=3_000_000)
    mode = int(g.choice([moe.MOE_COMBINE_TOPK, moe.MOE_COMBINE_RANKS, moe.MOE_COMBINE_TOPK_RANKS]))
    if mode != moe.MOE_COMBINE_TOPK:
        n = max(r, n - n % r)  # whole ranks of tokens
    res = synth.bf16_normal(g, (n, h))
    gamma = synth.bf16_normal(g, (h,))
    eps = float(g.choice([1e-6, 1e-5]))
    d = moe.MoeDesc(n, k, e, r, h)
    if mode == moe.MOE_COMBINE_RANKS:
        y = synth.bf16_normal(g, (r, n, h))
        normed, rout = moe.moe_combine_norm(d, mode, dev_bf16(y), None, None, None, dev_bf16(res),
                                            dev_bf16(gamma), eps)
        rn, rr = oracle.combine_norm(1, y, None, None, None, res, gamma, eps, e, r, h)
    else:
        ids = _ids(g, n, k, e)
        w = g.standard_normal((n, k)).astype(np.float32)
        lay = oracle.layout(ids, e, r)
        y = synth.bf16_normal(g, (max(lay["num_pairs"], 1), h))
        ids_d = dev_i32(ids)
        so_d = moe.moe_layout(d, ids_d)["slot_of"]
        normed, rout = moe.moe_combine_norm(d, mode, dev_bf16(y), ids_d, dev_f32(w), so_d,
                                            dev_bf16(res), dev_bf16(gamma), eps)
        rn, rr = oracle.combine_norm(mode, y, ids, w, lay["slot_of"], res, gamma, eps, e, r, h)
    torch.cuda.synchronize()
    gn, gr = host_bf16(normed), host_bf16(rout)
    np.testing.assert_array_equal(gr, rr, err_msg=f"case {i}: new residual (mode {mode})")
    assert_combine_close(gn, rn, f"case {i}: normed (mode {mode})")
    assert _steps(gn, rn).max() <= 1, f"case {i}: normed more than one BF16 step apart (mode {mode})"


def _steps(a, b):
    """BF16 steps between bit patterns on an ordered scale (+0 and -0 are 0 apart)."""
    def ordered(u):
        v = u.astype(np.int32)
        return np.where(v & 0x8000, -(v & 0x7FFF), v)
    return np.abs(ordered(a) - ordered(b))
