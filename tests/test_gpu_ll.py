"""GPU parity of the fixed-capacity, expert-major receive path (DeepEP
low-latency dispatch/combine) through the C ABI against the oracle: the
layout (positions, source info, ranges, counts) bit-exact, packed payload and
scales bit-exact, and the combine over the packed expert outputs within the
BF16 contract tolerance."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, assert_combine_close, dev_bf16, dev_f32, dev_i32, dev_u8, host, host_bf16

pytestmark = pytest.mark.gpu
LKEYS = ("ll_slot_of", "src_info", "layout_range", "recv_count")


def _gpu_ll(ids, e, r, max_t):
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, 8)
    lay = moe.moe_layout(d, dev_i32(ids))
    ll = moe.moe_ll_layout(d, max_t, dev_i32(ids), lay)
    torch.cuda.synchronize()
    return ll


def _ids(case):
    """(topk_idx, experts, ranks, max tokens per rank)"""
    if case == "decode_ll":    # 8 ranks x 128 tokens, top-8 of 256
        return synth.decode_ll_case(seed=11)["topk_idx"], 256, 8, 128
    if case == "prefill":      # group-limited routing, 8 x 512
        return synth.prefill_case(seed=12)["topk_idx"], 256, 8, 512
    if case == "skewed":       # Zipf popularity, 16 x 1024, headroom in max_t
        return synth.skewed_case(seed=13)["topk_idx"], 256, 16, 1100
    g = np.random.default_rng(14)
    if case == "overflow":     # ids drawn with repeats: experts overflow their capacity
        return g.integers(-1, 4, size=(4 * 50, 6)).astype(np.int32), 4, 4, 50
    if case == "ragged":       # masked ids, odd sizes
        return g.integers(-1, 42, size=(3 * 37, 5)).astype(np.int32), 42, 3, 41
    raise ValueError(case)


@pytest.mark.parametrize("case", ["decode_ll", "prefill", "skewed", "overflow", "ragged"])
def test_ll_layout(case):
    ids, e, r, max_t = _ids(case)
    ll = _gpu_ll(ids, e, r, max_t)
    ref = oracle.ll_layout(ids, e, r, max_t)
    for key in LKEYS:
        np.testing.assert_array_equal(host(ll[key]).reshape(ref[key].shape), ref[key], err_msg=key)
    if case == "overflow":
        assert (ref["ll_slot_of"][ids >= 0] < 0).any()  # the case really overflows


def test_ll_layout_empty_batch():
    from combine_moe_layout_03_gb300 import moe
    d = moe.MoeDesc(0, 8, 32, 4, 8)
    ids = torch.empty((0, 8), dtype=torch.int32, device=DEV)
    lay = moe.moe_layout(d, ids)
    ll = moe.moe_ll_layout(d, 16, ids, lay)
    torch.cuda.synchronize()
    assert (host(ll["src_info"]) == -1).all()
    assert (host(ll["recv_count"]) == 0).all() and (host(ll["layout_range"]) == 0).all()


def test_ll_layout_rejects_uneven_ranks():
    from combine_moe_layout_03_gb300 import moe
    ids = dev_i32(np.zeros((30, 2), np.int32))
    d = moe.MoeDesc(30, 2, 8, 4, 8)
    lay = moe.moe_layout(d, ids)
    with pytest.raises(RuntimeError):
        moe.moe_ll_layout(d, 16, ids, lay)
    d3 = moe.MoeDesc(30, 2, 9, 3, 8)
    lay3 = moe.moe_layout(d3, ids)
    with pytest.raises(RuntimeError):
        moe.moe_ll_layout(d3, 8, ids, lay3)


def _dispatch_case(out_kind, n, hidden, seed):
    if out_kind == oracle.RAW:
        c = synth.decode_case(seed=seed, n=n, payload_bytes=hidden, scale_bytes=hidden // 8)
        return c, c["payload"], c["scales"], oracle.RAW, hidden, hidden // 8
    if n == 1024 and hidden == 7168:
        c = synth.decode_ll_case(seed=seed)
    else:
        c = synth.prefill_case(seed=seed, n=n, hidden=hidden)
    return c, c["hidden_bf16"], None, oracle.BF16, 0, 0


@pytest.mark.parametrize("out_kind,n,hidden,r,max_t", [
    (oracle.FP8_E4M3_B128, 1024, 7168, 8, 128),   # the decode workload's shape
    (oracle.FP8_E4M3_B128, 96, 1536, 4, 30),
    (oracle.BF16, 64, 1024, 8, 8),
    (oracle.NVFP4_B16, 120, 2048, 8, 16),
    (oracle.RAW, 64, 3584, 8, 8),
])
def test_dispatch_ll(out_kind, n, hidden, r, max_t):
    from combine_moe_layout_03_gb300 import moe
    c, x, sc, in_kind, pbr, sbr = _dispatch_case(out_kind, n, hidden, seed=21)
    ids = c["topk_idx"]
    e, k = 256, 8
    hs = hidden if out_kind != oracle.RAW else 2 * hidden
    d = moe.MoeDesc(n, k, e, r, hs, in_kind=in_kind, out_kind=out_kind,
                    raw_payload_bytes=pbr, raw_scale_bytes=sbr)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    ll = moe.moe_ll_layout(d, max_t, ids_d, lay)
    x_d = dev_u8(x) if out_kind == oracle.RAW else dev_bf16(x)
    sc_d = dev_u8(sc) if sc is not None else None
    xo, so = moe.moe_dispatch_ll(d, x_d, sc_d, ll["ll_slot_of"], ll["capacity"])
    torch.cuda.synchronize()
    ll_h = oracle.ll_layout(ids, e, r, max_t)
    np.testing.assert_array_equal(host(ll["ll_slot_of"]), ll_h["ll_slot_of"])
    # compare the rows the pairs fill (at the full size, those of a seeded
    # sample of tokens, which the oracle packs one by one); the others are
    # not written
    so_h = ll_h["ll_slot_of"]
    if n > 256:
        pick = np.sort(np.random.default_rng(23).choice(n, 96, replace=False))
        x, so_h = x[pick], so_h[pick]
        sc = sc[pick] if sc is not None else None
    pos = so_h[so_h >= 0]
    rows = e * ll["capacity"]
    ref_x, ref_s = oracle.dispatch_ll(x, sc, so_h, rows, in_kind, out_kind, hs, pbr, sbr)
    idx = torch.from_numpy(pos.astype(np.int64)).to(DEV)
    np.testing.assert_array_equal(host(xo.index_select(0, idx)), ref_x[pos])
    if ref_s.shape[1]:
        np.testing.assert_array_equal(host(so.index_select(0, idx)), ref_s[pos])


def test_dispatch_ll_skips_rows_past_the_buffer():
    # a scale buffer one expert short: pairs of the last expert are dropped,
    # nothing is written past either buffer
    from combine_moe_layout_03_gb300 import moe
    n, hidden, e, r, max_t = 64, 1024, 16, 4, 16
    c = synth.prefill_case(seed=22, n=n, hidden=hidden, e=e, k=4, r=r, groups=4, topk_groups=2)
    ids = c["topk_idx"]
    d = moe.MoeDesc(n, 4, e, r, hidden, in_kind=oracle.BF16, out_kind=oracle.FP8_E4M3_B128)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    ll = moe.moe_ll_layout(d, max_t, ids_d, lay)
    cap = ll["capacity"]
    rows = e * cap
    guard = 4096
    xo = torch.full((rows + guard, hidden), 0x5A, dtype=torch.uint8, device=DEV)
    so = torch.full(((rows - cap) * 32 + guard,), 0x5A, dtype=torch.uint8, device=DEV)
    moe.moe_dispatch_ll(d, dev_bf16(c["hidden_bf16"]), None, ll["ll_slot_of"], cap,
                        x_out=xo[:rows], scales_out=so[: (rows - cap) * 32].view(rows - cap, 32))
    torch.cuda.synchronize()
    assert (host(xo[rows:]) == 0x5A).all() and (host(so[(rows - cap) * 32:]) == 0x5A).all()
    ll_h = oracle.ll_layout(ids, e, r, max_t)
    ref_x, ref_s = oracle.dispatch_ll(c["hidden_bf16"], None, ll_h["ll_slot_of"], rows, oracle.BF16,
                                      oracle.FP8_E4M3_B128, hidden)
    pos = ll_h["ll_slot_of"][ll_h["ll_slot_of"] >= 0]
    kept = pos[pos < rows - cap]
    dropped = pos[pos >= rows - cap]
    assert kept.size and dropped.size
    np.testing.assert_array_equal(host(xo[:rows])[kept], ref_x[kept])
    assert (host(xo[:rows])[dropped] == 0x5A).all()


@pytest.mark.parametrize("case,hidden", [("decode_ll", 7168), ("overflow", 256), ("ragged", 520)])
def test_ll_combine(case, hidden):
    from combine_moe_layout_03_gb300 import moe
    ids, e, r, max_t = _ids(case)
    n, k = ids.shape
    if case == "decode_ll":
        w = synth.decode_ll_case(seed=11)["topk_weights"]
    else:
        w = np.random.default_rng(15).standard_normal((n, k)).astype(np.float32)
    ll_h = oracle.ll_layout(ids, e, r, max_t)
    cap = r * max_t
    rows = e * cap
    # expert outputs only where a pair lands; the rest of the buffer is zero.
    # The oracle reads the same rows through a compacted copy.
    g = np.random.default_rng(16)
    so_h = ll_h["ll_slot_of"]
    used = np.unique(so_h[so_h >= 0])
    y_used = synth.bf16_normal(g, (used.size, hidden))
    y_d = torch.zeros((rows, hidden), dtype=torch.bfloat16, device=DEV)
    y_d[torch.from_numpy(used.astype(np.int64)).to(DEV)] = dev_bf16(y_used)
    compact = np.where(so_h >= 0, np.searchsorted(used, so_h), -1).astype(np.int32)
    d = moe.MoeDesc(n, k, e, r, hidden)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    ll = moe.moe_ll_layout(d, max_t, ids_d, lay)
    out = moe.moe_combine(d, moe.MOE_COMBINE_TOPK, y_d, ids_d, dev_f32(w), ll["ll_slot_of"])
    torch.cuda.synchronize()
    ref = oracle.combine_topk(y_used, w, compact, hidden)
    assert_combine_close(host_bf16(out), ref, case)


@pytest.mark.parametrize("out_kind,n,hidden,r,max_t", [
    (oracle.FP8_E4M3_B128, 1216, 512, 8, 160),
    (oracle.NVFP4_B16, 704, 1024, 4, 200),
    (oracle.FP8_E4M3_UE8M0, 1000, 256, 8, 125),
])
def test_dispatch_ll_persistent_every_token(out_kind, n, hidden, r, max_t):
    """Every token of a larger routing in each quantising format (the full-size
    case above samples tokens): every used row equals the oracle's, unused
    rows are untouched, with padding pairs in the routing."""
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=n, n=n, hidden=hidden)
    ids = c["topk_idx"].copy()
    ids[::13, 5] = -1  # padding pairs
    e, k = 256, 8
    d = moe.MoeDesc(n, k, e, r, hidden, in_kind=oracle.BF16, out_kind=out_kind)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    ll = moe.moe_ll_layout(d, max_t, ids_d, lay)
    cap = ll["capacity"]
    rows = e * cap
    lay_rec = moe.moe_record_layout(d)
    pb, sbp = lay_rec["payload_bytes"], (lay_rec["scale_bytes"] + 15) // 16 * 16
    xo = torch.full((rows, pb), 0x5A, dtype=torch.uint8, device=DEV)
    so = torch.full((rows, sbp), 0x5A, dtype=torch.uint8, device=DEV)
    moe.moe_dispatch_ll(d, dev_bf16(c["hidden_bf16"]), None, ll["ll_slot_of"], cap, x_out=xo, scales_out=so)
    torch.cuda.synchronize()
    ll_h = oracle.ll_layout(ids, e, r, max_t)
    np.testing.assert_array_equal(host(ll["ll_slot_of"]), ll_h["ll_slot_of"])
    ref_x, ref_s = oracle.dispatch_ll(c["hidden_bf16"], None, ll_h["ll_slot_of"], rows, oracle.BF16,
                                      out_kind, hidden)
    so_h = ll_h["ll_slot_of"]
    used = np.zeros(rows, bool)
    used[so_h[so_h >= 0]] = True
    gx, gs = host(xo), host(so)
    np.testing.assert_array_equal(gx[used], ref_x[used])
    np.testing.assert_array_equal(gs[used], ref_s[used])
    assert (gx[~used] == 0x5A).all() and (gs[~used] == 0x5A).all()
