"""GPU parity at the limits the C ABI declares (include/moe.h): hidden 16384
(the largest dispatch row) in every payload format, top-32, 1024 experts on
64 ranks, 64 KiB raw payloads and scales; the combine, its backward and the
fixed-capacity path at those shapes. Records and gradient rows bit-exact,
combines within the contract tolerance."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import (DEV, assert_combine_close, bf16_f64, dev_bf16, dev_f32, dev_i32, dev_u8,
                         host, host_bf16)

pytestmark = pytest.mark.gpu

MAX_H, MAX_K, MAX_E, MAX_R, MAX_RAW = 16384, 32, 1024, 64, 65536


def _route(seed, n, k, e):
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    ids[g.random((n, k)) < 0.05] = -1
    w = g.standard_normal((n, k)).astype(np.float32)
    return ids, w


def _dispatch(ids, w, e, r, h, in_kind, out_kind, x_dev, sc_dev=None, rp=0, rs=0):
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, h, in_kind, out_kind, rp, rs)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    rb = moe.moe_record_layout(d)["record_bytes"]
    rec = torch.full((n * k + 3, rb), 0xAB, dtype=torch.uint8, device=DEV)
    moe.moe_dispatch(d, ids_d, dev_f32(w), x_dev, sc_dev, lay["slot_of"], rec)
    torch.cuda.synchronize()
    return host(rec)


@pytest.mark.parametrize("out_kind", [oracle.BF16, oracle.FP8_E4M3_B128, oracle.NVFP4_B16,
                                      oracle.FP8_E4M3_UE8M0])
def test_dispatch_largest_row_top32_1024_experts_64_ranks(out_kind):
    n = 24
    ids, w = _route(1 + out_kind, n, MAX_K, MAX_E)
    x = synth.bf16_normal(np.random.default_rng(2), (n, MAX_H))
    got = _dispatch(ids, w, MAX_E, MAX_R, MAX_H, oracle.BF16, out_kind, dev_bf16(x))
    lay = oracle.layout(ids, MAX_E, MAX_R)
    P = lay["num_pairs"]
    ref = oracle.dispatch(ids, w, x, None, lay["slot_of"], P, oracle.BF16, out_kind, MAX_H)
    np.testing.assert_array_equal(got[:P], ref)
    assert np.all(got[P:] == 0xAB)


def test_dispatch_largest_raw_payload_and_scales():
    n, k, e, r = 12, MAX_K, 256, 8
    ids, w = _route(3, n, k, e)
    g = np.random.default_rng(4)
    pay = g.integers(0, 256, size=(n, MAX_RAW), dtype=np.uint8)
    sc = g.integers(0, 256, size=(n, MAX_RAW), dtype=np.uint8)
    got = _dispatch(ids, w, e, r, 7168, oracle.RAW, oracle.RAW, dev_u8(pay), dev_u8(sc),
                    MAX_RAW, MAX_RAW)
    lay = oracle.layout(ids, e, r)
    P = lay["num_pairs"]
    ref = oracle.dispatch(ids, w, pay, sc, lay["slot_of"], P, oracle.RAW, oracle.RAW, 7168,
                          MAX_RAW, MAX_RAW)
    np.testing.assert_array_equal(got[:P], ref)


@pytest.mark.parametrize("mode", [0, 2])
def test_combine_top32_1024_experts_64_ranks_largest_row(mode):
    from combine_moe_layout_03_gb300 import moe
    n = 128
    ids, w = _route(5, n, MAX_K, MAX_E)
    lay = oracle.layout(ids, MAX_E, MAX_R)
    P = lay["num_pairs"]
    y = synth.bf16_normal(np.random.default_rng(6), (P, MAX_H))
    d = moe.MoeDesc(n, MAX_K, MAX_E, MAX_R, MAX_H)
    out = moe.moe_combine(d, mode, dev_bf16(y), dev_i32(ids), dev_f32(w), dev_i32(lay["slot_of"]))
    torch.cuda.synchronize()
    if mode == 0:
        ref = oracle.combine_topk(y, w, lay["slot_of"], MAX_H)
    else:
        ref = oracle.combine_topk_ranks(y, ids, w, lay["slot_of"], MAX_E, MAX_R, MAX_H)
    np.testing.assert_array_equal(host_bf16(out), ref)
    assert_combine_close(host_bf16(out), ref, f"mode {mode}")


def test_combine_backward_top32_largest_row():
    from combine_moe_layout_03_gb300 import moe
    n = 48
    ids, w = _route(7, n, MAX_K, MAX_E)
    lay = oracle.layout(ids, MAX_E, MAX_R)
    P = lay["num_pairs"]
    g = np.random.default_rng(8)
    y = synth.bf16_normal(g, (P, MAX_H))
    go = synth.bf16_normal(g, (n, MAX_H))
    d = moe.MoeDesc(n, MAX_K, MAX_E, MAX_R, MAX_H)
    so = lay["slot_of"]
    gy, gw = moe.moe_combine_backward(d, dev_bf16(go), dev_f32(w), dev_i32(so), dev_bf16(y), P)
    gx = moe.moe_dispatch_backward(d, gy, dev_i32(so))
    torch.cuda.synchronize()
    ref_gy, ref_gw = oracle.combine_backward(go, w, so, y, P, MAX_H)
    np.testing.assert_array_equal(host_bf16(gy), ref_gy)
    gf, yf = bf16_f64(go), bf16_f64(y)
    got_gw = host(gw)
    for t in range(n):
        for j in range(MAX_K):
            s = so[t, j]
            if s < 0:
                assert got_gw[t, j] == 0.0
                continue
            tol = MAX_H * 2.0 ** -24 * np.abs(gf[t] * yf[s]).sum() + 2.0 ** -24 * abs(ref_gw[t, j])
            assert abs(float(got_gw[t, j]) - float(ref_gw[t, j])) <= tol
    np.testing.assert_array_equal(host_bf16(gx), oracle.dispatch_backward(ref_gy, so, MAX_H))


def test_fixed_capacity_path_at_1024_experts_64_ranks():
    from combine_moe_layout_03_gb300 import moe
    r, t_per, k, e, h = MAX_R, 4, MAX_K, MAX_E, 2048
    n = r * t_per
    ids, w = _route(9, n, k, e)
    d = moe.MoeDesc(n, k, e, r, h, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    ll = moe.moe_ll_layout(d, t_per, ids_d, lay)
    x = synth.bf16_normal(np.random.default_rng(10), (n, h))
    xo, so = moe.moe_dispatch_ll(d, dev_bf16(x), None, ll["ll_slot_of"], ll["capacity"])
    torch.cuda.synchronize()
    ref = oracle.ll_layout(ids, e, r, t_per)
    for key in ("ll_slot_of", "src_info", "layout_range", "recv_count"):
        np.testing.assert_array_equal(host(ll[key]).reshape(ref[key].shape), ref[key], err_msg=key)
    pos = ref["ll_slot_of"][ref["ll_slot_of"] >= 0]
    rows = e * ll["capacity"]
    ref_x, ref_s = oracle.dispatch_ll(x, None, ref["ll_slot_of"], rows, oracle.BF16,
                                      oracle.FP8_E4M3_B128, h)
    idx = torch.from_numpy(pos.astype(np.int64)).to(DEV)
    np.testing.assert_array_equal(host(xo.index_select(0, idx)), ref_x[pos])
    np.testing.assert_array_equal(host(so.index_select(0, idx)), ref_s[pos])
