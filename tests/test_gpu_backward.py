"""GPU parity of the backward calls (through the C ABI) against the oracle:
combine backward (gradient rows bit-exact, weight gradients within the fp32
summation bound), dispatch backward and the rank-row gather backward
bit-exact, on the per-pair, per-rank and fixed-capacity layouts."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, bf16_f64, dev_bf16, dev_f32, dev_i32, host, host_bf16

pytestmark = pytest.mark.gpu


def _route(seed, n, k, e, masked=0.05):
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    ids[g.random((n, k)) < masked] = -1
    return ids


def _check_grad_w(got, ref, go, y, so, h):
    """|gpu - ref| <= H * 2^-24 * sum_h |g_h y_h| (+ the fp32 rounding of ref):
    the worst case of an fp32 sum of H exact products in any order."""
    gf, yf = bf16_f64(go), bf16_f64(y)
    for t in range(so.shape[0]):
        for j in range(so.shape[1]):
            s = so[t, j]
            if s < 0:
                assert got[t, j] == 0.0
                continue
            mag = np.abs(gf[t] * yf[s]).sum()
            tol = h * 2.0 ** -24 * mag + 2.0 ** -24 * abs(ref[t, j]) + 1e-30
            assert abs(float(got[t, j]) - float(ref[t, j])) <= tol, (t, j)


@pytest.mark.parametrize("n,k,e,h,with_y", [
    (512, 8, 256, 7168, True),     # prefill-sized rows
    (300, 3, 32, 520, True),       # k <= 8 path, ragged H
    (96, 12, 64, 1024, True),      # k <= 16 path
    (40, 20, 64, 256, True),       # k <= 32 path
    (200, 8, 64, 2048, False),     # no expert rows: no weight gradient
])
def test_combine_backward(n, k, e, h, with_y):
    from combine_moe_layout_03_gb300 import moe
    ids = _route(n + k, n, k, e)
    lay = oracle.layout(ids, e, 1)
    P = lay["num_pairs"]
    rows = P + 5
    g = np.random.default_rng(k)
    y = synth.bf16_normal(g, (rows, h))
    go = synth.bf16_normal(g, (n, h))
    w = (g.standard_normal((n, k)) * 0.5).astype(np.float32)
    so = lay["slot_of"]
    d = moe.MoeDesc(n, k, e, 1, h)
    gy_d = torch.zeros((rows, h), dtype=torch.bfloat16, device=DEV)
    gy_d, gw_d = moe.moe_combine_backward(d, dev_bf16(go), dev_f32(w), dev_i32(so),
                                          dev_bf16(y) if with_y else None, rows, gy_d)
    torch.cuda.synchronize()
    ref_gy, ref_gw = oracle.combine_backward(go, w, so, y if with_y else None, rows, h)
    np.testing.assert_array_equal(host_bf16(gy_d), ref_gy)
    if with_y:
        _check_grad_w(host(gw_d), ref_gw, go, y, so, h)
    else:
        assert gw_d is None


def test_combine_backward_full_prefill_sampled():
    # the prefill workload at full size; the oracle checks a seeded sample of tokens
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=31)
    ids, w = c["topk_idx"], c["topk_weights"]
    n, k, e, h = 4096, 8, 256, 7168
    lay = oracle.layout(ids, e, 8)
    P = lay["num_pairs"]
    g = np.random.default_rng(32)
    go = synth.bf16_normal(g, (n, h))
    pick = np.sort(g.choice(n, 48, replace=False))
    so_p = lay["slot_of"][pick]
    named = so_p[so_p >= 0]
    # expert rows drawn for the sampled tokens' pairs, zero elsewhere
    y_rows = synth.bf16_normal(g, (named.size, h))
    y_d = torch.zeros((P, h), dtype=torch.bfloat16, device=DEV)
    y_d[torch.from_numpy(named.astype(np.int64)).to(DEV)] = dev_bf16(y_rows)
    d = moe.MoeDesc(n, k, e, 8, h)
    so_d = dev_i32(lay["slot_of"])
    gy_d, gw_d = moe.moe_combine_backward(d, dev_bf16(go), dev_f32(w), so_d, y_d, P)
    torch.cuda.synchronize()
    # the sample's rows, renumbered densely for the oracle
    dense = np.full_like(so_p, -1)
    dense[so_p >= 0] = np.arange(named.size)
    ref_gy, ref_gw = oracle.combine_backward(go[pick], w[pick], dense, y_rows, named.size, h)
    got_gy = host_bf16(gy_d.index_select(0, torch.from_numpy(named.astype(np.int64)).to(DEV)))
    np.testing.assert_array_equal(got_gy, ref_gy)
    _check_grad_w(host(gw_d)[pick], ref_gw, go[pick], y_rows, dense, h)


def test_combine_backward_rows_bound_and_guard():
    from combine_moe_layout_03_gb300 import moe
    n, k, e, h = 64, 4, 16, 256
    ids = _route(40, n, k, e, masked=0.0)
    lay = oracle.layout(ids, e, 1)
    P = lay["num_pairs"]
    cut = P - 37
    g = np.random.default_rng(41)
    go = synth.bf16_normal(g, (n, h))
    w = g.standard_normal((n, k)).astype(np.float32)
    y = synth.bf16_normal(g, (P, h))
    buf = torch.full((P + 64, h), 7.0, dtype=torch.bfloat16, device=DEV)
    d = moe.MoeDesc(n, k, e, 1, h)
    _, gw_d = moe.moe_combine_backward(d, dev_bf16(go), dev_f32(w), dev_i32(lay["slot_of"]),
                                       dev_bf16(y[:cut]), cut, buf[:cut])
    torch.cuda.synchronize()
    assert (buf[cut:].float() == 7.0).all()
    so_cut = np.where(lay["slot_of"] < cut, lay["slot_of"], -1)
    ref_gy, ref_gw = oracle.combine_backward(go, w, so_cut, y[:cut], cut, h)
    np.testing.assert_array_equal(host_bf16(buf[:cut]), ref_gy)
    _check_grad_w(host(gw_d), ref_gw, go, y[:cut], so_cut, h)


@pytest.mark.parametrize("n,k,e,h", [(4096, 8, 256, 7168), (100, 6, 48, 520), (1, 8, 256, 64)])
def test_dispatch_backward(n, k, e, h):
    from combine_moe_layout_03_gb300 import moe
    ids = _route(50 + n, n, k, e)
    lay = oracle.layout(ids, e, 1)
    P = max(lay["num_pairs"], 1)
    gi = synth.bf16_normal(np.random.default_rng(51), (P, h))
    d = moe.MoeDesc(n, k, e, 1, h)
    gx = moe.moe_dispatch_backward(d, dev_bf16(gi), dev_i32(lay["slot_of"]))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bf16(gx), oracle.dispatch_backward(gi, lay["slot_of"], h))


def test_gather_ranks_backward():
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=60, n=1024, hidden=7168)
    ids = c["topk_idx"]
    n, k, e, r, h = 1024, 8, 256, 8, 7168
    d = moe.MoeDesc(n, k, e, r, h)
    lay = moe.moe_layout(d, dev_i32(ids))
    rl = moe.moe_rank_layout(d, lay)
    rows = n * r
    go = synth.bf16_normal(np.random.default_rng(61), (n, h))
    gr = torch.zeros((rows, h), dtype=torch.bfloat16, device=DEV)
    moe.moe_combine_gather_ranks_backward(d, dev_bf16(go), rl["send_head"], gr)
    torch.cuda.synchronize()
    ref = oracle.gather_ranks_backward(go, host(rl["send_head"]), rows, h)
    np.testing.assert_array_equal(host_bf16(gr), ref)


def test_training_step_round_trip_on_fixed_capacity_buffers():
    # forward: LL layout, BF16 dispatch into [E * cap] rows, identity expert,
    # top-k combine; backward: combine backward over ll_slot_of, then dispatch
    # backward. Each GPU stage is compared with the oracle's stage.
    from combine_moe_layout_03_gb300 import moe
    c = synth.decode_ll_case(seed=70, tokens_per_rank=16, r=4, hidden=512, e=32, k=4)
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    n, k, e, r, h, max_t = 64, 4, 32, 4, 512, 16
    d = moe.MoeDesc(n, k, e, r, h, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_BF16)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    ll = moe.moe_ll_layout(d, max_t, ids_d, lay)
    xo, _ = moe.moe_dispatch_ll(d, dev_bf16(x), None, ll["ll_slot_of"], ll["capacity"])
    y_d = xo.view(torch.bfloat16)                   # identity expert
    cd = moe.MoeDesc(n, k, e, r, h)
    out = moe.moe_combine(cd, moe.MOE_COMBINE_TOPK, y_d, ids_d, dev_f32(w), ll["ll_slot_of"])
    go = synth.bf16_normal(np.random.default_rng(71), (n, h))
    rows = e * ll["capacity"]
    gy = torch.zeros((rows, h), dtype=torch.bfloat16, device=DEV)
    gy, gw = moe.moe_combine_backward(cd, dev_bf16(go), dev_f32(w), ll["ll_slot_of"], y_d, rows, gy)
    gx = moe.moe_dispatch_backward(cd, gy, ll["ll_slot_of"])
    torch.cuda.synchronize()
    so = oracle.ll_layout(ids, e, r, max_t)["ll_slot_of"]
    y_ref, _ = oracle.dispatch_ll(x, None, so, rows, oracle.BF16, oracle.BF16, h)
    y_ref = y_ref.view(np.uint16)
    np.testing.assert_array_equal(host_bf16(out), oracle.combine_topk(y_ref, w, so, h))
    ref_gy, ref_gw = oracle.combine_backward(go, w, so, y_ref, rows, h)
    np.testing.assert_array_equal(host_bf16(gy), ref_gy)
    _check_grad_w(host(gw), ref_gw, go, y_ref, so, h)
    np.testing.assert_array_equal(host_bf16(gx), oracle.dispatch_backward(ref_gy, so, h))
