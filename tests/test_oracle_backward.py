"""Pins of the oracle's backward routines against torch autograd (float64)
and the adjoint identity with the pinned forward routines:
<combine(y), g> = <y, combine_backward(g)>, <dispatch(x), G> =
<x, dispatch_backward(G)> and <gather(recv), g> = <recv, gather_backward(g)>,
exact on small-integer inputs with dyadic weights."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth


def _bf16(f):
    return torch.from_numpy(np.asarray(f, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f64(b):
    return oracle.bf16_to_f32_array(b).astype(np.float64)


def _route(seed, n, k, e, masked=0.1):
    g = np.random.default_rng(seed)
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    ids[g.random((n, k)) < masked] = -1
    return ids


@pytest.mark.parametrize("seed,n,k,e,h", [(1, 40, 8, 64, 256), (2, 17, 3, 16, 72), (3, 64, 8, 256, 1024)])
def test_combine_backward_matches_autograd(seed, n, k, e, h):
    ids = _route(seed, n, k, e)
    lay = oracle.layout(ids, e, 1)
    rows = max(lay["num_pairs"], 1) + 3  # a few rows no pair names
    g = np.random.default_rng(seed + 10)
    y = synth.bf16_normal(g, (rows, h))
    w = (g.standard_normal((n, k)) * 0.7).astype(np.float32)
    go = synth.bf16_normal(g, (n, h))
    so = lay["slot_of"]
    gy, gw = oracle.combine_backward(go, w, so, y, rows, h)
    # autograd of out[t] = sum over valid j of w[t,j] * y[slot_of[t,j]]
    yt = torch.tensor(_f64(y), requires_grad=True)
    wt = torch.tensor(w.astype(np.float64), requires_grad=True)
    valid = torch.from_numpy(so >= 0)
    idx = torch.from_numpy(np.where(so >= 0, so, 0).astype(np.int64))
    gathered = yt[idx]                                       # [n, k, h]
    out = (wt.unsqueeze(-1) * gathered * valid.unsqueeze(-1)).sum(1)
    out.backward(torch.tensor(_f64(go)))
    # grad_y: the exact product rounded to fp32, then to BF16 (bit-exact)
    ref_gy = yt.grad.float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(gy, ref_gy)
    # grad_w: the fp64 dot rounded once to fp32 (within one fp32 ulp of torch's own fp64 sum)
    ref_gw = wt.grad.numpy()
    np.testing.assert_allclose(gw, ref_gw, rtol=2 ** -23, atol=1e-30)
    assert np.all(gw[so < 0] == 0)


def test_combine_backward_adjoint_is_exact():
    g = np.random.default_rng(4)
    n, k, e, h = 24, 4, 32, 40
    ids = _route(5, n, k, e)
    lay = oracle.layout(ids, e, 4)
    P = lay["num_pairs"]
    y = _bf16(g.integers(-8, 9, size=(P, h)))
    go = _bf16(g.integers(-8, 9, size=(n, h)))
    w = g.choice([0.25, 0.5, -1.0, 2.0], size=(n, k)).astype(np.float32)
    out = oracle.combine_topk(y, w, lay["slot_of"], h)
    gy, gw = oracle.combine_backward(go, w, lay["slot_of"], y, P, h)
    lhs = (_f64(out) * _f64(go)).sum()
    rhs = (_f64(y) * _f64(gy)).sum()
    assert lhs == rhs
    # with these inputs every dot product is an exact small number
    for t in range(n):
        for j in range(k):
            s = lay["slot_of"][t, j]
            want = 0.0 if s < 0 else float((_f64(go[t]) * _f64(y[s])).sum())
            assert gw[t, j] == want


def test_combine_backward_without_expert_out_and_rows_bound():
    ids = _route(6, 10, 4, 16, masked=0.0)
    lay = oracle.layout(ids, 16, 1)
    P = lay["num_pairs"]
    go = synth.bf16_normal(np.random.default_rng(7), (10, 16))
    w = np.ones((10, 4), np.float32)
    full, _ = oracle.combine_backward(go, w, lay["slot_of"], None, P, 16)
    # rows past `rows` are skipped; the rows kept are unchanged
    cut = P // 2
    part, none = oracle.combine_backward(go, w, lay["slot_of"], None, cut, 16)
    assert none is None
    np.testing.assert_array_equal(part, full[:cut])
    # unit weights: every named row is the token's gradient row itself
    src = lay["src_of_slot"][:P] // 4
    np.testing.assert_array_equal(full, go[src])


def test_dispatch_backward_matches_autograd_and_adjoint():
    g = np.random.default_rng(8)
    n, k, e, h = 30, 6, 48, 64
    ids = _route(9, n, k, e)
    lay = oracle.layout(ids, e, 4)
    P = lay["num_pairs"]
    # adjoint with the BF16 dispatch on integers: <payload rows, G> = <x, dispatch_backward(G)>
    x = _bf16(g.integers(-6, 7, size=(n, h)))
    w = np.ones((n, k), np.float32)
    rec = oracle.dispatch(ids, w, x, None, lay["slot_of"], P, oracle.BF16, oracle.BF16, h)
    rl = oracle.record_layout(k, h, oracle.BF16, oracle.BF16)
    rows = rec[:, rl["off_payload"]:rl["off_payload"] + 2 * h].copy().view(np.uint16)
    G = _bf16(g.integers(-6, 7, size=(P, h)))
    gx = oracle.dispatch_backward(G, lay["slot_of"], h)
    assert (_f64(rows) * _f64(G)).sum() == (_f64(x) * _f64(gx)).sum()
    # autograd of the copy rows[s] = x[token of s] on random values: the sum of
    # the k copies' gradients, rounded once (fp32 sum of at most 6 BF16 values
    # is exact here up to one rounding, checked against fp64)
    Gr = synth.bf16_normal(g, (P, h))
    xt = torch.zeros((n, h), dtype=torch.float64, requires_grad=True)
    src = torch.from_numpy((lay["src_of_slot"][:P] // k).astype(np.int64))
    (xt[src] * torch.tensor(_f64(Gr))).sum().backward()
    gx2 = oracle.dispatch_backward(Gr, lay["slot_of"], h)
    ref = xt.grad.numpy()
    got = _f64(gx2)
    # bound: k-1 fp32 additions then one BF16 rounding
    bound = 2 ** -8 * np.abs(ref) + k * 2 ** -24 * np.abs(_f64(Gr)).max() * k
    assert np.all(np.abs(got - ref) <= bound)
    # equal to the combine with unit weights (the duality the pages state)
    np.testing.assert_array_equal(gx2, oracle.combine_topk(Gr, w, lay["slot_of"], h))


def test_gather_ranks_backward_matches_autograd_and_adjoint():
    g = np.random.default_rng(10)
    n, k, e, r, h = 20, 4, 16, 4, 24
    ids = _route(11, n, k, e, masked=0.2)
    lay = oracle.layout(ids, e, r)
    rl = oracle.rank_layout(lay["is_token_in_rank"], lay["tokens_per_expert"])
    rows = int(rl["recv_offset"][-1])
    recv = _bf16(g.integers(-5, 6, size=(rows, h)))
    go = _bf16(g.integers(-5, 6, size=(n, h)))
    out = oracle.combine_gather_ranks(recv, rl["send_head"], h)
    gr = oracle.gather_ranks_backward(go, rl["send_head"], rows, h)
    assert (_f64(out) * _f64(go)).sum() == (_f64(recv) * _f64(gr)).sum()
    # autograd: every named row gets the token's gradient; others stay zero
    rt = torch.zeros((rows, h), dtype=torch.float64, requires_grad=True)
    sh = rl["send_head"]
    idx = torch.from_numpy(np.where(sh >= 0, sh, 0).astype(np.int64))
    m = torch.from_numpy(sh >= 0).unsqueeze(-1)
    (rt[idx] * m).sum(1).mul(torch.tensor(_f64(go))).sum().backward()
    np.testing.assert_array_equal(_f64(gr), rt.grad.numpy())
