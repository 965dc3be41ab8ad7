"""Pins of the oracle's combine (top-k weighted reduction, cross-rank sum and
the fused form) against exact arithmetic on exactly representable inputs, an
fp64 reference with the closed-form fp32/BF16 error bound, the identity-expert
property combine(dispatch(x)) = sum_j w_j x, orders that change the result,
and special cases that reduce to one another."""
import numpy as np
import torch

import oracle
from combine_moe_layout_03_gb300 import synth


def _bf16(f):
    f = np.asarray(f, np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f32(b):
    return oracle.bf16_to_f32_array(b).astype(np.float64)


def test_combine_topk_exact_on_dyadic_inputs():
    # Small integers times powers of two: every fp32 step is exact, so the
    # result is the exact sum (also exact in BF16 when it has <= 8 bits).
    n, k, e, h = 10, 4, 8, 16
    g = np.random.default_rng(0)
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    ids[2, 3] = -1
    lay = oracle.layout(ids, e, 2)
    w = g.choice([0.25, 0.5, 1.0, 2.0], size=(n, k)).astype(np.float32)
    y = _bf16(g.integers(-8, 9, size=(lay["num_pairs"], h)))
    out = oracle.combine_topk(y, w, lay["slot_of"], h)
    exact = np.zeros((n, h))
    for t in range(n):
        for j in range(k):
            s = lay["slot_of"][t, j]
            if s >= 0:
                exact[t] += float(w[t, j]) * _f32(y[s])
    np.testing.assert_array_equal(_f32(out), exact)


def test_combine_topk_within_fp32_bf16_bound_of_f64():
    c = synth.tiny_case(seed=4)
    ids, w, h = c["topk_idx"], c["topk_weights"], c["hidden"]
    lay = oracle.layout(ids, c["num_experts"], c["num_ranks"])
    y = synth.bf16_normal(synth.rng_for(9), (lay["num_pairs"], h))
    out = _f32(oracle.combine_topk(y, w, lay["slot_of"], h))
    ref = oracle.combine_topk_f64(y, w, lay["slot_of"], h)
    absum = np.zeros_like(ref)
    for j in range(ids.shape[1]):
        absum += np.abs(w[:, j:j + 1].astype(np.float64)) * np.abs(_f32(y[lay["slot_of"][:, j]]))
    k = ids.shape[1]
    bound = 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * k * 2.0 ** -24 * absum + 2.0 ** -133
    assert np.all(np.abs(out - ref) <= bound)
    # the contract tolerance holds with room to spare
    assert np.all(np.abs(out - ref) <= 1e-2 * np.maximum(1, np.abs(ref)))


def test_identity_expert_combine_equals_weighted_token_bf16():
    c = synth.tiny_case(seed=5)
    ids, w, x, h = c["topk_idx"], c["topk_weights"], c["hidden_bf16"], c["hidden"]
    lay = oracle.layout(ids, c["num_experts"], c["num_ranks"])
    rec = oracle.dispatch(ids, w, x, None, lay["slot_of"], lay["num_pairs"], oracle.BF16,
                          oracle.BF16, h)
    y = oracle.identity_expert(rec, ids.shape[1], h, oracle.BF16)
    out = _f32(oracle.combine_topk(y, w, lay["slot_of"], h))
    ref = w.astype(np.float64).sum(1, keepdims=True) * _f32(x)
    k = ids.shape[1]
    bound = 2.0 ** -8 * np.abs(ref) + 2 * k * 2.0 ** -24 * np.abs(ref) + 2.0 ** -133
    assert np.all(np.abs(out - ref) <= bound)


def test_identity_expert_fp8_and_nvfp4_within_format_bound():
    c = synth.prefill_case(seed=6, n=32, hidden=256)
    ids, w, x, h = c["topk_idx"], c["topk_weights"], c["hidden_bf16"], 256
    lay = oracle.layout(ids, 256, 8)
    xf = _f32(x)
    sw = np.abs(w.astype(np.float64)).sum(1, keepdims=True)
    for kind in (oracle.FP8_E4M3_B128, oracle.NVFP4_B16):
        rec = oracle.dispatch(ids, w, x, None, lay["slot_of"], lay["num_pairs"], oracle.BF16,
                              kind, h)
        y = oracle.identity_expert(rec, 8, h, kind)
        out = _f32(oracle.combine_topk(y, w, lay["slot_of"], h))
        ref = sw * xf
        if kind == oracle.FP8_E4M3_B128:
            amax = np.abs(xf).reshape(32, -1, 128).max(-1).repeat(128, axis=1)
            fmt = np.maximum(np.abs(xf) * 2.0 ** -4, amax / 448 * 2.0 ** -10)
        else:
            amax = np.abs(xf).reshape(32, -1, 16).max(-1).repeat(16, axis=1)
            fmt = amax / 6 * (1 + 2.0 ** -4)  # <= one scale step d
        # format error, then BF16 rounding of y and of the output
        bound = sw * (fmt * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(xf)) * 1.01 + 2.0 ** -8 * np.abs(out)
        assert np.all(np.abs(out - ref) <= bound + 1e-30), kind


def test_combine_ranks_exact_and_ascending_order():
    r, n, h = 4, 8, 32
    g = np.random.default_rng(1)
    p = _bf16(g.integers(-100, 101, size=(r, n, h)))
    out = oracle.combine_ranks(p)
    np.testing.assert_array_equal(_f32(out), _f32(p).sum(0))
    # order matters: (((0 + 2^24) + 1) + (-2^24)) + 0 = 0 in fp32 ascending,
    # while any order that adds the 1 last gives 1.
    q = _bf16(np.array([2.0 ** 24, 1.0, -(2.0 ** 24), 0.0]).reshape(4, 1, 1).repeat(4, 1))
    assert np.all(_f32(oracle.combine_ranks(q)) == 0.0)
    # library pin (order-free, so within tolerance)
    p = synth.bf16_normal(synth.rng_for(2), (4, 16, 64))
    ref = torch.from_numpy(_f32(p)).float().sum(0).to(torch.bfloat16).float().numpy()
    got = _f32(oracle.combine_ranks(p))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.maximum(1, np.abs(ref)))


def test_combine_topk_ranks_reduces_to_topk_with_one_rank():
    c = synth.rs_case(seed=3, tokens_per_rank=4, hidden=64, r=4, with_partials=False,
                      with_expert_out=False)
    ids, w = c["topk_idx"], c["topk_weights"]
    lay = oracle.layout(ids, 256, 1)
    y = synth.bf16_normal(synth.rng_for(5), (lay["num_pairs"], 64))
    a = oracle.combine_topk(y, w, lay["slot_of"], 64)
    b = oracle.combine_topk_ranks(y, ids, w, lay["slot_of"], 256, 1, 64)
    np.testing.assert_array_equal(a, b)


def test_combine_topk_ranks_groups_by_rank_then_sums():
    # Token with experts on ranks (1, 0, 1): rank 0's partial is w1*y1, rank
    # 1's is fma(w2, y2, w0*y0); the sum adds rank 0 first. Values chosen so
    # the grouping is visible in fp32: 2^24 + 1 - 2^24 depends on order.
    # token 0 has experts on ranks (1, 0, 1); token 1 is padding (-1) so that
    # N % R == 0
    ids = np.array([[5, 1, 6], [-1, -1, -1]], np.int32)  # E=8, R=2
    w = np.ones((2, 3), np.float32)
    lay = oracle.layout(ids, 8, 2)
    ys = np.zeros((3, 1), np.float32)
    vals = {0: 2.0 ** 24, 1: 1.0, 2: -(2.0 ** 24)}  # by j
    for j in range(3):
        ys[lay["slot_of"][0, j]] = vals[j]
    y = _bf16(ys)
    fused = _f32(oracle.combine_topk_ranks(y, ids, w, lay["slot_of"], 8, 2, 1))
    plain = _f32(oracle.combine_topk(y, w, lay["slot_of"], 1))
    # grouped: rank0 = 1; rank1 = 2^24 - 2^24 = 0; total = 1
    assert fused[0, 0] == 1.0 and fused[1, 0] == 0.0
    # ascending j in one chain: (2^24 + 1) rounds to 2^24, then - 2^24 = 0
    assert plain[0, 0] == 0.0


def test_combine_single_term_returns_the_row():
    ids = np.array([[2], [0], [-1]], np.int32)
    lay = oracle.layout(ids, 4, 2)
    y = synth.bf16_normal(synth.rng_for(8), (lay["num_pairs"], 48))
    out = oracle.combine_topk(y, np.ones((3, 1), np.float32), lay["slot_of"], 48)
    np.testing.assert_array_equal(out[0], y[lay["slot_of"][0, 0]])
    np.testing.assert_array_equal(out[1], y[lay["slot_of"][1, 0]])
    assert np.all(out[2] == 0)
