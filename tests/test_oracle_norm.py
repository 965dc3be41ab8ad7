"""Pins of the oracle's combine + residual add + RMSNorm against torch's own
RMSNorm (independent library code), exact cases and reductions to the plain
combine."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth


def _bf16(f):
    return torch.from_numpy(np.asarray(f, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(b):
    return oracle.bf16_to_f32_array(b).astype(np.float64)


def test_residual_out_is_the_combine_when_residual_is_zero():
    c = synth.tiny_case(seed=2)
    ids, w, h = c["topk_idx"], c["topk_weights"], 256
    lay = oracle.layout(ids, 16, 2)
    y = synth.bf16_normal(synth.rng_for(3), (lay["num_pairs"], h))
    zero = np.zeros((ids.shape[0], h), np.uint16)
    gamma = _bf16(np.ones(h))
    _, r0 = oracle.combine_norm(0, y, ids, w, lay["slot_of"], zero, gamma, 1e-6, 16, 2, h)
    np.testing.assert_array_equal(r0, oracle.combine_topk(y, w, lay["slot_of"], h))
    _, r2 = oracle.combine_norm(2, y, ids, w, lay["slot_of"], zero, gamma, 1e-6, 16, 2, h)
    np.testing.assert_array_equal(r2, oracle.combine_topk_ranks(y, ids, w, lay["slot_of"], 16, 2, h))
    p = synth.bf16_normal(synth.rng_for(4), (4, 8, h))
    _, r1 = oracle.combine_norm(1, p, None, None, None, np.zeros((8, h), np.uint16), gamma, 1e-6,
                                4, 4, h)
    np.testing.assert_array_equal(r1, oracle.combine_ranks(p))


def test_normed_matches_torch_rms_norm():
    # Small-integer partials and residual: x is exact in fp32 and in BF16, so
    # torch's fp64 RMSNorm of x is the exact reference; the oracle's fp32
    # products may move the BF16 result by at most one step.
    g = np.random.default_rng(5)
    r, n, h = 4, 8, 512
    p = _bf16(g.integers(-20, 21, size=(r, n, h)))
    res = _bf16(g.integers(-20, 21, size=(n, h)))
    gamma = _bf16(np.abs(g.standard_normal(h)) + 0.5)
    eps = 1e-6
    normed, rout = oracle.combine_norm(1, p, None, None, None, res, gamma, eps, r, r, h)
    x = _f(p).sum(0) + _f(res)
    np.testing.assert_array_equal(_f(rout), x)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (h,),
                                       weight=torch.from_numpy(_f(gamma)), eps=eps).numpy()
    assert np.all(np.abs(_f(normed) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)


def test_constant_row_with_zero_eps_gives_gamma():
    # x = 2 everywhere: mean(x^2) = 4, scale = 1/2 exactly, x * scale = 1.
    h = 64
    gamma = synth.bf16_normal(synth.rng_for(6), (h,))
    res = _bf16(np.full((2, h), 2.0))
    p = np.zeros((2, 2, h), np.uint16)
    normed, rout = oracle.combine_norm(1, p, None, None, None, res, gamma, 0.0, 2, 2, h)
    np.testing.assert_array_equal(normed[0], gamma)
    np.testing.assert_array_equal(normed[1], gamma)
    assert np.all(_f(rout) == 2.0)


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.combine_norm(1, np.zeros((2, 3, 8), np.uint16), None, None, None,
                            np.zeros((3, 8), np.uint16), np.zeros(8, np.uint16), 1e-6, 2, 2, 8)
