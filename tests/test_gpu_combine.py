"""GPU parity of moe_combine (through the C ABI) against the oracle: top-k
weighted reduction, cross-rank sum and the rank-grouped form, within
|gpu - ref| <= 1e-2 * max(1, |ref|) (and, since both sides run the same fp32
operations in the same order, bit-exact); full-size workloads on sampled
token ranges; the identity-expert round trip combine(dispatch(x))."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, assert_combine_close, dev_bf16, dev_f32, dev_i32, host_bf16

pytestmark = pytest.mark.gpu


def gpu_combine(mode, ids, w, y_u16, e, r, h, slot_of=None):
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, h)
    ids_d = dev_i32(ids)
    if slot_of is None:
        lay = moe.moe_layout(d, ids_d)
        slot_of = lay["slot_of"]
    out = moe.moe_combine(d, mode, dev_bf16(y_u16), ids_d, dev_f32(w), slot_of)
    torch.cuda.synchronize()
    return host_bf16(out)


def check_topk(ids, w, e, r, h, seed=0, mode=0, ranges=None):
    lay = oracle.layout(ids, e, r)
    y = synth.bf16_normal(synth.rng_for(seed, 77), (max(lay["num_pairs"], 1), h))
    got = gpu_combine(mode, ids, w, y, e, r, h)
    fn = (lambda a, b, c_: oracle.combine_topk(y, b, c_, h)) if mode == 0 else \
         (lambda a, b, c_: oracle.combine_topk_ranks(y, a, b, c_, e, r, h))
    if ranges is None:
        ref = fn(ids, w, lay["slot_of"])
        assert_combine_close(got, ref, f"mode {mode}")
        np.testing.assert_array_equal(got, ref)
        return
    for t0, t1 in ranges:
        s = slice(t0, t1)
        ref = fn(ids[s], w[s], lay["slot_of"][s])
        assert_combine_close(got[s], ref, f"mode {mode} tokens {t0}:{t1}")
        np.testing.assert_array_equal(got[s], ref)


@pytest.mark.parametrize("mode", [0, 2])
def test_tiny(mode):
    c = synth.tiny_case(seed=1)
    check_topk(c["topk_idx"], c["topk_weights"], 16, 2, 1024, mode=mode)


@pytest.mark.parametrize("n", [1, 8, 64, 256])
def test_decode_shapes(n):
    c = synth.decode_case(seed=n, n=n)
    check_topk(c["topk_idx"], c["topk_weights"], 256, 8, 7168, seed=n)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_decode_sweep_in_the_bench_mode(n):
    # every N of the decode sweep, in the mode the benchmark's step runs: the
    # top-k reduction grouped by rank where N % R == 0, else the plain one
    c = synth.decode_case(seed=300 + n, n=n)
    check_topk(c["topk_idx"], c["topk_weights"], 256, 8, 7168, seed=300 + n, mode=2 if n % 8 == 0 else 0)


@pytest.mark.parametrize("mode", [0, 2])
def test_prefill_full_size_sampled(mode):
    c = synth.prefill_case(seed=0)
    check_topk(c["topk_idx"], c["topk_weights"], 256, 8, 7168, mode=mode,
               ranges=[(0, 64), (2000, 2048), (4032, 4096)])


@pytest.mark.parametrize("t", [32, 64, 128, 256, 512])
def test_rs_topk_ranks_full(t):
    c = synth.rs_case(seed=t, tokens_per_rank=t, with_partials=False, with_expert_out=False)
    check_topk(c["topk_idx"], c["topk_weights"], 256, 4, 8192, seed=t, mode=2)


@pytest.mark.parametrize("t", [32, 64, 128, 256, 512])
def test_rs_ranks_full(t):
    from combine_moe_layout_03_gb300 import moe
    c = synth.rs_case(seed=t, tokens_per_rank=t, with_expert_out=False)
    p = c["partials_bf16"]
    r, n, h = p.shape
    d = moe.MoeDesc(n, 8, 256, r, h)
    out = moe.moe_combine(d, moe.MOE_COMBINE_RANKS, dev_bf16(p), None, None, None)
    torch.cuda.synchronize()
    got = host_bf16(out)
    ref = oracle.combine_ranks(p)
    assert_combine_close(got, ref, "ranks")
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("r", [1, 3, 8, 9])
def test_ranks_other_rank_counts(r):
    from combine_moe_layout_03_gb300 import moe
    p = synth.bf16_normal(synth.rng_for(r, 5), (r, 6 * r, 136))
    d = moe.MoeDesc(6 * r, 1, r, r, 136)
    got = host_bf16(moe.moe_combine(d, moe.MOE_COMBINE_RANKS, dev_bf16(p), None, None, None))
    np.testing.assert_array_equal(got, oracle.combine_ranks(p))


@pytest.mark.parametrize("n,k,e,r,h", [
    (50, 32, 64, 4, 264),     # k = 32 (four load batches), ragged hidden chunks
    (37, 1, 8, 8, 1032),      # k = 1: the row itself
    (64, 6, 96, 12, 8),       # smallest hidden
    (40, 8, 16, 2, 65536),    # wide rows: grid.y > 1 many times
])
def test_shapes(n, k, e, r, h):
    g = np.random.default_rng(n + k)
    ids = g.integers(-1, e, size=(n, k)).astype(np.int32)
    w = g.standard_normal((n, k)).astype(np.float32)
    for mode in (0, 2):
        if mode == 2 and n % r:
            continue
        check_topk(ids, w, e, r, h, seed=n, mode=mode)


def test_identity_expert_round_trip_fp8():
    """combine(identity(dispatch(x))) on the GPU against the same chain in the
    oracle; also close to sum_j w_j x within the FP8 format bound."""
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=5, n=256)
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    n, k, h = 256, 8, 7168
    d = moe.MoeDesc(n, k, 256, 8, h, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    ids_d, w_d = dev_i32(ids), dev_f32(w)
    lay = moe.moe_layout(d, ids_d)
    rec = moe.moe_dispatch(d, ids_d, w_d, dev_bf16(x), None, lay["slot_of"])
    rl = moe.moe_record_layout(d)
    q = rec[:, rl["off_payload"]:rl["off_payload"] + h].contiguous().view(torch.float8_e4m3fn)
    sc = rec[:, rl["off_scales"]:rl["off_scales"] + 4 * h // 128].contiguous().view(torch.float32)
    y = (q.float() * sc.repeat_interleave(128, dim=1)).to(torch.bfloat16)  # identity expert
    out = moe.moe_combine(moe.MoeDesc(n, k, 256, 8, h), moe.MOE_COMBINE_TOPK, y, ids_d, w_d,
                          lay["slot_of"])
    got = host_bf16(out)
    ol = oracle.layout(ids, 256, 8)
    orec = oracle.dispatch(ids, w, x, None, ol["slot_of"], ol["num_pairs"], oracle.BF16,
                           oracle.FP8_E4M3_B128, h)
    oy = oracle.identity_expert(orec, k, h, oracle.FP8_E4M3_B128)
    ref = oracle.combine_topk(oy, w, ol["slot_of"], h)
    assert_combine_close(got, ref, "identity round trip")
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    approx = w.astype(np.float64).sum(1, keepdims=True) * xf
    gf = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    amax = np.abs(xf).reshape(n, -1, 128).max(-1).repeat(128, axis=1)
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, amax / 448 * 2.0 ** -10) * 1.01 + \
        2.0 ** -7 * np.abs(approx) + 1e-30
    assert np.all(np.abs(gf - approx) <= bound)


def test_empty_combine_is_a_no_op():
    from combine_moe_layout_03_gb300 import moe
    d = moe.MoeDesc(0, 8, 256, 8, 64)
    e = torch.empty((0, 8), dtype=torch.int32, device=DEV)
    out = moe.moe_combine(d, moe.MOE_COMBINE_TOPK, torch.empty((1, 64), dtype=torch.bfloat16,
                                                               device=DEV), e, e.float(), e)
    assert out.shape == (0, 64)


def test_prepared_calls_match_direct_calls():
    """The binding's pre-marshalled calls launch the same kernels on the same
    buffers: repeated calls give the direct calls' results."""
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=8, n=512)
    n, k, e, r, h = 512, 8, 256, 8, 7168
    d = moe.MoeDesc(n, k, e, r, h, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    ids, w, x = dev_i32(c["topk_idx"]), dev_f32(c["topk_weights"]), dev_bf16(c["hidden_bf16"])
    ref_lay = moe.moe_layout(d, ids)
    ref_rec = moe.moe_dispatch(d, ids, w, x, None, ref_lay["slot_of"])
    y = dev_bf16(synth.bf16_normal(synth.rng_for(1), (n * k, h)))
    cd = moe.MoeDesc(n, k, e, r, h)
    ref_out = moe.moe_combine(cd, moe.MOE_COMBINE_TOPK_RANKS, y, ids, w, ref_lay["slot_of"])
    lay = moe.layout_outputs(d, DEV)
    ws = torch.empty(moe.moe_workspace_size(d), dtype=torch.uint8, device=DEV)
    rec = torch.zeros_like(ref_rec)
    out = torch.zeros_like(ref_out)
    pl = moe.prepare_layout(d, ids, lay, ws)
    pd = moe.prepare_dispatch(d, ids, w, x, None, lay["slot_of"], rec)
    pc = moe.prepare_combine(cd, moe.MOE_COMBINE_TOPK_RANKS, y, ids, w, lay["slot_of"], out)
    for _ in range(2):
        pl()
        pd()
        pc()
    torch.cuda.synchronize()
    assert torch.equal(lay["slot_of"], ref_lay["slot_of"])
    assert torch.equal(rec, ref_rec)
    assert torch.equal(out, ref_out)


def _check_norm(mode, n, k, e, r, h, seed, ranges=None):
    """Fused combine + residual + RMSNorm against the oracle: residual_out
    bit-exact, normed within the contract tolerance and at most one BF16 step
    apart (the sum of squares and rsqrt round differently)."""
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(seed)
    res = synth.bf16_normal(g, (n, h))
    gamma = synth.bf16_normal(g, (h,))
    eps = 1e-6
    d = moe.MoeDesc(n, k, e, r, h)
    if mode == moe.MOE_COMBINE_RANKS:
        y = synth.bf16_normal(g, (r, n, h))
        ids = w = None
        so_d = ids_d = w_d = None
        so = None
    else:
        ids = synth.route_uniform(g, n, e, k)
        ids[: max(1, n // 10), -1] = -1
        w = synth.weights_softmax(g, n, k)
        lay = oracle.layout(ids, e, r)
        so = lay["slot_of"]
        y = synth.bf16_normal(g, (max(lay["num_pairs"], 1), h))
        ids_d, w_d = dev_i32(ids), dev_f32(w)
        so_d = moe.moe_layout(d, ids_d)["slot_of"]
    normed, rout = moe.moe_combine_norm(d, mode, dev_bf16(y), ids_d, w_d, so_d, dev_bf16(res),
                                        dev_bf16(gamma), eps)
    torch.cuda.synchronize()
    gn, gr = host_bf16(normed), host_bf16(rout)
    for t0, t1 in (ranges or [(0, n)]):
        s = slice(t0, t1)
        if mode == moe.MOE_COMBINE_RANKS:
            rn, rr = oracle.combine_norm(1, y[:, s], None, None, None, res[s], gamma, eps, e, r, h)
        else:
            rn, rr = oracle.combine_norm(mode, y, ids[s], w[s], so[s], res[s], gamma, eps, e, r, h)
        np.testing.assert_array_equal(gr[s], rr)
        assert_combine_close(gn[s], rn, f"norm mode {mode}")
        ulps = np.abs(gn[s].astype(np.int32) - rn.astype(np.int32))
        assert ulps.max() <= 1


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_combine_norm_tiny_and_ragged(mode):
    _check_norm(mode, 16, 2, 16, 2, 1024, seed=mode)
    _check_norm(mode, 24, 6, 96, 12, 264, seed=10 + mode)   # ragged chunks, odd k


@pytest.mark.parametrize("mode", [0, 2])
def test_combine_norm_prefill_size_sampled(mode):
    _check_norm(mode, 4096, 8, 256, 8, 7168, seed=20 + mode, ranges=[(0, 24), (4072, 4096)])


@pytest.mark.parametrize("h", [2048, 8192, 16384])
def test_combine_norm_rs_shapes(h):
    from combine_moe_layout_03_gb300 import moe
    _check_norm(moe.MOE_COMBINE_RANKS, 64, 8, 256, 4, h, seed=h)
    _check_norm(moe.MOE_COMBINE_TOPK_RANKS, 64, 8, 256, 4, h, seed=h + 1)
