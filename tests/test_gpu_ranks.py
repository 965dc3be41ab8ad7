"""GPU parity of the per-(token, rank) path (through the C ABI) against the
oracle: receive layout and records bit-exact, rank-gathered combine
bit-exact, and the identity round trip."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, assert_combine_close, dev_bf16, dev_f32, dev_i32, host, host_bf16

pytestmark = pytest.mark.gpu
RKEYS = ("send_head", "recv_src_idx", "recv_offset", "recv_tokens_per_expert")


def _gpu_rank_layout(ids, e, r, align):
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, 8)
    lay = moe.moe_layout(d, dev_i32(ids))
    rl = moe.moe_rank_layout(d, lay, align)
    torch.cuda.synchronize()
    return d, lay, rl


@pytest.mark.parametrize("case,align", [("prefill", 1), ("prefill", 128), ("skewed", 16),
                                        ("decode", 1), ("ragged", 8)])
def test_rank_layout(case, align):
    if case == "prefill":
        ids, e, r = synth.prefill_case(seed=1)["topk_idx"], 256, 8
    elif case == "skewed":
        ids, e, r = synth.skewed_case(seed=1)["topk_idx"], 256, 16
    elif case == "decode":
        ids, e, r = synth.decode_case(seed=1, n=256)["topk_idx"], 256, 8
    else:
        g = np.random.default_rng(4)
        ids, e, r = g.integers(-1, 96, size=(1001, 6)).astype(np.int32), 96, 12
    _, _, rl = _gpu_rank_layout(ids, e, r, align)
    lay = oracle.layout(ids, e, r)
    ref = oracle.rank_layout(lay["is_token_in_rank"], lay["tokens_per_expert"], align)
    for key in RKEYS:
        np.testing.assert_array_equal(host(rl[key]).reshape(ref[key].shape), ref[key], err_msg=key)


def _check_dispatch_ranks(c, e, r, in_kind, out_kind, x_host, x_dev, sc_host=None, sc_dev=None,
                          rp=0, rs=0, ranges=None):
    from combine_moe_layout_03_gb300 import moe
    ids, w = c["topk_idx"], c["topk_weights"]
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, c["hidden"], in_kind, out_kind, rp, rs)
    ids_d, w_d = dev_i32(ids), dev_f32(w)
    lay = moe.moe_layout(d, ids_d)
    rl = moe.moe_rank_layout(d, lay)
    rb = moe.moe_record_layout(d)["record_bytes"]
    rec = torch.full((n * r, rb), 0xAB, dtype=torch.uint8, device=DEV)
    moe.moe_dispatch_ranks(d, ids_d, w_d, x_dev, sc_dev, rl["send_head"], rec)
    torch.cuda.synchronize()
    got = host(rec)
    ol = oracle.layout(ids, e, r)
    orl = oracle.rank_layout(ol["is_token_in_rank"], ol["tokens_per_expert"])
    P = int(orl["recv_offset"][-1])
    assert np.all(got[P:] == 0xAB)
    for t0, t1 in (ranges or [(0, n)]):
        s = slice(t0, t1)
        ref = oracle.dispatch_ranks(ids[s], w[s], x_host[s], None if sc_host is None else sc_host[s],
                                    orl["send_head"][s], P, e, in_kind, out_kind, c["hidden"], rp, rs)
        slots = orl["send_head"][s].ravel()
        slots = slots[slots >= 0]
        want = ref[slots].copy()
        want[:, :4].view(np.int32)[:] += t0
        np.testing.assert_array_equal(got[slots], want)


def test_dispatch_ranks_prefill_fp8_sampled():
    c = synth.prefill_case(seed=0)
    _check_dispatch_ranks(c, 256, 8, oracle.BF16, oracle.FP8_E4M3_B128, c["hidden_bf16"],
                          dev_bf16(c["hidden_bf16"]), ranges=[(0, 32), (4064, 4096)])


def test_dispatch_ranks_small_kinds():
    c = synth.tiny_case(seed=3)
    _check_dispatch_ranks(c, 16, 2, oracle.BF16, oracle.BF16, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]))
    c = synth.prefill_case(seed=4, n=64, hidden=512)
    _check_dispatch_ranks(c, 256, 8, oracle.BF16, oracle.NVFP4_B16, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]))
    c = synth.decode_case(seed=5, n=48)
    _check_dispatch_ranks(c, 256, 8, oracle.RAW, oracle.RAW, c["payload"],
                          torch.from_numpy(c["payload"]).to(DEV), c["scales"],
                          torch.from_numpy(c["scales"]).to(DEV), 3584, 448)


@pytest.mark.parametrize("n,r,h", [(4096, 8, 7168), (1000, 16, 264), (37, 4, 8)])
def test_combine_gather_ranks(n, r, h):
    from combine_moe_layout_03_gb300 import moe
    e = 16 * r
    g = np.random.default_rng(n)
    ids = synth.route_uniform(g, n, e, 8)
    ids[: n // 7, 3] = -1
    _, _, rl = _gpu_rank_layout(ids, e, r, 1)
    P = int(host(rl["recv_offset"])[-1])
    y = synth.bf16_normal(g, (max(P, 1), h))
    d = moe.MoeDesc(n, 8, e, r, h)
    out = moe.moe_combine_gather_ranks(d, dev_bf16(y), rl["send_head"])
    torch.cuda.synchronize()
    got = host_bf16(out)
    ol = oracle.layout(ids, e, r)
    orl = oracle.rank_layout(ol["is_token_in_rank"], ol["tokens_per_expert"])
    ref = oracle.combine_gather_ranks(y, orl["send_head"], h)
    assert_combine_close(got, ref, "gather ranks")
    np.testing.assert_array_equal(got, ref)


def test_prepared_rank_calls_match_direct_calls():
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=5, n=256, hidden=1024)
    ids, w, x = dev_i32(c["topk_idx"]), dev_f32(c["topk_weights"]), dev_bf16(c["hidden_bf16"])
    d = moe.MoeDesc(256, 8, 256, 8, 1024, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    lay = moe.moe_layout(d, ids)
    direct = moe.moe_rank_layout(d, lay, 4)
    rec_direct = moe.moe_dispatch_ranks(d, ids, w, x, None, direct["send_head"])
    y = dev_bf16(synth.bf16_normal(np.random.default_rng(6), (256 * 8, 1024)))
    out_direct = moe.moe_combine_gather_ranks(moe.MoeDesc(256, 8, 256, 8, 1024), y, direct["send_head"])
    prep = {key: torch.full_like(v, -7) for key, v in direct.items()}
    rec = torch.zeros_like(rec_direct)
    out = torch.zeros_like(out_direct)
    moe.prepare_rank_layout(d, lay, 4, prep)()
    moe.prepare_dispatch_ranks(d, ids, w, x, None, prep["send_head"], rec)()
    moe.prepare_combine_gather_ranks(moe.MoeDesc(256, 8, 256, 8, 1024), y, prep["send_head"], out)()
    torch.cuda.synchronize()
    for key in direct:
        assert torch.equal(prep[key], direct[key]), key
    recv = int(direct["recv_offset"][-1])  # rows past the received ones are not written
    assert torch.equal(rec[:recv], rec_direct[:recv]) and torch.equal(out, out_direct)
