"""moe_layout_dispatch of a small routing (at most 2048 pairs: decode up to
256 tokens of top-8) runs as one kernel that computes the layout inside every
dispatch block. Its outputs -- every layout array including the -1 tail of
src_of_slot, the status word and the records -- equal the oracle's bit for
bit, on both sides of the 2048-pair limit (above it the call runs the
cluster layout kernel and the dispatch), for padding, duplicate and invalid
ids, up to 64 ranks and 1024 experts, and every payload format."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_bf16, dev_f32, dev_i32, dev_u8, host

pytestmark = pytest.mark.gpu

KEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset",
        "rank_offset", "slot_of", "src_of_slot")


def _ids(g, n, k, e, distinct=True, pad=0.0):
    ids = np.empty((n, k), np.int32)
    for t in range(n):
        ids[t] = g.choice(e, size=k, replace=not distinct)
    if pad > 0:
        ids[g.random((n, k)) < pad] = -1
    return ids


def _run(ids, w, e, r, kind, h, x_host, x_dev, sc_host=None, sc_dev=None, rp=0, rs=0,
         expect_status=None):
    """moe_layout_dispatch against the oracle; returns the layout dict."""
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    ikind = oracle.RAW if kind == oracle.RAW else oracle.BF16
    d = moe.MoeDesc(n, k, e, r, h, ikind, kind, rp, rs)
    rb = moe.moe_record_layout(d)["record_bytes"]
    rec = torch.full((n * k + 3, rb), 0xAB, dtype=torch.uint8, device=DEV)
    out = moe.layout_outputs(d, DEV)
    for key in KEYS:  # stale values that every entry must overwrite
        out[key].fill_(0x55)
    lay, rec = moe.moe_layout_dispatch(d, dev_i32(ids), dev_f32(w), x_dev, sc_dev, out=out, records=rec)
    torch.cuda.synchronize()
    status = moe.moe_layout_status(lay["workspace"])
    clean = ids.copy()
    clean[(clean < -1) | (clean >= e)] = -1
    ref = oracle.layout(clean, e, r)
    assert status == (moe.MOE_OK if expect_status is None else expect_status)
    for key in KEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key], err_msg=key)
    P = ref["num_pairs"]
    want = oracle.dispatch(ids, w, x_host, sc_host, ref["slot_of"], P, ikind, kind, h, rp, rs)
    got = host(rec)
    np.testing.assert_array_equal(got[:P], want)
    assert np.all(got[P:] == 0xAB)  # no record beyond P is touched
    return lay


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_decode_sweep_raw(n):
    """The decode workload: top-8 of 256, 8 ranks, NVFP4-sized raw payload."""
    c = synth.decode_case(seed=n, n=n)
    x, sc = c["payload"], c["scales"]
    _run(c["topk_idx"], c["topk_weights"], 256, 8, oracle.RAW, 7168, x, dev_u8(x), sc, dev_u8(sc),
         rp=x.shape[1], rs=sc.shape[1])


@pytest.mark.parametrize("n,k,e,r", [
    (2048, 1, 64, 8),     # exactly 2048 pairs: one kernel, 8 token chunks per block
    (2049, 1, 64, 8),     # one pair more: layout kernel + dispatch
    (682, 3, 96, 6),      # 2046 pairs
    (683, 3, 96, 6),      # 2049 pairs
    (256, 8, 1024, 64),   # the most experts and ranks
    (64, 32, 1024, 64),   # the largest k
    (300, 5, 64, 64),     # one expert per rank
    (2048, 1, 1, 1),      # every pair on one expert
    (3, 8, 256, 64),      # fewer tokens than ranks: blocks count several ranks
    (7, 32, 40, 4),
])
def test_limit_and_shapes(n, k, e, r):
    g = np.random.default_rng(n * 131 + k)
    ids = _ids(g, n, k, e, distinct=k <= e)
    w = g.standard_normal((n, k)).astype(np.float32)
    x = synth.bf16_normal(g, (n, 256))
    _run(ids, w, e, r, oracle.FP8_E4M3_B128, 256, x, dev_bf16(x))


@pytest.mark.parametrize("kind,h", [(oracle.BF16, 520), (oracle.FP8_E4M3_B128, 7168),
                                    (oracle.FP8_E4M3_UE8M0, 1024), (oracle.NVFP4_B16, 7168)])
def test_formats_with_padding_and_duplicates(kind, h):
    g = np.random.default_rng(h)
    n, k, e, r = 61, 8, 32, 4
    ids = _ids(g, n, k, e, distinct=False, pad=0.2)
    ids[3] = -1          # a token with no expert at all
    ids[5] = ids[5, 0]   # a token whose k ids are all the same expert
    w = g.standard_normal((n, k)).astype(np.float32)
    x = synth.bf16_normal(g, (n, h))
    _run(ids, w, e, r, kind, h, x, dev_bf16(x))


def test_invalid_ids_are_reported_and_skipped():
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(11)
    n, k, e, r = 40, 4, 64, 8
    ids = _ids(g, n, k, e)
    ids[7, 2] = 64
    ids[n - 1, 0] = -5
    ids[0, 3] = 1 << 30
    w = g.standard_normal((n, k)).astype(np.float32)
    x = synth.bf16_normal(g, (n, 128))
    _run(ids, w, e, r, oracle.BF16, 128, x, dev_bf16(x), expect_status=moe.MOE_ERR_DEVICE_IDS)
    # the next call on the same shapes reports a clean routing again
    ids2 = _ids(g, n, k, e)
    _run(ids2, w, e, r, oracle.BF16, 128, x, dev_bf16(x))


def test_every_pair_padded():
    g = np.random.default_rng(3)
    n, k, e, r = 9, 4, 16, 2
    ids = np.full((n, k), -1, np.int32)
    w = g.standard_normal((n, k)).astype(np.float32)
    x = synth.bf16_normal(g, (n, 64))
    lay = _run(ids, w, e, r, oracle.BF16, 64, x, dev_bf16(x))
    assert np.all(host(lay["src_of_slot"]) == -1)


def test_same_as_two_calls():
    """The one-kernel form and moe_layout + moe_dispatch agree bit for bit,
    without src_of_slot as well."""
    from combine_moe_layout_03_gb300 import moe
    c = synth.decode_case(seed=5, n=200)
    ids_d, w_d = dev_i32(c["topk_idx"]), dev_f32(c["topk_weights"])
    x, sc = dev_u8(c["payload"]), dev_u8(c["scales"])
    d = moe.MoeDesc(200, 8, 256, 8, 7168, oracle.RAW, oracle.RAW, c["payload"].shape[1],
                    c["scales"].shape[1])
    lay = moe.moe_layout(d, ids_d)
    rec = moe.moe_dispatch(d, ids_d, w_d, x, sc, lay["slot_of"])
    out = moe.layout_outputs(d, DEV)
    del out["src_of_slot"]
    lay2, rec2 = moe.moe_layout_dispatch(d, ids_d, w_d, x, sc, out=out)
    torch.cuda.synchronize()
    for key in KEYS[:-1]:
        assert torch.equal(lay[key], lay2[key]), key
    assert torch.equal(rec, rec2)
