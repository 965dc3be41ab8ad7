"""The skewed workload at its full size against the oracle: N=16384 tokens,
hidden 7168, top-8 of 256 experts with Zipf(1.2) popularity (8 experts never
chosen), R=16 virtual ranks; FP8 e4m3 per-128 dispatch and the BF16 combine
grouped by rank, through the calls the benchmark times (moe_layout_dispatch,
then moe_combine in TOPK_RANKS mode).

* layout: every output array, bit for bit;
* records: every record's header, id row and weight row against the routing;
  all k records of a token carry the same payload; the payload and scales
  byte for byte against the oracle on sampled tokens -- the first, middle
  and last tokens, the first and last tokens routed to the hottest expert,
  and the tokens whose records border the empty experts' (empty) regions;
* combine: the same sampled tokens plus more of the hottest expert's, bit for
  bit and within |gpu - ref| <= 1e-2 * max(1, |ref|)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, assert_combine_close, dev_bf16, dev_f32, dev_i32, host, host_bf16

pytestmark = pytest.mark.gpu

E, R, H = 256, 16, 7168
LAYOUT_KEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset",
               "rank_offset", "slot_of", "src_of_slot")


@pytest.fixture(scope="module")
def skewed():
    c = synth.skewed_case(seed=3)
    ref = oracle.layout(c["topk_idx"], E, R)
    return c, ref


def _sample_tokens(c, ref, per_edge=24):
    """Token indices to check one by one (sorted, unique)."""
    ids = c["topk_idx"]
    n = ids.shape[0]
    tok = set(range(0, 32)) | set(range(n // 2 - 16, n // 2 + 16)) | set(range(n - 32, n))
    hot = int(np.argmax(ref["tokens_per_expert"]))
    hot_tokens = np.flatnonzero((ids == hot).any(axis=1))
    tok |= set(hot_tokens[:per_edge].tolist()) | set(hot_tokens[-per_edge:].tolist())
    # the records on either side of every empty expert's (empty) region
    src = ref["src_of_slot"]
    P = ref["num_pairs"]
    for e in np.flatnonzero(ref["tokens_per_expert"] == 0):
        off = int(ref["expert_offset"][e])
        for s in (off - 1, off):
            if 0 <= s < P:
                tok.add(int(src[s]) // ids.shape[1])
    return np.array(sorted(tok), dtype=np.int64), hot


def test_skewed_routing_has_the_configured_shape(skewed):
    c, ref = skewed
    tpe = ref["tokens_per_expert"]
    assert (tpe == 0).sum() >= 8
    assert tpe.max() / tpe.mean() > 10          # a strongly skewed expert load
    assert ref["num_pairs"] == 16384 * 8


def test_skewed_layout_dispatch_full_size(skewed):
    from combine_moe_layout_03_gb300 import moe
    c, ref = skewed
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    n, k = ids.shape
    d = moe.MoeDesc(n, k, E, R, H, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    lay_rec = moe.moe_record_layout(d)
    rb = lay_rec["record_bytes"]
    assert rb == 7472
    rec = torch.full((n * k + 4, rb), 0xAB, dtype=torch.uint8, device=DEV)
    lay, rec = moe.moe_layout_dispatch(d, dev_i32(ids), dev_f32(w), dev_bf16(x), None, records=rec)
    torch.cuda.synchronize()
    assert moe.moe_layout_status(lay["workspace"]) == moe.MOE_OK
    for key in LAYOUT_KEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key], err_msg=key)
    P = ref["num_pairs"]
    got = host(rec)
    del rec
    assert np.all(got[P:] == 0xAB)
    got = got[:P]

    # every record: header, id row, weight row and zero padding
    hdr = got[:, :16].view(np.int32)
    t_of, j_of = hdr[:, 0], hdr[:, 1]
    np.testing.assert_array_equal(ref["slot_of"][t_of, j_of], np.arange(P))
    np.testing.assert_array_equal(hdr[:, 2], ids[t_of, j_of])
    assert np.all(hdr[:, 3] == 0)
    oi, ow, op = lay_rec["off_ids"], lay_rec["off_weights"], lay_rec["off_payload"]
    np.testing.assert_array_equal(got[:, oi:oi + 4 * k].view(np.int32), ids[t_of])
    np.testing.assert_array_equal(got[:, ow:ow + 4 * k].view(np.uint32), w.view(np.uint32)[t_of])
    # the k records of a token carry one payload + scales image
    first = got[ref["slot_of"][:, 0], op:]
    for j in range(1, k):
        np.testing.assert_array_equal(got[ref["slot_of"][:, j], op:], first, err_msg=f"j={j}")
    del first

    # payload and scales byte for byte on the sampled tokens (the oracle
    # writes them to records 0, 1, ... in pair order and numbers the tokens
    # from 0)
    tok, _ = _sample_tokens(c, ref)
    m = tok.size
    want = oracle.dispatch(ids[tok], w[tok], x[tok], None, np.arange(m * k, dtype=np.int32).reshape(m, k),
                           m * k, oracle.BF16, oracle.FP8_E4M3_B128, H)
    want[:, :4].view(np.int32)[:, 0] = np.repeat(tok, k).astype(np.int32)
    np.testing.assert_array_equal(got[ref["slot_of"][tok].ravel()], want)


def test_skewed_topk_ranks_combine_full_size(skewed):
    from combine_moe_layout_03_gb300 import moe
    c, ref = skewed
    ids, w = c["topk_idx"], c["topk_weights"]
    n, k = ids.shape
    P = ref["num_pairs"]
    tok, hot = _sample_tokens(c, ref, per_edge=64)
    # pad the sample to whole groups of R tokens (the oracle's rank-grouped
    # combine takes N % R == 0; a token's result does not depend on the rest)
    have = set(tok.tolist())
    extra = [t for t in range(n) if t not in have][: (-len(tok)) % R]
    tok = np.array(sorted(tok.tolist() + extra), dtype=np.int64)
    need = np.unique(ref["slot_of"][tok].ravel())
    # expert outputs in slot order, drawn chunk by chunk and uploaded; only the
    # rows of the sampled tokens are kept on the host
    g = synth.rng_for(3, 55)
    y_dev = torch.empty((P, H), dtype=torch.bfloat16, device=DEV)
    y_need = np.empty((need.size, H), np.uint16)
    step = 8192
    for s0 in range(0, P, step):
        s1 = min(P, s0 + step)
        chunk = synth.bf16_normal(g, (s1 - s0, H))
        y_dev[s0:s1] = dev_bf16(chunk)
        sel = (need >= s0) & (need < s1)
        y_need[sel] = chunk[need[sel] - s0]
    d = moe.MoeDesc(n, k, E, R, H)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    out = moe.moe_combine(d, moe.MOE_COMBINE_TOPK_RANKS, y_dev, ids_d, dev_f32(w), lay["slot_of"])
    torch.cuda.synchronize()
    got = host_bf16(out[torch.from_numpy(tok).to(DEV)])
    # the oracle on the sampled tokens, their slots renumbered into y_need
    remap = np.searchsorted(need, ref["slot_of"][tok])
    want = oracle.combine_topk_ranks(y_need, ids[tok], w[tok], remap.astype(np.int32), E, R, H)
    assert_combine_close(got, want, "skewed TOPK_RANKS")
    np.testing.assert_array_equal(got, want)
    assert (ids[tok] == hot).any(axis=1).sum() >= 64
