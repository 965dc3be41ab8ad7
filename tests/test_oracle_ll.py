"""Pins of the oracle's fixed-capacity, expert-major receive layout (DeepEP
low-latency dispatch): per-expert and per-(expert, source rank) counts from
numpy bincounts over each rank's token range, positions that are a
permutation of 0..count-1 in ascending (token, k) order, the token index
within its source rank, overflow past the capacity, agreement with the
pinned stable slot map, and packed rows equal to the pinned records'
payload and scales."""
import numpy as np
import pytest

import oracle
from combine_moe_layout_03_gb300 import synth


def _route(seed, n, k, e):
    g = np.random.default_rng(seed)
    return np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)


@pytest.mark.parametrize("seed,R,T,maxT,k,E", [(1, 4, 24, 32, 4, 16), (2, 8, 16, 16, 8, 64),
                                                (3, 2, 40, 40, 6, 8)])
def test_ll_layout_counts_and_positions(seed, R, T, maxT, k, E):
    ids = _route(seed, R * T, k, E)
    ll = oracle.ll_layout(ids, E, R, maxT)
    cap = R * maxT
    for e in range(E):
        per_src = np.array([np.count_nonzero(ids[s * T:(s + 1) * T] == e) for s in range(R)])
        assert ll["recv_count"][e] == min(per_src.sum(), cap)
        begins = np.concatenate([[0], np.cumsum(per_src)[:-1]])
        for s in range(R):
            b, c = int(ll["layout_range"][e, s] >> 32), int(ll["layout_range"][e, s] & 0xFFFFFFFF)
            assert b == min(begins[s], cap) and c == min(begins[s] + per_src[s], cap) - b
        # the pairs routed to e, in ascending (t, k) order, take 0, 1, ...
        t_of, j_of = np.nonzero(ids == e)
        pos = ll["ll_slot_of"][t_of, j_of]
        np.testing.assert_array_equal(pos, e * cap + np.arange(t_of.size))
        np.testing.assert_array_equal(ll["src_info"][e, : t_of.size], t_of % T)
        assert np.all(ll["src_info"][e, t_of.size:] == -1)
    # every pair has a position (no overflow here) and the positions are distinct
    assert np.all(ll["ll_slot_of"] >= 0)
    assert np.unique(ll["ll_slot_of"]).size == ids.size


def test_ll_layout_equals_stable_slot_offset_within_expert():
    c = synth.decode_case(seed=4, n=256)
    ids = c["topk_idx"]
    E, R, maxT = 256, 8, 32
    lay = oracle.layout(ids, E, R)
    ll = oracle.ll_layout(ids, E, R, maxT)
    cap = R * maxT
    within = lay["slot_of"] - lay["expert_offset"][ids]
    np.testing.assert_array_equal(ll["ll_slot_of"], np.where(within < cap, ids * cap + within, -1))
    np.testing.assert_array_equal(ll["recv_count"], np.minimum(lay["tokens_per_expert"], cap))


def test_ll_layout_overflow_keeps_the_first_pairs():
    # every token sends its k pairs to experts 0..k-1: each expert receives N
    # pairs but holds only R * max_tokens_per_rank of them
    R, T, maxT, k, E = 4, 8, 8, 2, 4
    ids = np.tile(np.arange(k, dtype=np.int32), (R * T, 1))
    ll = oracle.ll_layout(ids, E, R, maxT)  # capacity 32 = N: no overflow yet
    assert np.all(ll["ll_slot_of"] >= 0)
    ids2 = np.zeros((R * T, k), np.int32)
    ids2[:, 1] = -1
    ids2[::2, 1] = 0  # expert 0 gets 48 pairs > 32 slots
    ll2 = oracle.ll_layout(ids2, E, R, maxT)
    t_of, j_of = np.nonzero(ids2 == 0)
    pos = ll2["ll_slot_of"][t_of, j_of]
    np.testing.assert_array_equal(pos[:32], np.arange(32))
    assert np.all(pos[32:] == -1)
    assert ll2["recv_count"][0] == 32 and np.all(ll2["recv_count"][1:] == 0)
    lr = ll2["layout_range"][0]
    begin, cnt = lr >> 32, lr & 0xFFFFFFFF
    # source ranks 0 and 1 hold 12 pairs each, rank 2 the last 8, rank 3 none
    np.testing.assert_array_equal(begin, [0, 12, 24, 32])
    np.testing.assert_array_equal(cnt, [12, 12, 8, 0])
    assert np.all(ll2["ll_slot_of"][ids2 < 0] == -1)


def test_ll_layout_rejects_uneven_or_oversize_ranks():
    ids = _route(5, 30, 2, 8)
    with pytest.raises(ValueError):
        oracle.ll_layout(ids, 8, 4, 16)  # 30 tokens do not split over 4 ranks
    with pytest.raises(ValueError):
        oracle.ll_layout(ids, 8, 3, 8)   # 10 tokens per rank > 8


@pytest.mark.parametrize("out_kind", [oracle.BF16, oracle.FP8_E4M3_B128, oracle.NVFP4_B16, oracle.RAW,
                                      oracle.FP8_E4M3_UE8M0])
def test_dispatch_ll_rows_are_the_records_payload(out_kind):
    E, R, maxT = 256, 8, 4
    if out_kind == oracle.RAW:
        c = synth.decode_case(seed=6, n=32, payload_bytes=512, scale_bytes=64)
        x, sc, H, pbr, sbr = c["payload"], c["scales"], 512, 512, 64
    else:
        c = synth.prefill_case(seed=6, n=32, hidden=256)
        x, sc, H, pbr, sbr = c["hidden_bf16"], None, 256, 0, 0
    ids, w = c["topk_idx"], c["topk_weights"]
    in_kind = oracle.RAW if out_kind == oracle.RAW else oracle.BF16
    lay = oracle.layout(ids, E, R)
    rec = oracle.dispatch(ids, w, x, sc, lay["slot_of"], lay["num_pairs"], in_kind, out_kind, H, pbr, sbr)
    rl = oracle.record_layout(8, H, in_kind, out_kind, pbr, sbr)
    ll = oracle.ll_layout(ids, E, R, maxT)
    rows = E * R * maxT
    xo, so = oracle.dispatch_ll(x, sc, ll["ll_slot_of"], rows, in_kind, out_kind, H, pbr, sbr)
    pb, sb = rl["payload_bytes"], rl["scale_bytes"]
    sr = (sb + 15) // 16 * 16  # scale rows padded to 16 bytes
    assert xo.shape == (rows, pb) and so.shape == (rows, sr)
    filled = np.zeros(rows, bool)
    for t in range(32):
        for j in range(8):
            p, s = ll["ll_slot_of"][t, j], lay["slot_of"][t, j]
            np.testing.assert_array_equal(xo[p], rec[s, rl["off_payload"]:rl["off_payload"] + pb])
            np.testing.assert_array_equal(so[p, :sb], rec[s, rl["off_scales"]:rl["off_scales"] + sb])
            assert not so[p, sb:].any()
            filled[p] = True
    assert not xo[~filled].any() and not so[~filled].any()
