"""Pins of the oracle's layout (counts, rank mask, scans, slot map) and its
records against brute force on tiny inputs, numpy library routines, closed
forms, invariants and the record sizes the pages' formulas give."""
import itertools
import os

import numpy as np
import pytest

import oracle
from combine_moe_layout_03_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_layout(ids: np.ndarray, e: int, r: int) -> dict:
    """The definitions written as direct counting, O(P^2): every slot is
    offset of its expert + number of earlier pairs with the same expert."""
    n, k = ids.shape
    per = e // r
    flat = ids.ravel().tolist()
    cnt = [sum(1 for v in flat if v == x) for x in range(e)]
    off = [sum(cnt[:x]) for x in range(e + 1)]
    mask = [[int(any(v >= 0 and v // per == q for v in ids[t])) for q in range(r)] for t in range(n)]
    slot = []
    for p, v in enumerate(flat):
        slot.append(-1 if v < 0 else off[v] + sum(1 for pp in range(p) if flat[pp] == v))
    return dict(tokens_per_expert=cnt, expert_offset=off, is_token_in_rank=mask,
                tokens_per_rank=[sum(m[q] for m in mask) for q in range(r)],
                rank_offset=[off[q * per] for q in range(r)] + [off[e]], slot_of=slot)


def _check_against_brute(ids, e, r):
    got = oracle.layout(ids, e, r)
    ref = brute_layout(ids, e, r)
    assert got["tokens_per_expert"].tolist() == ref["tokens_per_expert"]
    assert got["expert_offset"].tolist() == ref["expert_offset"]
    assert got["rank_offset"].tolist() == ref["rank_offset"]
    assert got["tokens_per_rank"].tolist() == ref["tokens_per_rank"]
    assert got["is_token_in_rank"].tolist() == ref["is_token_in_rank"]
    assert got["slot_of"].ravel().tolist() == ref["slot_of"]


def test_layout_brute_force_every_routing_tiny():
    # Every routing of N*k = 4 pairs over ids {-1, 0, 1, 2, 3}, E=4, R in {1,2,4}.
    for n, k in ((2, 2), (4, 1), (1, 4)):
        for combo in itertools.product(range(-1, 4), repeat=n * k):
            ids = np.array(combo, np.int32).reshape(n, k)
            for r in (1, 2, 4):
                _check_against_brute(ids, 4, r)


def test_layout_brute_force_random_small():
    g = np.random.default_rng(7)
    for trial in range(60):
        n, k, r = int(g.integers(1, 9)), int(g.integers(1, 5)), int(g.choice([1, 2, 4]))
        e = r * int(g.integers(1, 4))
        ids = g.integers(-1, e, size=(n, k)).astype(np.int32)
        _check_against_brute(ids, e, r)


def test_layout_library_pins_and_invariants():
    c = synth.prefill_case(seed=1, n=512)
    ids, e, r = c["topk_idx"], c["num_experts"], c["num_ranks"]
    got = oracle.layout(ids, e, r)
    flat = ids.ravel()
    valid = flat[flat >= 0]
    np.testing.assert_array_equal(got["tokens_per_expert"], np.bincount(valid, minlength=e))
    assert got["tokens_per_expert"].sum() == ids.size  # no -1 here: counts sum to N*k
    # the slot map is the stable sort of pairs by expert
    order = np.argsort(np.where(flat >= 0, flat, e), kind="stable")[: valid.size]
    np.testing.assert_array_equal(got["src_of_slot"][: valid.size], order)
    assert np.all(got["src_of_slot"][valid.size:] == -1)
    # bijection between valid pairs and [0, P)
    assert sorted(got["slot_of"].ravel().tolist()) == list(range(ids.size))
    np.testing.assert_array_equal(got["slot_of"].ravel()[got["src_of_slot"]], np.arange(ids.size))
    # rank mask and per-rank token counts
    per = e // r
    mask = np.zeros((ids.shape[0], r), np.uint8)
    for q in range(r):
        mask[:, q] = np.any(ids // per == q, axis=1)
    np.testing.assert_array_equal(got["is_token_in_rank"], mask)
    np.testing.assert_array_equal(got["tokens_per_rank"], mask.sum(0))
    np.testing.assert_array_equal(got["rank_offset"], got["expert_offset"][::per])


def test_layout_closed_form_round_robin():
    # ids[t, j] = (t*k + j) mod E gives count[e] = floor(Nk/E) + [e < Nk mod E]
    # and slot_of[t, j] = offset[e] + (t*k + j) div E.
    n, k, e, r = 37, 3, 8, 4
    p = np.arange(n * k)
    ids = (p % e).astype(np.int32).reshape(n, k)
    got = oracle.layout(ids, e, r)
    cnt = n * k // e + (np.arange(e) < (n * k) % e)
    np.testing.assert_array_equal(got["tokens_per_expert"], cnt)
    off = np.concatenate([[0], np.cumsum(cnt)])
    np.testing.assert_array_equal(got["slot_of"].ravel(), off[p % e] + p // e)


def test_layout_special_cases():
    # all tokens padded (-1): nothing routed anywhere
    got = oracle.layout(np.full((5, 4), -1, np.int32), 8, 2)
    assert got["num_pairs"] == 0 and np.all(got["slot_of"] == -1)
    assert np.all(got["is_token_in_rank"] == 0) and np.all(got["src_of_slot"] == -1)
    # all pairs to one expert: slots in (t, j) order
    got = oracle.layout(np.full((6, 2), 5, np.int32), 8, 4)
    assert got["tokens_per_expert"][5] == 12 and got["expert_offset"][5] == 0
    np.testing.assert_array_equal(got["slot_of"].ravel(), np.arange(12))
    assert got["tokens_per_rank"].tolist() == [0, 0, 6, 0]
    # duplicate experts in a row get two slots, the token counts once per rank
    got = oracle.layout(np.array([[3, 3]], np.int32), 4, 2)
    assert got["tokens_per_expert"].tolist() == [0, 0, 0, 2]
    assert got["tokens_per_rank"].tolist() == [0, 1]
    assert got["slot_of"].tolist() == [[0, 1]]
    # empty input
    got = oracle.layout(np.zeros((0, 8), np.int32), 16, 4)
    assert got["num_pairs"] == 0 and got["expert_offset"].tolist() == [0] * 17


@pytest.mark.parametrize("bad", [-2, 16, 1000])
def test_layout_rejects_ids_out_of_range(bad):
    ids = np.zeros((3, 2), np.int32)
    ids[1, 1] = bad
    with pytest.raises(ValueError):
        oracle.layout(ids, 16, 4)


def test_layout_rejects_experts_not_divisible_by_ranks():
    with pytest.raises(ValueError):
        oracle.layout(np.zeros((2, 2), np.int32), 10, 4)


# ------------------------------------------------------------------ records --

def _golden_sizes():
    rows = []
    with open(os.path.join(GOLDEN, "record_sizes.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, *vals = line.split()
                rows.append((name, *map(int, vals)))
    return rows


@pytest.mark.parametrize("row", _golden_sizes(), ids=lambda r: r[0])
def test_record_sizes_match_page_formulas(row):
    name, k, h, ik, ok, rp, rs, rec_bytes, body = row
    lay = oracle.record_layout(k, h, ik, ok, rp, rs)
    assert lay["record_bytes"] == rec_bytes
    pad = lambda x: (x + 15) // 16 * 16
    assert lay["record_bytes"] - 16 - 2 * pad(4 * k) == body
    for key in ("off_ids", "off_weights", "off_payload", "off_scales", "record_bytes"):
        assert lay[key] % 16 == 0


def _parse(rec: np.ndarray, lay: dict, k: int):
    hdr = rec[:16].view(np.int32)
    ids = rec[lay["off_ids"]: lay["off_ids"] + 4 * k].view(np.int32)
    w = rec[lay["off_weights"]: lay["off_weights"] + 4 * k].view(np.float32)
    pay = rec[lay["off_payload"]: lay["off_payload"] + lay["payload_bytes"]]
    sc = rec[lay["off_scales"]: lay["off_scales"] + lay["scale_bytes"]]
    return hdr, ids, w, pay, sc


def _padding_mask(lay: dict, k: int) -> np.ndarray:
    used = np.zeros(lay["record_bytes"], bool)
    used[:12] = True
    used[lay["off_ids"]: lay["off_ids"] + 4 * k] = True
    used[lay["off_weights"]: lay["off_weights"] + 4 * k] = True
    used[lay["off_payload"]: lay["off_payload"] + lay["payload_bytes"]] = True
    used[lay["off_scales"]: lay["off_scales"] + lay["scale_bytes"]] = True
    return ~used


def test_records_round_trip_bf16_with_rank_markers():
    # Markers in the spirit of the all-gather test on the ds-exp-ag page: each
    # token's hidden row, ids and weights encode the token and its virtual
    # source rank, so a misplaced record is visible.
    n, k, e, r, h = 24, 3, 12, 3, 64
    g = np.random.default_rng(11)
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    ids[4, 1] = -1
    src_rank = np.arange(n) // (n // r)
    w = (src_rank[:, None] + 1) * 0.125 + np.arange(k)[None, :] * 0.001
    w = w.astype(np.float32)
    hid = (np.arange(n)[:, None] * 1000 + src_rank[:, None] * 100000 + np.arange(h)[None, :])
    hid = (hid.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    lay_o = oracle.layout(ids, e, r)
    rec = oracle.dispatch(ids, w, hid, None, lay_o["slot_of"], lay_o["num_pairs"], oracle.BF16,
                          oracle.BF16, h)
    lay = oracle.record_layout(k, h, oracle.BF16, oracle.BF16)
    pad = _padding_mask(lay, k)
    per = e // r
    for s in range(lay_o["num_pairs"]):
        hdr, rids, rw, pay, sc = _parse(rec[s], lay, k)
        t, j, ex = hdr[0], hdr[1], hdr[2]
        assert hdr[3] == 0
        assert ids[t, j] == ex and lay_o["slot_of"][t, j] == s
        assert lay_o["rank_offset"][ex // per] <= s < lay_o["rank_offset"][ex // per + 1]
        np.testing.assert_array_equal(rids, ids[t])
        np.testing.assert_array_equal(rw.view(np.uint32), w[t].view(np.uint32))
        np.testing.assert_array_equal(pay.view(np.uint16), hid[t])
        assert np.all(rec[s][pad] == 0)


def test_records_raw_bytes_survive_with_marker_words():
    c = synth.decode_case(seed=3, n=16)
    ids, w = c["topk_idx"], c["topk_weights"]
    lay_o = oracle.layout(ids, 256, 8)
    rec = oracle.dispatch(ids, w, c["payload"], c["scales"], lay_o["slot_of"], lay_o["num_pairs"],
                          oracle.RAW, oracle.RAW, c["hidden"], 3584, 448)
    lay = oracle.record_layout(8, c["hidden"], oracle.RAW, oracle.RAW, 3584, 448)
    assert np.any(c["payload"].view(np.uint32) == synth.PAGE_SENTINEL_WORD)
    for s in range(lay_o["num_pairs"]):
        hdr, rids, rw, pay, sc = _parse(rec[s], lay, 8)
        np.testing.assert_array_equal(pay, c["payload"][hdr[0]])
        np.testing.assert_array_equal(sc, c["scales"][hdr[0]])


def test_records_fp8_payload_equals_group_quantiser():
    c = synth.prefill_case(seed=2, n=8, hidden=512)
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    lay_o = oracle.layout(ids, 256, 8)
    rec = oracle.dispatch(ids, w, x, None, lay_o["slot_of"], lay_o["num_pairs"], oracle.BF16,
                          oracle.FP8_E4M3_B128, 512)
    lay = oracle.record_layout(8, 512, oracle.BF16, oracle.FP8_E4M3_B128)
    for s in range(lay_o["num_pairs"]):
        hdr, _, _, pay, sc = _parse(rec[s], lay, 8)
        for gi in range(4):
            q, scale = oracle.fp8_group(x[hdr[0], gi * 128:(gi + 1) * 128])
            np.testing.assert_array_equal(pay[gi * 128:(gi + 1) * 128], q)
            assert sc.view(np.float32)[gi] == np.float32(scale)
