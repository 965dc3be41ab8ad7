"""Pins of the oracle's rank-slot packing and padded-token mask: slot sizes
from the decode benchmark's per-token formula, numpy slicing of the packed
bytes, round trips and the mask's closed-form counts."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "slot_sizes.txt")


def _rows():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append(tuple(int(v) for v in line.split()))
    return out


@pytest.mark.parametrize("row", _rows(), ids=lambda r: f"n{r[0]}")
def test_slot_layout_matches_page_formula(row):
    n, k, hd, sd, o0, o1, o2, o3, sb = row
    off, got_sb = oracle.slot_layout([4 * k * n, 4 * k * n, hd * n, sd * n])
    assert off == [o0, o1, o2, o3] and got_sb == sb
    assert sb == n * (4 * k + 4 * k + hd + sd)


def test_slot_layout_rejects_sizes_not_multiple_of_16():
    with pytest.raises(ValueError):
        oracle.slot_layout([32, 24])


def test_pack_places_each_tensor_and_unpack_inverts():
    g = np.random.default_rng(0)
    r, n = 3, 5
    ids = g.integers(0, 256, size=(r * n, 8)).astype(np.int32)
    w = g.standard_normal((r * n, 8)).astype(np.float32)
    pay = g.integers(0, 256, size=(r * n, 64), dtype=np.uint8)
    sc = g.integers(0, 256, size=(r * n, 16), dtype=np.uint8)
    slots = oracle.pack_slots([ids, w, pay, sc], r)
    off, sb = oracle.slot_layout([n * 32, n * 32, n * 64, n * 16])
    assert slots.shape == (r, sb)
    for q in range(r):
        rows = slice(q * n, (q + 1) * n)
        np.testing.assert_array_equal(slots[q, off[0]:off[1]].view(np.int32).reshape(n, 8), ids[rows])
        np.testing.assert_array_equal(slots[q, off[1]:off[2]].view(np.float32).reshape(n, 8), w[rows])
        np.testing.assert_array_equal(slots[q, off[2]:off[3]].reshape(n, 64), pay[rows])
        np.testing.assert_array_equal(slots[q, off[3]:].reshape(n, 16), sc[rows])
    outs = oracle.unpack_slots(slots, [n * 32, n * 32, n * 64, n * 16], r)
    np.testing.assert_array_equal(outs[0].view(np.int32).reshape(r * n, 8), ids)
    np.testing.assert_array_equal(outs[2].reshape(r * n, 64), pay)


@pytest.mark.parametrize("n_act", [0, 3, 10, 12, -1])
def test_mask_topk_ids_counts(n_act):
    ids = np.arange(40, dtype=np.int32).reshape(10, 4)
    got = oracle.mask_topk_ids(ids, n_act)
    keep = max(0, min(n_act, 10))
    np.testing.assert_array_equal(got[:keep], ids[:keep])
    assert np.all(got[keep:] == -1)
