"""The host record functions of the C ABI against the oracle's records.

moe_pack_record and moe_unpack_record are the library's host-side statement of
the record format (one record per (token, top-k) pair: an int4 header, the id
row, the weight row, the payload and its scales, each at a 16-byte boundary;
DeepEP repository, csrc/config.hpp LowLatencyLayout; vLLM compare view
ds-exp-2...ds-exp-ag, moe_allgather.cu "Host launcher"). Here, for every pair
of small seeded routings in every payload format, the record that
moe_pack_record builds from the pair's rows equals, byte for byte, the record
that the oracle's dispatch wrote at the pair's slot, and moe_unpack_record of
the oracle's record gives back the routing and the payload. No GPU needed."""
import numpy as np
import pytest

import oracle
from combine_moe_layout_03_gb300 import synth
from format_cases import quantised_row


@pytest.fixture(scope="module")
def moe():
    from combine_moe_layout_03_gb300 import build
    build.build_library()
    from combine_moe_layout_03_gb300 import moe as m
    return m


def _cases():
    # (name, n, k, e, r, hidden, in_kind, out_kind, raw payload bytes, raw scale bytes)
    return [
        ("tiny_bf16", 24, 2, 16, 2, 1024, oracle.BF16, oracle.BF16, 0, 0),
        ("fp8_b128", 10, 8, 256, 8, 7168, oracle.BF16, oracle.FP8_E4M3_B128, 0, 0),
        ("nvfp4_b16", 12, 8, 256, 8, 256, oracle.BF16, oracle.NVFP4_B16, 0, 0),
        ("fp8_ue8m0", 9, 5, 40, 4, 512, oracle.BF16, oracle.FP8_E4M3_UE8M0, 0, 0),
        ("decode_raw", 16, 8, 256, 8, 7168, oracle.RAW, oracle.RAW, 3584, 448),
        ("raw_no_scales_odd_k", 11, 3, 12, 3, 64, oracle.RAW, oracle.RAW, 48, 0),
    ]


def _inputs(name, n, k, e, h, in_kind, rp, rs):
    g = synth.rng_for(len(name), 11)
    ids = synth.route_uniform(g, n, e, k)
    ids[1, 0] = -1                       # a "no expert" pair gets no record
    w = synth.weights_softmax(g, n, k)
    if in_kind == oracle.RAW:
        pay = synth.raw_bytes_with_marker_words(g, n, rp)
        sc = synth.raw_bytes_with_marker_words(g, n, rs) if rs else None
        return ids, w, pay, sc
    return ids, w, synth.bf16_normal(g, (n, h)), None


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_pack_record_equals_oracle_record(moe, case):
    name, n, k, e, r, h, ik, ok, rp, rs = case
    ids, w, x, sc = _inputs(name, n, k, e, h, ik, rp, rs)
    lay = oracle.layout(ids, e, r)
    P = lay["num_pairs"]
    ref = oracle.dispatch(ids, w, x, sc, lay["slot_of"], P, ik, ok, h, rp, rs)
    d = moe.MoeDesc(n, k, e, r, h, ik, ok, rp, rs)
    assert moe.moe_record_layout(d)["record_bytes"] == ref.shape[1]
    seen = 0
    for t in range(n):
        if ik == oracle.RAW:
            pay, scl = x[t], (None if sc is None else sc[t])
        else:
            pay, scl = quantised_row(x[t], ok)
        for j in range(k):
            s = int(lay["slot_of"][t, j])
            if s < 0:
                assert ids[t, j] < 0
                continue
            rec = moe.moe_pack_record(d, t, j, int(ids[t, j]), ids[t], w[t], pay, scl)
            np.testing.assert_array_equal(rec, ref[s], err_msg=f"{name}: pair ({t}, {j}) slot {s}")
            seen += 1
    assert seen == P


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_unpack_record_of_oracle_records(moe, case):
    name, n, k, e, r, h, ik, ok, rp, rs = case
    ids, w, x, sc = _inputs(name, n, k, e, h, ik, rp, rs)
    lay = oracle.layout(ids, e, r)
    P = lay["num_pairs"]
    ref = oracle.dispatch(ids, w, x, sc, lay["slot_of"], P, ik, ok, h, rp, rs)
    d = moe.MoeDesc(n, k, e, r, h, ik, ok, rp, rs)
    for s in range(P):
        u = moe.moe_unpack_record(d, ref[s])
        t, j = u["src_token"], u["slot_j"]
        assert 0 <= t < n and 0 <= j < k
        assert lay["slot_of"][t, j] == s
        assert u["expert"] == ids[t, j]
        np.testing.assert_array_equal(u["ids"], ids[t])
        np.testing.assert_array_equal(u["weights"].view(np.uint32), w[t].view(np.uint32))
        if ik == oracle.RAW:
            np.testing.assert_array_equal(u["payload"], x[t])
            if sc is not None:
                np.testing.assert_array_equal(u["scales"], sc[t])
        else:
            pay, scl = quantised_row(x[t], ok)
            np.testing.assert_array_equal(u["payload"], pay)
            if scl is not None:
                np.testing.assert_array_equal(u["scales"], scl)
