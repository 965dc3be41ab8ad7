"""Seeded random shapes through the whole path on the GPU, checked against
the oracle: for each drawn case (tokens, top-k, experts, ranks, hidden size,
payload format, padding ids and duplicate ids) the layout and the records
equal the oracle's bit for bit, through moe_layout + moe_dispatch and through
the one-call moe_layout_dispatch, and both combine forms equal it within
|gpu - ref| <= 1e-2 * max(1, |ref|) (and bit for bit, since both sides run
the same fp32 operations in the same order).

The draws reach shapes that no hand-written case names: odd k, experts per
rank that are not powers of two, more than 32 ranks (64-bit rank masks),
layouts of one cluster block and of many, ragged hidden sizes of every
payload format."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import assert_combine_close, dev_bf16, dev_f32, dev_i32, dev_u8, host, host_bf16

pytestmark = pytest.mark.gpu

LAYOUT_KEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset",
               "rank_offset", "slot_of", "src_of_slot")
NUM_CASES = 80
KINDS = {"bf16": oracle.BF16, "fp8": oracle.FP8_E4M3_B128, "ue8m0": oracle.FP8_E4M3_UE8M0,
         "nvfp4": oracle.NVFP4_B16, "raw": oracle.RAW}


def draw(i):
    """Case i: shape, format and routing, all from one seeded generator."""
    g = np.random.default_rng(7000 + i)
    r = int(g.choice([1, 2, 3, 4, 6, 8, 12, 16, 33, 64]))
    e = r * int(g.integers(1, max(2, 1024 // r) + 1))
    k = int(g.integers(1, 13))
    n = int(g.choice([1, 2, 7, 31, 32, 33, 100, 255, 256, 257, 1000, 2047, 4096, 5000]))
    kind = str(g.choice(list(KINDS)))
    rp = rs = 0
    if kind in ("fp8", "ue8m0"):
        h = 128 * int(g.integers(1, 12))
    elif kind == "nvfp4":
        h = 16 * int(g.integers(1, 80))
    elif kind == "bf16":
        h = 8 * int(g.integers(1, 160))
    else:
        rp = 16 * int(g.integers(1, 120))
        rs = 16 * int(g.integers(0, 8))
        h = 8 * int(g.integers(1, 160))  # the combine's row width
    while n * k * h > 12_000_000 and n > 1:  # keep each case to a few seconds of oracle time
        n //= 2
    distinct = k <= e and g.random() < 0.7
    ids = np.empty((n, k), np.int32)
    for t in range(n):
        ids[t] = g.choice(e, size=k, replace=not distinct)
    pad = float(g.choice([0.0, 0.0, 0.05, 0.3]))
    if pad > 0:
        ids[g.random((n, k)) < pad] = -1
    w = g.standard_normal((n, k)).astype(np.float32)
    return dict(n=n, k=k, e=e, r=r, h=h, kind=kind, rp=rp, rs=rs, ids=ids, w=w, g=g)


@pytest.mark.parametrize("i", range(NUM_CASES))
def test_random_case(i):
    from combine_moe_layout_03_gb300 import moe
    c = draw(i)
    n, k, e, r, h, kind, rp, rs = (c[x] for x in ("n", "k", "e", "r", "h", "kind", "rp", "rs"))
    g, ids, w = c["g"], c["ids"], c["w"]
    okind = KINDS[kind]
    ikind = oracle.RAW if kind == "raw" else oracle.BF16
    if kind == "raw":
        x_host = g.integers(0, 256, size=(n, rp), dtype=np.uint8)
        x_host[:, :4] = [0, 0, 0, 0x80]  # a 0x80000000 word must survive unchanged
        sc_host = g.integers(0, 256, size=(n, rs), dtype=np.uint8) if rs else None
        x_dev, sc_dev = dev_u8(x_host), (dev_u8(sc_host) if rs else None)
    else:
        x_host = synth.bf16_normal(g, (n, h))
        sc_host, x_dev, sc_dev = None, dev_bf16(x_host), None

    ref = oracle.layout(ids, e, r)
    P = ref["num_pairs"]
    want = oracle.dispatch(ids, w, x_host, sc_host, ref["slot_of"], P, ikind, okind, h, rp, rs)

    # layout, then dispatch
    d = moe.MoeDesc(n, k, e, r, h, ikind, okind, rp, rs)
    ids_d, w_d = dev_i32(ids), dev_f32(w)
    lay = moe.moe_layout(d, ids_d)
    rec = moe.moe_dispatch(d, ids_d, w_d, x_dev, sc_dev, lay["slot_of"])
    torch.cuda.synchronize()
    assert moe.moe_layout_status(lay["workspace"]) == moe.MOE_OK
    for key in LAYOUT_KEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key],
                                      err_msg=f"case {i}: {key}")
    np.testing.assert_array_equal(host(rec)[:P], want, err_msg=f"case {i}: records")

    # the same through the one-call form
    lay2, rec2 = moe.moe_layout_dispatch(d, ids_d, w_d, x_dev, sc_dev)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(lay2["slot_of"]).reshape(ref["slot_of"].shape), ref["slot_of"],
                                  err_msg=f"case {i}: fused slot_of")
    np.testing.assert_array_equal(host(rec2)[:P], want, err_msg=f"case {i}: fused records")

    # both combine forms over expert outputs in slot order
    y = synth.bf16_normal(g, (max(P, 1), h))
    dc = moe.MoeDesc(n, k, e, r, h)
    modes = [(moe.MOE_COMBINE_TOPK, lambda: oracle.combine_topk(y, w, ref["slot_of"], h))]
    if n % r == 0:
        modes.append((moe.MOE_COMBINE_TOPK_RANKS,
                      lambda: oracle.combine_topk_ranks(y, ids, w, ref["slot_of"], e, r, h)))
    for mode, fn in modes:
        out = moe.moe_combine(dc, mode, dev_bf16(y), ids_d, w_d, lay["slot_of"])
        torch.cuda.synchronize()
        got, exp = host_bf16(out), fn()
        assert_combine_close(got, exp, f"case {i}: combine mode {mode}")
        np.testing.assert_array_equal(got, exp, err_msg=f"case {i}: combine mode {mode}")


def test_draws_reach_the_intended_shapes():
    """The seeded draws include the shapes this file exists for."""
    cases = [draw(i) for i in range(NUM_CASES)]
    assert any(c["r"] > 32 for c in cases)                       # 64-bit rank masks
    assert any((c["e"] // c["r"]) & (c["e"] // c["r"] - 1) for c in cases)  # experts per rank not 2^m
    assert any(c["k"] % 2 for c in cases)                        # odd k
    assert len({c["kind"] for c in cases}) == len(KINDS)         # every payload format
    assert any(c["n"] * c["k"] <= 256 for c in cases)            # one cluster block
    assert any(c["n"] * c["k"] > 8192 for c in cases)            # many cluster blocks
