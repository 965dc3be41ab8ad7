"""GPU parity of moe_dispatch (through the C ABI) against the oracle: records
bit-exact, byte for byte, for BF16 pass-through, raw NVFP4 bytes, FP8 e4m3
per-128 and NVFP4 per-16 quantisation; full-size workloads on sampled token
ranges; untouched slots; determinism; NVFP4 groups that fall on e2m1
midpoints; GPU records read back with the host function moe_unpack_record."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from format_cases import NVFP4_MIDPOINT_SCALES, nvfp4_midpoint_group, quantised_row
from gpu_helpers import DEV, dev_bf16, dev_f32, dev_i32, dev_u8, host

pytestmark = pytest.mark.gpu

FILL = 0xAB


def gpu_dispatch(c, e, r, in_kind, out_kind, hidden_dev, scales_dev=None, rp=0, rs=0):
    from combine_moe_layout_03_gb300 import moe
    ids = c["topk_idx"]
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, c["hidden"], in_kind, out_kind, rp, rs)
    ids_d, w_d = dev_i32(ids), dev_f32(c["topk_weights"])
    lay = moe.moe_layout(d, ids_d)
    rb = moe.moe_record_layout(d)["record_bytes"]
    rec = torch.full((n * k, rb), FILL, dtype=torch.uint8, device=DEV)
    moe.moe_dispatch(d, ids_d, w_d, hidden_dev, scales_dev, lay["slot_of"], rec)
    torch.cuda.synchronize()
    return host(rec)


def compare(c, e, r, in_kind, out_kind, hidden_host, hidden_dev, scales_host=None,
            scales_dev=None, rp=0, rs=0, ranges=None):
    ids, w = c["topk_idx"], c["topk_weights"]
    got = gpu_dispatch(c, e, r, in_kind, out_kind, hidden_dev, scales_dev, rp, rs)
    lay = oracle.layout(ids, e, r)
    P = lay["num_pairs"]
    assert np.all(got[P:] == FILL), "slots past P were written"
    if ranges is None:
        ref = oracle.dispatch(ids, w, hidden_host, scales_host, lay["slot_of"], P, in_kind,
                              out_kind, c["hidden"], rp, rs)
        np.testing.assert_array_equal(got[:P], ref)
        return got
    for t0, t1 in ranges:
        sub = slice(t0, t1)
        ref = oracle.dispatch(ids[sub], w[sub], hidden_host[sub],
                              None if scales_host is None else scales_host[sub],
                              lay["slot_of"][sub], P, in_kind, out_kind, c["hidden"], rp, rs)
        slots = lay["slot_of"][sub].ravel()
        slots = slots[slots >= 0]
        want = ref[slots].copy()
        # the oracle numbered the sub-range's tokens from 0
        hdr = want[:, :4].view(np.int32)
        hdr += t0
        np.testing.assert_array_equal(got[slots], want)
    # every record's header names a pair that maps back to its slot
    hdr = got[:P, :12].view(np.int32).reshape(P, 3)
    np.testing.assert_array_equal(lay["slot_of"][hdr[:, 0], hdr[:, 1]], np.arange(P))
    np.testing.assert_array_equal(ids[hdr[:, 0], hdr[:, 1]], hdr[:, 2])
    return got


@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_bf16(seed):
    c = synth.tiny_case(seed=seed)
    compare(c, 16, 2, oracle.BF16, oracle.BF16, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]))


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_decode_raw_bytes(n):
    c = synth.decode_case(seed=n, n=n)
    compare(c, 256, 8, oracle.RAW, oracle.RAW, c["payload"], dev_u8(c["payload"]), c["scales"],
            dev_u8(c["scales"]), 3584, 448)


def test_prefill_fp8_full_size_sampled():
    c = synth.prefill_case(seed=0)
    ranges = [(0, 24), (2040, 2056), (4072, 4096)]
    compare(c, 256, 8, oracle.BF16, oracle.FP8_E4M3_B128, c["hidden_bf16"],
            dev_bf16(c["hidden_bf16"]), ranges=ranges)


def test_fp8_small_full_compare_with_edge_values():
    c = synth.prefill_case(seed=4, n=96, hidden=1024)
    x = c["hidden_bf16"].copy()
    x[3] = 0                        # all-zero groups -> scale floor
    x[5, :128] = 0x3F80             # constant group of 1.0
    x[6, 7] = 0xC2C8                # a single large value (-100)
    x[7, :] = 0x0001                # BF16 subnormals
    c["hidden_bf16"] = x
    compare(c, 256, 8, oracle.BF16, oracle.FP8_E4M3_B128, x, dev_bf16(x))


@pytest.mark.parametrize("n,h", [(64, 7168), (40, 16), (33, 1024)])
def test_nvfp4_full_compare(n, h):
    c = synth.prefill_case(seed=n, n=n, hidden=h)
    x = c["hidden_bf16"].copy()
    x[0] = 0
    x[1, :16] = 0x3A00  # tiny values: the e4m3 scale rounds to 0 or a subnormal
    c["hidden_bf16"] = x
    compare(c, 256, 8, oracle.BF16, oracle.NVFP4_B16, x, dev_bf16(x))


def test_bf16_hidden_7168_with_padding_ids():
    c = synth.prefill_case(seed=7, n=200)
    c["topk_idx"] = c["topk_idx"].copy()
    c["topk_idx"][150:] = -1
    c["topk_idx"][3, 5] = -1
    compare(c, 256, 8, oracle.BF16, oracle.BF16, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]))


def test_odd_topk_and_raw_without_scales():
    g = np.random.default_rng(3)
    n, k, e, r = 77, 5, 40, 4
    ids = g.integers(-1, e, size=(n, k)).astype(np.int32)
    c = dict(topk_idx=ids, topk_weights=g.standard_normal((n, k)).astype(np.float32), hidden=64)
    pay = g.integers(0, 256, size=(n, 48), dtype=np.uint8)
    compare(c, e, r, oracle.RAW, oracle.RAW, pay, dev_u8(pay), None, None, 48, 0)


def test_skewed_fp8_sampled():
    c = synth.skewed_case(seed=1, n=4096)
    compare(c, 256, 16, oracle.BF16, oracle.FP8_E4M3_B128, c["hidden_bf16"],
            dev_bf16(c["hidden_bf16"]), ranges=[(0, 16), (4080, 4096)])


def test_dispatch_is_deterministic():
    c = synth.prefill_case(seed=9, n=512)
    x = dev_bf16(c["hidden_bf16"])
    a = gpu_dispatch(c, 256, 8, oracle.BF16, oracle.FP8_E4M3_B128, x)
    b = gpu_dispatch(c, 256, 8, oracle.BF16, oracle.FP8_E4M3_B128, x)
    np.testing.assert_array_equal(a, b)


def test_empty_dispatch_is_a_no_op():
    from combine_moe_layout_03_gb300 import moe
    d = moe.MoeDesc(0, 8, 256, 8, 7168, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    rec = torch.full((4, 7472), FILL, dtype=torch.uint8, device=DEV)
    e = torch.empty((0, 8), dtype=torch.int32, device=DEV)
    moe.moe_dispatch(d, e, e.float(), torch.empty((0, 7168), dtype=torch.bfloat16, device=DEV),
                     None, e, rec)
    torch.cuda.synchronize()
    assert bool((rec == FILL).all())


@pytest.mark.parametrize("scale_code", NVFP4_MIDPOINT_SCALES)
def test_nvfp4_midpoints_divide_by_the_scale(scale_code):
    """Rows made of groups whose elements divide exactly onto e2m1 midpoints
    (scale 1.875 * 2^e, an inexact reciprocal): the kernel's codes are the
    even neighbours, as IEEE division gives, and equal the oracle's."""
    grp, want = nvfp4_midpoint_group(scale_code)
    n, h = 8, 256
    g = np.random.default_rng(scale_code)
    x = np.tile(grp, (n, h // 16))
    for t in range(n):  # shuffle within groups so lanes see different positions
        for gi in range(h // 16):
            perm = g.permutation(16)
            x[t, gi * 16:(gi + 1) * 16] = grp[perm]
    c = synth.prefill_case(seed=scale_code, n=n, hidden=h)
    c["hidden_bf16"] = x
    got = compare(c, 256, 8, oracle.BF16, oracle.NVFP4_B16, x, dev_bf16(x))
    from combine_moe_layout_03_gb300 import moe
    lay = moe.moe_record_layout(moe.MoeDesc(n, 8, 256, 8, h, oracle.BF16, oracle.NVFP4_B16))
    slot_of = oracle.layout(c["topk_idx"], 256, 8)["slot_of"]
    for t in range(n):
        rec = got[slot_of[t, 0]]
        pay = rec[lay["off_payload"]:lay["off_payload"] + h // 2]
        codes = np.empty(h, np.uint8)
        codes[0::2], codes[1::2] = pay & 15, pay >> 4
        sc = rec[lay["off_scales"]:lay["off_scales"] + h // 16]
        assert np.all(sc == scale_code)
        by_value = {int(v): code for v, code in zip(grp, (want[i] for i in range(16)))}
        np.testing.assert_array_equal(codes, [by_value[int(v)] for v in x[t]])


@pytest.mark.parametrize("in_kind,out_kind,h", [
    (oracle.BF16, oracle.FP8_E4M3_B128, 7168),
    (oracle.BF16, oracle.NVFP4_B16, 1024),
    (oracle.BF16, oracle.FP8_E4M3_UE8M0, 1024),
    (oracle.BF16, oracle.BF16, 1024),
    (oracle.RAW, oracle.RAW, 0),
])
def test_unpack_gpu_records(in_kind, out_kind, h):
    """Every record moe_dispatch wrote on the GPU, split by the host function
    moe_unpack_record: header, id row, weight row, payload and scales agree
    with the routing and with the oracle's quantisation of the token's row."""
    from combine_moe_layout_03_gb300 import moe
    if in_kind == oracle.RAW:
        c = synth.decode_case(seed=31, n=48)
        x, sc, rp, rs = c["payload"], c["scales"], 3584, 448
        got = gpu_dispatch(c, 256, 8, in_kind, out_kind, dev_u8(x), dev_u8(sc), rp, rs)
    else:
        c = synth.prefill_case(seed=31, n=48, hidden=h)
        c["topk_idx"] = c["topk_idx"].copy()
        c["topk_idx"][5, 2] = -1
        x, sc, rp, rs = c["hidden_bf16"], None, 0, 0
        got = gpu_dispatch(c, 256, 8, in_kind, out_kind, dev_bf16(x))
    ids, w = c["topk_idx"], c["topk_weights"]
    n, k = ids.shape
    d = moe.MoeDesc(n, k, 256, 8, c["hidden"], in_kind, out_kind, rp, rs)
    lay = oracle.layout(ids, 256, 8)
    rows = {}
    for s in range(lay["num_pairs"]):
        u = moe.moe_unpack_record(d, got[s])
        t, j = u["src_token"], u["slot_j"]
        assert lay["slot_of"][t, j] == s and u["expert"] == ids[t, j]
        np.testing.assert_array_equal(u["ids"], ids[t])
        np.testing.assert_array_equal(u["weights"].view(np.uint32), w[t].view(np.uint32))
        if in_kind == oracle.RAW:
            pay, scl = x[t], sc[t]
        else:
            if t not in rows:
                rows[t] = quantised_row(x[t], out_kind)
            pay, scl = rows[t]
        np.testing.assert_array_equal(u["payload"], pay)
        if scl is not None:
            np.testing.assert_array_equal(u["scales"], scl)
