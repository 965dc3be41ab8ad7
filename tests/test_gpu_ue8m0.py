"""GPU parity of FP8 e4m3 with power-of-two UE8M0 scales against the oracle,
bit for bit, in every dispatch path: per-pair records (full prefill shape,
sampled; edge values), the fused layout + dispatch, per-(token, rank)
records, and the fixed-capacity packed rows (56-byte scale rows padded to
64)."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_bf16, dev_f32, dev_i32, host
from test_gpu_fused import _check as _check_fused
from test_gpu_ranks import _check_dispatch_ranks

pytestmark = pytest.mark.gpu
UE = oracle.FP8_E4M3_UE8M0


def _records(c, e, r):
    from combine_moe_layout_03_gb300 import moe
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, c["hidden"], oracle.BF16, UE)
    rb = moe.moe_record_layout(d)["record_bytes"]
    rec = torch.full((n * k + 2, rb), 0xAB, dtype=torch.uint8, device=DEV)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    moe.moe_dispatch(d, ids_d, dev_f32(w), dev_bf16(x), None, lay["slot_of"], rec)
    torch.cuda.synchronize()
    return host(rec)


def test_prefill_records_sampled():
    c = synth.prefill_case(seed=100)
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    got = _records(c, 256, 8)
    lay = oracle.layout(ids, 256, 8)
    P = lay["num_pairs"]
    assert np.all(got[P:] == 0xAB)
    for t0, t1 in [(0, 16), (2048, 2064), (4080, 4096)]:
        sub = slice(t0, t1)
        want = oracle.dispatch(ids[sub], w[sub], x[sub], None, lay["slot_of"][sub], P, oracle.BF16, UE,
                               c["hidden"])
        slots = lay["slot_of"][sub].ravel()
        slots = slots[slots >= 0]
        rows = want[slots].copy()
        rows[:, :4].view(np.int32)[:] += t0  # the oracle numbered the sub-range from 0
        np.testing.assert_array_equal(got[slots], rows)


def test_edge_values_full_compare():
    c = synth.prefill_case(seed=101, n=48, hidden=1024)
    x = c["hidden_bf16"].copy()
    x[0] = 0                    # all zero: the 1e-4 floor decides the exponent
    x[1, :128] = 0x43E0         # 448: amax/448 is a power of two and keeps its exponent
    x[2, 5] = 0x7F7F            # the largest BF16 value
    x[3, :] = 0x0001            # BF16 subnormals
    x[4, :128] = 0x3F81         # just above 1.0
    x[5, 256:384] = 0x8000      # negative zero
    c["hidden_bf16"] = x
    got = _records(c, 256, 8)
    lay = oracle.layout(c["topk_idx"], 256, 8)
    P = lay["num_pairs"]
    want = oracle.dispatch(c["topk_idx"], c["topk_weights"], x, None, lay["slot_of"], P, oracle.BF16, UE,
                           1024)
    np.testing.assert_array_equal(got[:P], want)


def test_fused_prefill_sampled():
    c = synth.prefill_case(seed=102)
    _check_fused(c, 256, 8, oracle.BF16, UE, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]),
                 sample=[(0, 32), (4064, 4096)])


def test_fused_ragged():
    c = synth.prefill_case(seed=103, n=77, hidden=1536, e=48, k=6, r=6, groups=6, topk_groups=3)
    _check_fused(c, 48, 6, oracle.BF16, UE, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]))


def test_rank_records():
    c = synth.prefill_case(seed=104, n=200, hidden=2048)
    _check_dispatch_ranks(c, 256, 8, oracle.BF16, UE, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]))


@pytest.mark.parametrize("n,hidden,r,max_t", [(128, 7168, 8, 16), (96, 1536, 4, 30)])
def test_fixed_capacity_rows_with_padded_scales(n, hidden, r, max_t):
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=105, n=n, hidden=hidden)
    ids, x = c["topk_idx"], c["hidden_bf16"]
    e, k = 256, 8
    d = moe.MoeDesc(n, k, e, r, hidden, oracle.BF16, UE)
    ids_d = dev_i32(ids)
    lay = moe.moe_layout(d, ids_d)
    ll = moe.moe_ll_layout(d, max_t, ids_d, lay)
    xo, so = moe.moe_dispatch_ll(d, dev_bf16(x), None, ll["ll_slot_of"], ll["capacity"])
    torch.cuda.synchronize()
    assert so.shape[1] == (hidden // 128 + 15) // 16 * 16  # 56 -> 64, 12 -> 16
    so_h = oracle.ll_layout(ids, e, r, max_t)["ll_slot_of"]
    np.testing.assert_array_equal(host(ll["ll_slot_of"]), so_h)
    ref_x, ref_s = oracle.dispatch_ll(x, None, so_h, e * ll["capacity"], oracle.BF16, UE, hidden)
    pos = so_h[so_h >= 0]
    idx = torch.from_numpy(pos.astype(np.int64)).to(DEV)
    np.testing.assert_array_equal(host(xo.index_select(0, idx)), ref_x[pos])
    np.testing.assert_array_equal(host(so.index_select(0, idx)), ref_s[pos])
