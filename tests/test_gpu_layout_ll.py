"""moe_layout_ll (the routing layout and the fixed-capacity, expert-major
layout in one call) gives the oracle's layout and fixed-capacity layout bit for
bit: on the low-latency decode workload and other shapes whose source ranks are
a whole number of cluster blocks (computed inside the cluster layout launch),
on shapes where they are not or where the layout takes two kernels (the
fixed-capacity layout then runs as its own kernel), with padding ids,
duplicate experts that overflow an expert's capacity, and an empty batch.
Outputs start with stale values the call must overwrite."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import dev_i32, host

pytestmark = pytest.mark.gpu

LKEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset", "rank_offset",
         "slot_of", "src_of_slot")
LLKEYS = ("ll_slot_of", "src_info", "layout_range", "recv_count")


def _check(ids, e, r, max_t):
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, 8)
    ids_d = dev_i32(ids)
    out = moe.layout_outputs(d, ids_d.device)
    llo = moe.ll_layout_outputs(d, max_t, ids_d.device)
    for key, t in list(out.items()) + list(llo.items()):
        if isinstance(t, torch.Tensor):
            t.fill_(0x55)
    lay, ll = moe.moe_layout_ll(d, max_t, ids_d, out=out, ll_out=llo)
    torch.cuda.synchronize()
    ref = oracle.layout(ids, e, r)
    lref = oracle.ll_layout(ids, e, r, max_t)
    for key in LKEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key], err_msg=key)
    for key in LLKEYS:
        np.testing.assert_array_equal(host(ll[key]).reshape(lref[key].shape), lref[key], err_msg=key)
    assert moe.moe_layout_status(lay["workspace"]) == moe.MOE_OK


def test_layout_ll_decode_workload():
    c = synth.decode_ll_case(seed=3)
    _check(c["topk_idx"], 256, 8, 128)


@pytest.mark.parametrize("n,k,e,r,max_t", [
    (1000, 8, 256, 8, 125),   # T = 125: blocks of 125 tokens
    (4096, 8, 256, 8, 512),   # prefill-sized
    (96, 4, 32, 4, 30),       # small, capacity above T
    (2018, 3, 64, 2, 1009),   # T = 1009 is prime: no block size fits, separate kernel
    (256, 8, 1024, 64, 4),    # 64 ranks of 4 tokens
])
def test_layout_ll_shapes(n, k, e, r, max_t):
    g = np.random.default_rng(n + k + e)
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    ids[g.random((n, k)) < 0.1] = -1  # padding pairs
    _check(ids, e, r, max_t)


def test_layout_ll_overflowing_capacity():
    # tokens that name an expert twice push it past its capacity: the extra
    # pairs get -1 and the ranges are clamped
    g = np.random.default_rng(5)
    n, k, e, r, max_t = 256, 8, 16, 4, 64
    ids = g.integers(0, e, size=(n, k)).astype(np.int32)
    ids[:, :2] = 3  # expert 3: 512 pairs for a capacity of 4 * 64
    _check(ids, e, r, max_t)


def test_layout_ll_empty_batch():
    _check(np.zeros((0, 8), np.int32), 256, 8, 4)


def test_layout_ll_on_the_two_kernel_layout():
    g = np.random.default_rng(8)
    n, k, e, r = 90000, 8, 512, 16
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    _check(ids, e, r, n // r)


@pytest.mark.parametrize("out_kind,n,hidden,r,max_t", [
    (oracle.FP8_E4M3_B128, 1024, 7168, 8, 128),   # the low-latency workload
    (oracle.NVFP4_B16, 1000, 1024, 8, 125),
    (oracle.BF16, 2018, 256, 2, 1009),            # the separate fixed-capacity kernel
])
def test_layout_ll_dispatch_one_call(out_kind, n, hidden, r, max_t):
    """Layout, fixed-capacity layout and the packed payload rows in one call, the
    dispatch building its rows while the layout runs: all equal the oracle."""
    from combine_moe_layout_03_gb300 import moe
    from gpu_helpers import dev_bf16
    e = 256
    k = 8 if n != 2018 else 3
    g = np.random.default_rng(n)
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    x = synth.bf16_normal(g, (n, hidden))
    d = moe.MoeDesc(n, k, e, r, hidden, moe.MOE_PAYLOAD_BF16, out_kind)
    ids_d = dev_i32(ids)
    out = moe.layout_outputs(d, ids_d.device)
    llo = moe.ll_layout_outputs(d, max_t, ids_d.device)
    ws = torch.empty(max(moe.moe_workspace_size(d), 256), dtype=torch.uint8, device=ids_d.device)
    lay_rec = moe.moe_record_layout(d)
    rows = e * llo["capacity"]
    pb, sbp = lay_rec["payload_bytes"], (lay_rec["scale_bytes"] + 15) // 16 * 16
    xo = torch.full((rows, pb), 0x5A, dtype=torch.uint8, device=ids_d.device)
    so = torch.full((rows, max(sbp, 16)), 0x5A, dtype=torch.uint8, device=ids_d.device) if sbp else None
    moe.prepare_layout_ll_dispatch(d, max_t, ids_d, dev_bf16(x), None, out, llo, ws, xo, so)()
    torch.cuda.synchronize()
    lref = oracle.ll_layout(ids, e, r, max_t)
    for key in LLKEYS:
        np.testing.assert_array_equal(host(llo[key]).reshape(lref[key].shape), lref[key], err_msg=key)
    ref_x, ref_s = oracle.dispatch_ll(x, None, lref["ll_slot_of"], rows, oracle.BF16, out_kind, hidden)
    so_h = lref["ll_slot_of"]
    used = np.zeros(rows, bool)
    used[so_h[so_h >= 0]] = True
    gx = host(xo)
    np.testing.assert_array_equal(gx[used], ref_x[used])
    assert (gx[~used] == 0x5A).all()
    if so is not None:
        gs = host(so)
        np.testing.assert_array_equal(gs[used], ref_s[used])
