"""Whole steps captured once in a CUDA graph (with the programmatic-dependent
launch edges the library's kernels carry) and replayed on new inputs copied
into the captured buffers: each replay matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_bf16, host, host_bf16

pytestmark = pytest.mark.gpu


def _capture(calls):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in calls:  # warm up outside the capture
            c(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            c(s)
    return g


def test_layout_dispatch_combine_graph_replays_on_new_inputs():
    from combine_moe_layout_03_gb300 import moe
    n, k, e, r, h = 512, 8, 256, 8, 1024
    d = moe.MoeDesc(n, k, e, r, h, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    cd = moe.MoeDesc(n, k, e, r, h)
    ids = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    x = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((n * k, h), dtype=torch.bfloat16, device=DEV)
    lay = moe.layout_outputs(d, DEV)
    ws = torch.empty(max(moe.moe_workspace_size(d), 256), dtype=torch.uint8, device=DEV)
    rec = torch.empty((n * k, moe.moe_record_layout(d)["record_bytes"]), dtype=torch.uint8, device=DEV)
    out = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)

    def fill(seed):
        c = synth.prefill_case(seed=seed, n=n, hidden=h)
        ids.copy_(torch.from_numpy(c["topk_idx"]))
        w.copy_(torch.from_numpy(c["topk_weights"]))
        x.copy_(dev_bf16(c["hidden_bf16"]))
        yy = synth.bf16_normal(np.random.default_rng(seed + 100), (n * k, h))
        y.copy_(dev_bf16(yy))
        return c, yy

    fill(0)
    calls = [
        lambda s: moe.prepare_layout(d, ids, lay, ws, s.cuda_stream)(),
        lambda s: moe.prepare_dispatch(d, ids, w, x, None, lay["slot_of"], rec, s.cuda_stream)(),
        lambda s: moe.prepare_combine(cd, moe.MOE_COMBINE_TOPK_RANKS, y, ids, w, lay["slot_of"], out,
                                      s.cuda_stream)(),
    ]
    g = _capture(calls)
    for seed in (1, 2, 3):
        c, yy = fill(seed)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.layout(c["topk_idx"], e, r)
        np.testing.assert_array_equal(host(lay["slot_of"]), ref["slot_of"])
        P = ref["num_pairs"]
        want = oracle.dispatch(c["topk_idx"], c["topk_weights"], c["hidden_bf16"], None, ref["slot_of"], P,
                               oracle.BF16, oracle.FP8_E4M3_B128, h)
        np.testing.assert_array_equal(host(rec)[:P], want)
        np.testing.assert_array_equal(
            host_bf16(out), oracle.combine_topk_ranks(yy, c["topk_idx"], c["topk_weights"], ref["slot_of"],
                                                      e, r, h))


def test_fixed_capacity_forward_and_backward_graph():
    # layout, fixed-capacity layout, BF16 packed dispatch, top-k combine, then
    # combine backward and dispatch backward: one graph, replayed twice
    from combine_moe_layout_03_gb300 import moe
    r, t_per, k, e, h = 4, 32, 4, 32, 512
    n = r * t_per
    d = moe.MoeDesc(n, k, e, r, h, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_BF16)
    cd = moe.MoeDesc(n, k, e, r, h)
    cap = r * t_per
    rows = e * cap
    ids = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    x = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    go = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    lay = moe.layout_outputs(d, DEV)
    ws = torch.empty(max(moe.moe_workspace_size(d), 256), dtype=torch.uint8, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    ll = dict(ll_slot_of=torch.empty((n, k), **i32), src_info=torch.empty((e, cap), **i32),
              layout_range=torch.empty((e, r), dtype=torch.int64, device=DEV),
              recv_count=torch.empty(e, **i32))
    xo = torch.zeros((rows, 2 * h), dtype=torch.uint8, device=DEV)
    y = xo.view(torch.bfloat16)  # identity expert
    out = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    gy = torch.zeros((rows, h), dtype=torch.bfloat16, device=DEV)
    gw = torch.empty((n, k), dtype=torch.float32, device=DEV)
    gx = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)

    def fill(seed):
        c = synth.decode_ll_case(seed=seed, tokens_per_rank=t_per, r=r, hidden=h, e=e, k=k)
        ids.copy_(torch.from_numpy(c["topk_idx"]))
        w.copy_(torch.from_numpy(c["topk_weights"]))
        x.copy_(dev_bf16(c["hidden_bf16"]))
        gg = synth.bf16_normal(np.random.default_rng(seed + 7), (n, h))
        go.copy_(dev_bf16(gg))
        return c, gg

    fill(10)
    calls = [
        lambda s: moe.prepare_layout(d, ids, lay, ws, s.cuda_stream)(),
        lambda s: moe.prepare_ll_layout(d, t_per, ids, lay, ll, s.cuda_stream)(),
        lambda s: moe.prepare_dispatch_ll(d, x, None, ll["ll_slot_of"], xo, None, s.cuda_stream)(),
        lambda s: moe.prepare_combine(cd, moe.MOE_COMBINE_TOPK, y, ids, w, ll["ll_slot_of"], out,
                                      s.cuda_stream)(),
        lambda s: moe.prepare_combine_backward(cd, go, w, ll["ll_slot_of"], y, rows, gy, gw,
                                               s.cuda_stream)(),
        lambda s: moe.prepare_dispatch_backward(cd, gy, ll["ll_slot_of"], gx, s.cuda_stream)(),
    ]
    g = _capture(calls)
    for seed in (11, 12):
        c, gg = fill(seed)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        so = oracle.ll_layout(c["topk_idx"], e, r, t_per)["ll_slot_of"]
        np.testing.assert_array_equal(host(ll["ll_slot_of"]), so)
        y_ref, _ = oracle.dispatch_ll(c["hidden_bf16"], None, so, rows, oracle.BF16, oracle.BF16, h)
        y_ref = y_ref.view(np.uint16)
        pos = so[so >= 0]
        np.testing.assert_array_equal(host_bf16(y)[pos], y_ref[pos])
        np.testing.assert_array_equal(host_bf16(out), oracle.combine_topk(y_ref, c["topk_weights"], so, h))
        ref_gy, _ = oracle.combine_backward(gg, c["topk_weights"], so, y_ref, rows, h)
        np.testing.assert_array_equal(host_bf16(gy)[pos], ref_gy[pos])
        np.testing.assert_array_equal(host_bf16(gx), oracle.dispatch_backward(ref_gy, so, h))


def test_pipelined_combine_graph_replays_on_new_inputs():
    # 4 ranks x 64 tokens of hidden 8192, top-8 of 256 grouped by rank: the
    # shape moe_combine sends to its pipelined kernel (bulk copies into
    # shared-memory stages); layout + combine captured once, replayed twice
    from combine_moe_layout_03_gb300 import moe
    r, t_per, k, e, h = 4, 64, 8, 256, 8192
    n = r * t_per
    d = moe.MoeDesc(n, k, e, r, h)
    ids = torch.empty((n, k), dtype=torch.int32, device=DEV)
    w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    y = torch.empty((n * k, h), dtype=torch.bfloat16, device=DEV)
    lay = moe.layout_outputs(d, DEV)
    ws = torch.empty(max(moe.moe_workspace_size(d), 256), dtype=torch.uint8, device=DEV)
    out = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)

    def fill(seed):
        c = synth.rs_case(seed=seed, tokens_per_rank=t_per, hidden=h, r=r, e=e, k=k, with_partials=False)
        ids.copy_(torch.from_numpy(c["topk_idx"]))
        w.copy_(torch.from_numpy(c["topk_weights"]))
        y.copy_(dev_bf16(c["expert_out_bf16"]))
        return c

    fill(20)
    calls = [
        lambda s: moe.prepare_layout(d, ids, lay, ws, s.cuda_stream)(),
        lambda s: moe.prepare_combine(d, moe.MOE_COMBINE_TOPK_RANKS, y, ids, w, lay["slot_of"], out,
                                      s.cuda_stream)(),
    ]
    g = _capture(calls)
    for seed in (21, 22):
        c = fill(seed)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.layout(c["topk_idx"], e, r)
        np.testing.assert_array_equal(host(lay["slot_of"]), ref["slot_of"])
        np.testing.assert_array_equal(
            host_bf16(out), oracle.combine_topk_ranks(c["expert_out_bf16"], c["topk_idx"], c["topk_weights"],
                                                      ref["slot_of"], e, r, h))
    assert moe.moe_device_status(clear=False) == moe.MOE_OK
