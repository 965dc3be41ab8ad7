"""moe_layout_noalloc, the routing layout for callers that cannot allocate.

Some callers of this library cannot give it device scratch memory: a plugin
inside a host program that owns every device allocation through its own pool
and forbids direct cudaMalloc, or a service that fixes its device footprint at
start-up. moe_layout_noalloc serves them with a fixed scratch array inside the
library's device image instead of a caller workspace.

These tests call it through the C ABI (ctypes, no binding helper) twice in a
row on different inputs -- so the second call runs on scratch the first one
left behind -- and compare every output with the existing moe_layout's,
exactly, since all layout outputs are integers. The file is named to be
collected last; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_moe_layout_03_gb300 import synth

pytestmark = pytest.mark.gpu

KEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset",
        "rank_offset", "slot_of", "src_of_slot")


def _noalloc(moe, desc, ids):
    out = moe.layout_outputs(desc, ids.device)
    for t in out.values():
        t.fill_(0x55)  # stale values the call must overwrite
    status = torch.full((1,), 12345, dtype=torch.int32, device=ids.device)
    rc = moe._lib.moe_layout_noalloc(
        ctypes.byref(desc.c()), ids.data_ptr(), out["tokens_per_expert"].data_ptr(),
        out["tokens_per_rank"].data_ptr(), out["is_token_in_rank"].data_ptr(),
        out["expert_offset"].data_ptr(), out["rank_offset"].data_ptr(), out["slot_of"].data_ptr(),
        out["src_of_slot"].data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == moe.MOE_OK, moe.moe_strerror(rc)
    return out, status


def _compare(moe, desc, ids):
    got, status = _noalloc(moe, desc, ids)
    ref = moe.moe_layout(desc, ids)  # the existing entry point, with its own workspace
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(got[key], ref[key]), key
    return int(status.item()), int(moe.moe_layout_status(ref["workspace"]))


def test_noalloc_matches_moe_layout_on_two_calls_in_a_row():
    from combine_moe_layout_03_gb300 import moe
    dev = torch.device("cuda:0")
    # Two calls in a row on shapes large enough for the layout to keep
    # per-chunk counts in scratch (the two-kernel path): the second call runs
    # on the scratch the first one left behind, with fewer chunks and other E.
    g = np.random.default_rng(12)
    ids1 = synth.route_uniform(g, 100000, 256, 8)
    st, ref_st = _compare(moe, moe.MoeDesc(100000, 8, 256, 8, 8), torch.from_numpy(ids1).to(dev))
    assert st == ref_st == moe.MOE_OK
    ids2 = g.integers(-1, 512, size=(90000, 8)).astype(np.int32)
    st, ref_st = _compare(moe, moe.MoeDesc(90000, 8, 512, 16, 8), torch.from_numpy(ids2).to(dev))
    assert st == ref_st == moe.MOE_OK


def test_noalloc_matches_moe_layout_on_the_pages_workloads():
    from combine_moe_layout_03_gb300 import moe
    dev = torch.device("cuda:0")
    c = synth.prefill_case(seed=11)
    st, ref_st = _compare(moe, moe.MoeDesc(4096, 8, 256, 8, 7168),
                          torch.from_numpy(c["topk_idx"]).to(dev))
    assert st == ref_st == moe.MOE_OK
    c = synth.skewed_case(seed=4)
    st, ref_st = _compare(moe, moe.MoeDesc(16384, 8, 256, 16, 7168),
                          torch.from_numpy(c["topk_idx"]).to(dev))
    assert st == ref_st == moe.MOE_OK


def test_noalloc_status_and_small_path():
    from combine_moe_layout_03_gb300 import moe
    dev = torch.device("cuda:0")
    ids = synth.decode_case(seed=3, n=64)["topk_idx"].copy()
    ids[5, 1] = 300  # outside [-1, E): reported, treated as -1
    st, ref_st = _compare(moe, moe.MoeDesc(64, 8, 256, 8, 8), torch.from_numpy(ids).to(dev))
    assert st == ref_st == moe.MOE_ERR_DEVICE_IDS
    ids[5, 1] = 7
    st, ref_st = _compare(moe, moe.MoeDesc(64, 8, 256, 8, 8), torch.from_numpy(ids).to(dev))
    assert st == ref_st == moe.MOE_OK


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from combine_moe_layout_03_gb300 import moe
    n = 300_000  # needs about 2.4 MiB of scratch at E=256, R=8
    desc = moe.MoeDesc(n, 8, 256, 8, 8)
    assert moe.moe_workspace_size(desc) > moe.MOE_NOALLOC_SCRATCH_BYTES
    rc = moe._lib.moe_layout_noalloc(ctypes.byref(desc.c()), 16, 16, 16, 16, 16, 16, 16, None,
                                     None, None)
    assert rc == moe.MOE_ERR_TOO_LARGE
    ok = moe.MoeDesc(250_000, 8, 256, 8, 8)
    assert moe.moe_workspace_size(ok) <= moe.MOE_NOALLOC_SCRATCH_BYTES


def test_noalloc_python_wrapper_with_and_without_status():
    """The binding's moe_layout_noalloc marshals the same call: with a status
    tensor and without one, its outputs equal moe_layout's."""
    from combine_moe_layout_03_gb300 import moe
    dev = torch.device("cuda:0")
    c = synth.decode_case(seed=21, n=256)
    ids = torch.from_numpy(c["topk_idx"]).to(dev)
    desc = moe.MoeDesc(256, 8, 256, 8, 8)
    ref = moe.moe_layout(desc, ids)
    status = torch.full((1,), 777, dtype=torch.int32, device=dev)
    a = moe.moe_layout_noalloc(desc, ids, status=status)
    b = moe.moe_layout_noalloc(desc, ids)
    torch.cuda.synchronize()
    for key in KEYS:
        assert torch.equal(a[key], ref[key]), key
        assert torch.equal(b[key], ref[key]), key
    assert int(status.item()) == moe.MOE_OK


def test_noalloc_at_the_largest_shape_its_scratch_holds():
    """The largest N (E=256, R=8) whose scratch fits the fixed array runs and
    matches moe_layout exactly; one more token is rejected before any launch."""
    from combine_moe_layout_03_gb300 import moe
    dev = torch.device("cuda:0")
    lo, hi = 1, 1 << 20
    while lo < hi:  # the largest N with moe_workspace_size <= the array
        mid = (lo + hi + 1) // 2
        if moe.moe_workspace_size(moe.MoeDesc(mid, 8, 256, 8, 8)) <= moe.MOE_NOALLOC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    n = lo
    assert 250_000 <= n < 260_000
    g = np.random.default_rng(99)
    ids = g.integers(-1, 256, size=(n, 8)).astype(np.int32)
    ids[g.random((n, 8)) < 0.25] = -1  # a sparse routing: about a quarter of the pairs empty
    st, ref_st = _compare(moe, moe.MoeDesc(n, 8, 256, 8, 8), torch.from_numpy(ids).to(dev))
    assert st == ref_st == moe.MOE_OK
    over = moe.MoeDesc(n + 1, 8, 256, 8, 8)
    rc = moe._lib.moe_layout_noalloc(ctypes.byref(over.c()), 16, 16, 16, 16, 16, 16, 16, None,
                                     None, None)
    assert rc == moe.MOE_ERR_TOO_LARGE
