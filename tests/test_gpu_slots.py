"""GPU parity of the rank-slot packing and the padded-token mask (through the
C ABI) against the oracle: bytes exact; the mask replayed in a CUDA graph
follows the device-side token count."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_i32, host

pytestmark = pytest.mark.gpu


def _decode_tensors(seed, r, n):
    c = synth.decode_case(seed=seed, n=r * n)
    return [c["topk_idx"], c["topk_weights"], c["payload"], c["scales"]]


@pytest.mark.parametrize("n", [1, 4, 32])
def test_pack_unpack_decode_payload(n):
    from combine_moe_layout_03_gb300 import moe
    r = 8
    ts = _decode_tensors(n, r, n)
    dev_ts = [torch.from_numpy(np.ascontiguousarray(t)).to(DEV) for t in ts]
    slots = moe.moe_pack_slots(dev_ts, r)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(slots), oracle.pack_slots(ts, r))
    outs = [torch.empty_like(t) for t in dev_ts]
    moe.moe_unpack_slots(slots, outs, r)
    torch.cuda.synchronize()
    for t, o in zip(ts, outs):
        np.testing.assert_array_equal(host(o), t)


def test_pack_unpack_odd_sizes_and_empty_tensor():
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(3)
    r = 5
    ts = [g.integers(0, 256, size=r * b, dtype=np.uint8) for b in (48, 0, 4096 + 16)]
    dev_ts = [torch.from_numpy(t).to(DEV) for t in ts]
    slots = moe.moe_pack_slots(dev_ts, r)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(slots), oracle.pack_slots(ts, r))
    outs = [torch.zeros_like(t) for t in dev_ts]
    moe.moe_unpack_slots(slots, outs, r)
    torch.cuda.synchronize()
    for t, o in zip(ts, outs):
        np.testing.assert_array_equal(host(o), t)


@pytest.mark.parametrize("n_act", [0, 17, 255, 256, 1000, -4])
def test_mask_topk_ids(n_act):
    from combine_moe_layout_03_gb300 import moe
    ids = synth.decode_case(seed=1, n=256)["topk_idx"]
    d = dev_i32(ids)
    moe.moe_mask_topk_ids(d, torch.tensor([n_act], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(d), oracle.mask_topk_ids(ids, n_act))


def test_mask_topk_ids_in_a_replayed_graph():
    """The count lives on the device, so one captured graph serves any count."""
    from combine_moe_layout_03_gb300 import moe
    ids = synth.decode_case(seed=2, n=128)["topk_idx"]
    src = dev_i32(ids)
    work = src.clone()
    n_act = torch.tensor([128], dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        moe.moe_mask_topk_ids(work, n_act, stream=s)  # first call outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_mask_topk_ids(work, n_act)
    for count in (100, 7, 128, 0):
        work.copy_(src)
        n_act.fill_(count)
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(work), oracle.mask_topk_ids(ids, count))
