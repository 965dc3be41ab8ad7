"""GPU parity of moe_layout (through the C ABI) against the oracle: bit-exact
counts, rank mask, offsets, slot map and inverse map on every workload shape,
ragged sizes and the degenerate cases."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_i32, host

pytestmark = pytest.mark.gpu

KEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset",
        "rank_offset", "slot_of", "src_of_slot")


def run_layout(ids, e, r, workspace=None):
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, 8)
    out = moe.moe_layout(d, dev_i32(ids), workspace=workspace)
    torch.cuda.synchronize()
    status = moe.moe_layout_status(out["workspace"])
    return {key: host(out[key]) for key in KEYS}, status


def check(ids, e, r):
    from combine_moe_layout_03_gb300 import moe
    got, status = run_layout(ids, e, r)
    ref = oracle.layout(ids, e, r)
    assert status == moe.MOE_OK
    for key in KEYS:
        np.testing.assert_array_equal(got[key].reshape(ref[key].shape), ref[key], err_msg=key)
    return got


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny(seed):
    c = synth.tiny_case(seed=seed)
    check(c["topk_idx"], 16, 2)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_decode_sweep(n):
    c = synth.decode_case(seed=n, n=n)
    check(c["topk_idx"], 256, 8)


def test_prefill_full_size():
    c = synth.prefill_case(seed=0)
    check(c["topk_idx"], 256, 8)


def test_skewed_full_size_with_empty_experts():
    c = synth.skewed_case(seed=0)
    got = check(c["topk_idx"], 256, 16)
    assert (got["tokens_per_expert"] == 0).sum() >= 8


@pytest.mark.parametrize("t", [32, 64, 128, 256, 512])
def test_rs_sizes(t):
    c = synth.rs_case(seed=t, tokens_per_rank=t, with_partials=False, with_expert_out=False)
    check(c["topk_idx"], 256, 4)


@pytest.mark.parametrize("n,k,e,r", [
    (1000, 8, 256, 8),     # ragged: not a multiple of the 128-token chunk
    (4097, 6, 96, 12),     # odd k, chunk tail of one token
    (513, 1, 1024, 64),    # largest E and R
    (700, 32, 64, 1),      # largest k, one rank
    (3000, 3, 7, 7),       # one expert per rank
    (129, 2, 2, 2),
    (600, 8, 1024, 8),     # two cluster blocks
    (512, 8, 1024, 8),     # exactly one cluster block of 4096 pairs
    (50000, 8, 256, 8),    # sixteen cluster blocks of 25000 pairs
    (20000, 8, 1024, 16),  # largest E in the cluster path
    (33000, 3, 64, 4),
    (100000, 8, 256, 8),   # ids of a cluster block exceed shared memory: two-kernel path
    (90000, 8, 512, 16),   # two-kernel path, larger E
    (4096, 1, 1, 1),       # one expert, one id a token: the pair pass is shortest here
    (4096, 1, 2, 2),
    (8192, 2, 4, 4),
    (3000, 4, 8, 2),
    (1000, 5, 128, 64),    # 64-bit rank masks, k not a multiple of 2
    (777, 3, 120, 12),     # experts per rank not a power of two
])
def test_ragged_and_extreme_shapes(n, k, e, r):
    g = np.random.default_rng(n * 31 + k)
    ids = g.integers(-1, e, size=(n, k)).astype(np.int32)
    check(ids, e, r)


def test_degenerate_cases():
    check(np.full((300, 4), -1, np.int32), 32, 4)       # all padding
    check(np.full((2000, 8), 17, np.int32), 32, 4)      # everything to one expert
    ids = np.tile(np.int32([[5, 5, 5, 1]]), (1500, 1))   # duplicate experts in a row
    check(ids, 8, 2)
    check(np.zeros((1, 1), np.int32), 1, 1)              # smallest case
    # padded tail, as vLLM's mask_topk_ids leaves it
    c = synth.prefill_case(seed=3, n=1024)
    ids = c["topk_idx"].copy()
    ids[900:] = -1
    check(ids, 256, 8)


def test_empty_input():
    from combine_moe_layout_03_gb300 import moe
    d = moe.MoeDesc(0, 8, 256, 8, 8)
    out = moe.moe_layout(d, torch.empty((0, 8), dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert host(out["tokens_per_expert"]).sum() == 0
    assert host(out["expert_offset"]).tolist() == [0] * 257
    assert host(out["rank_offset"]).tolist() == [0] * 9
    assert moe.moe_layout_status(out["workspace"]) == moe.MOE_OK


@pytest.mark.parametrize("n", [100, 3000])
def test_invalid_ids_are_reported_and_skipped(n):
    from combine_moe_layout_03_gb300 import moe
    g = np.random.default_rng(5)
    ids = g.integers(0, 64, size=(n, 4)).astype(np.int32)
    ids[7, 2] = 64
    ids[n - 1, 0] = -5
    ws = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)
    got, status = run_layout(ids, 64, 8, ws)
    assert status == moe.MOE_ERR_DEVICE_IDS
    clean = ids.copy()
    clean[(clean < -1) | (clean >= 64)] = -1
    ref = oracle.layout(clean, 64, 8)
    for key in KEYS:
        np.testing.assert_array_equal(got[key].reshape(ref[key].shape), ref[key], err_msg=key)
    # the next call on the same workspace clears the word
    c = synth.prefill_case(seed=1, n=n, e=64, groups=8, topk_groups=4, k=4)
    _, status = run_layout(c["topk_idx"], 64, 8, ws)
    assert status == moe.MOE_OK


def test_deterministic_repeat():
    c = synth.skewed_case(seed=2, n=5000)
    a, _ = run_layout(c["topk_idx"], 256, 16)
    b, _ = run_layout(c["topk_idx"], 256, 16)
    for key in KEYS:
        np.testing.assert_array_equal(a[key], b[key])


def test_without_src_of_slot():
    """src_of_slot is optional: the other outputs are the same without it."""
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=5)
    ids = c["topk_idx"]
    d = moe.MoeDesc(ids.shape[0], ids.shape[1], 256, 8, 8)
    out = moe.layout_outputs(d, DEV)
    del out["src_of_slot"]
    out = moe.moe_layout(d, dev_i32(ids), out=out)
    torch.cuda.synchronize()
    assert moe.moe_layout_status(out["workspace"]) == moe.MOE_OK
    ref = oracle.layout(ids, 256, 8)
    for key in KEYS:
        if key == "src_of_slot":
            continue
        np.testing.assert_array_equal(host(out[key]).reshape(ref[key].shape), ref[key], err_msg=key)
