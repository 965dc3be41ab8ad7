"""moe_layout_ranks (the routing layout and the per-rank receive layout in one
call) gives the oracle's layout and receive layout bit for bit: on the pages'
workloads and ragged shapes (the receive layout computed inside the cluster
layout launch), with more than 32 ranks (64-bit rank masks), on an empty batch,
and on a shape whose layout takes the two-kernel path (the receive layout then
runs as its own kernel). Output buffers start with stale values the call must
overwrite, and the receive slots past the last are -1."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import dev_i32, host

pytestmark = pytest.mark.gpu

LKEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset", "rank_offset",
         "slot_of", "src_of_slot")
RKEYS = ("send_head", "recv_src_idx", "recv_offset", "recv_tokens_per_expert")


def _check(ids, e, r, align):
    from combine_moe_layout_03_gb300 import moe
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, 8)
    ids_d = dev_i32(ids)
    out = moe.layout_outputs(d, ids_d.device)
    rout = moe.rank_layout_outputs(d, ids_d.device)
    for t in list(out.values()) + list(rout.values()):
        t.fill_(0x55)
    lay, rl = moe.moe_layout_ranks(d, ids_d, align, out=out, rank_out=rout)
    torch.cuda.synchronize()
    clean = ids.copy()
    clean[(clean < -1) | (clean >= e)] = -1
    ref = oracle.layout(clean, e, r)
    rref = oracle.rank_layout(ref["is_token_in_rank"], ref["tokens_per_expert"], align)
    for key in LKEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key], err_msg=key)
    for key in RKEYS:
        np.testing.assert_array_equal(host(rl[key]).reshape(rref[key].shape), rref[key], err_msg=key)
    assert moe.moe_layout_status(lay["workspace"]) == moe.MOE_OK


@pytest.mark.parametrize("case,align", [("prefill", 1), ("prefill", 128), ("skewed", 16),
                                        ("decode", 1), ("tiny", 4)])
def test_layout_ranks_pages_workloads(case, align):
    if case == "prefill":
        ids, e, r = synth.prefill_case(seed=2)["topk_idx"], 256, 8
    elif case == "skewed":
        ids, e, r = synth.skewed_case(seed=2)["topk_idx"], 256, 16
    elif case == "decode":
        ids, e, r = synth.decode_case(seed=2, n=256)["topk_idx"], 256, 8
    else:
        ids, e, r = synth.tiny_case(seed=2)["topk_idx"], 16, 2
    _check(ids, e, r, align)


@pytest.mark.parametrize("n,k,e,r", [
    (1001, 6, 96, 12),    # ragged: not a multiple of 32 tokens per block, padding ids
    (1, 8, 256, 8),       # one token, one block
    (33, 3, 64, 64),      # 64 ranks: 64-bit masks
    (4100, 8, 320, 40),   # more than 32 ranks on many blocks
    (5000, 1, 16, 16),
])
def test_layout_ranks_shapes(n, k, e, r):
    g = np.random.default_rng(n + k + r)
    ids = g.integers(-1, e, size=(n, k)).astype(np.int32)
    _check(ids, e, r, 2)


def test_layout_ranks_empty_batch():
    _check(np.zeros((0, 8), np.int32), 256, 8, 1)


def test_layout_ranks_on_the_two_kernel_path():
    # ids too many for the cluster blocks' shared memory: the layout runs as two
    # kernels and the receive layout as a third
    g = np.random.default_rng(7)
    n, k, e, r = 90000, 8, 512, 16
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    _check(ids, e, r, 8)

