"""Seeded random shapes through the one-call layouts that compute a second
layout inside the cluster launch: moe_layout_ranks (the per-rank receive
layout) and moe_layout_ll (the fixed-capacity layout). Each draw picks tokens,
top-k, experts per rank, ranks (up to 64, so 64-bit rank masks), padding ids,
duplicate ids, the expert alignment or the per-rank capacity; every output
equals the oracle's bit for bit."""
import numpy as np
import pytest
import torch

import oracle

from gpu_helpers import dev_i32, host

pytestmark = pytest.mark.gpu

NUM_CASES = 40
LKEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset", "rank_offset",
         "slot_of", "src_of_slot")


def draw(i):
    g = np.random.default_rng(9100 + i)
    r = int(g.choice([1, 2, 3, 4, 8, 12, 16, 33, 64]))
    e = r * int(g.integers(1, max(2, 512 // r) + 1))
    k = int(g.integers(1, 10))
    t_per = int(g.choice([1, 3, 16, 31, 64, 100, 128, 257, 512]))
    n = r * t_per
    ids = g.integers(-1, e, size=(n, k)).astype(np.int32)
    if g.random() < 0.5:  # distinct experts per token where possible
        ids = np.stack([g.permutation(e)[:k] if k <= e else g.integers(0, e, k) for _ in range(n)]).astype(np.int32)
        ids[g.random((n, k)) < 0.05] = -1
    return g, n, k, e, r, t_per, ids


@pytest.mark.parametrize("i", range(NUM_CASES))
def test_random_layout_ranks(i):
    from combine_moe_layout_03_gb300 import moe
    g, n, k, e, r, _, ids = draw(i)
    align = int(g.choice([1, 2, 16, 128]))
    d = moe.MoeDesc(n, k, e, r, 8)
    lay, rl = moe.moe_layout_ranks(d, dev_i32(ids), align)
    torch.cuda.synchronize()
    ref = oracle.layout(ids, e, r)
    rref = oracle.rank_layout(ref["is_token_in_rank"], ref["tokens_per_expert"], align)
    for key in LKEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key], err_msg=f"{i} {key}")
    for key in ("send_head", "recv_src_idx", "recv_offset", "recv_tokens_per_expert"):
        np.testing.assert_array_equal(host(rl[key]).reshape(rref[key].shape), rref[key], err_msg=f"{i} {key}")


@pytest.mark.parametrize("i", range(NUM_CASES))
def test_random_layout_ll(i):
    from combine_moe_layout_03_gb300 import moe
    g, n, k, e, r, t_per, ids = draw(i)
    max_t = t_per + int(g.choice([0, 0, 1, 7]))
    if e * r * max_t >= 1 << 31:
        pytest.skip("capacity beyond int32 positions")
    d = moe.MoeDesc(n, k, e, r, 8)
    lay, ll = moe.moe_layout_ll(d, max_t, dev_i32(ids))
    torch.cuda.synchronize()
    ref = oracle.layout(ids, e, r)
    lref = oracle.ll_layout(ids, e, r, max_t)
    for key in LKEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key], err_msg=f"{i} {key}")
    for key in ("ll_slot_of", "src_info", "layout_range", "recv_count"):
        np.testing.assert_array_equal(host(ll[key]).reshape(lref[key].shape), lref[key], err_msg=f"{i} {key}")
