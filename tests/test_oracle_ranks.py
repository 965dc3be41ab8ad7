"""Pins of the oracle's per-(token, rank) layout, dispatch and combine:
numpy cumulative sums and nonzero per rank column, closed-form aligned
counts, record fields against the routing, exact sums, and agreement with the
rank-grouped pair combine on exactly representable inputs."""
import numpy as np
import torch

import oracle
from combine_moe_layout_03_gb300 import synth


def _bf16(f):
    return torch.from_numpy(np.asarray(f, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(b):
    return oracle.bf16_to_f32_array(b).astype(np.float64)


def test_rank_layout_matches_numpy():
    c = synth.prefill_case(seed=1, n=300)
    lay = oracle.layout(c["topk_idx"], 256, 8)
    m = lay["is_token_in_rank"]
    rl = oracle.rank_layout(m, lay["tokens_per_expert"], expert_alignment=16)
    counts = m.sum(0)
    np.testing.assert_array_equal(rl["recv_offset"], np.concatenate([[0], np.cumsum(counts)]))
    expect_src = np.concatenate([np.nonzero(m[:, r])[0] for r in range(8)])
    np.testing.assert_array_equal(rl["recv_src_idx"][: expect_src.size], expect_src)
    assert np.all(rl["recv_src_idx"][expect_src.size:] == -1)
    for r in range(8):
        pos = np.cumsum(m[:, r]) - 1 + rl["recv_offset"][r]
        np.testing.assert_array_equal(rl["send_head"][:, r], np.where(m[:, r] == 1, pos, -1))
    np.testing.assert_array_equal(rl["recv_tokens_per_expert"],
                                  -(-lay["tokens_per_expert"] // 16) * 16)
    # group-limited routing with one group per rank: a token reaches at most
    # its 4 chosen groups' ranks (fewer when its top-8 fall in 3 groups)
    assert np.all(m.sum(1) <= 4) and np.all(m.sum(1) >= 1)


def test_dispatch_ranks_records_follow_the_routing():
    c = synth.prefill_case(seed=2, n=24, hidden=256)
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    lay = oracle.layout(ids, 256, 8)
    rl = oracle.rank_layout(lay["is_token_in_rank"], lay["tokens_per_expert"])
    P = int(rl["recv_offset"][-1])
    rec = oracle.dispatch_ranks(ids, w, x, None, rl["send_head"], P, 256, oracle.BF16,
                                oracle.FP8_E4M3_B128, 256)
    rlay = oracle.record_layout(8, 256, oracle.BF16, oracle.FP8_E4M3_B128)
    for s in range(P):
        t, r, nloc, z = rec[s, :16].view(np.int32)
        assert rl["recv_src_idx"][s] == t and rl["send_head"][t, r] == s and z == 0
        lid = rec[s, rlay["off_ids"]:rlay["off_ids"] + 32].view(np.int32)
        lw = rec[s, rlay["off_weights"]:rlay["off_weights"] + 32].view(np.float32)
        local = ids[t] // 32 == r
        assert nloc == local.sum()
        np.testing.assert_array_equal(lid, np.where(local, ids[t] - 32 * r, -1))
        np.testing.assert_array_equal(lw, np.where(local, w[t], 0.0).astype(np.float32))
        q, sc = oracle.fp8_group(x[t, :128])
        np.testing.assert_array_equal(rec[s, rlay["off_payload"]:rlay["off_payload"] + 128], q)


def test_combine_gather_exact_and_equal_to_grouped_pair_combine():
    # Dyadic weights and small integers: every rank partial is exact in BF16,
    # so summing BF16 rank rows equals the rank-grouped pair combine.
    g = np.random.default_rng(3)
    n, k, e, r, h = 16, 4, 16, 4, 32
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    w = g.choice([0.25, 0.5, 1.0], size=(n, k)).astype(np.float32)
    lay = oracle.layout(ids, e, r)
    y = _bf16(g.integers(-4, 5, size=(lay["num_pairs"], h)))
    rl = oracle.rank_layout(lay["is_token_in_rank"], lay["tokens_per_expert"])
    P = int(rl["recv_offset"][-1])
    rows = np.zeros((P, h))
    for t in range(n):
        for j in range(k):
            rr = ids[t, j] // (e // r)
            rows[rl["send_head"][t, rr]] += float(w[t, j]) * _f(y[lay["slot_of"][t, j]])
    got = oracle.combine_gather_ranks(_bf16(rows), rl["send_head"], h)
    np.testing.assert_array_equal(got, oracle.combine_topk_ranks(y, ids, w, lay["slot_of"], e, r, h))
    exact = np.zeros((n, h))
    for t in range(n):
        for j in range(k):
            exact[t] += float(w[t, j]) * _f(y[lay["slot_of"][t, j]])
    np.testing.assert_array_equal(_f(got), exact)
