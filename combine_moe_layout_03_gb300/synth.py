"""Seeded synthetic inputs for MoE dispatch and combine.

This module is shared by the CUDA path's callers (tests, bench) and by the
oracle's callers. It only draws inputs: routing ids and weights, BF16 hidden
rows, raw byte payloads and expert outputs. None of the method's arithmetic
(layout, packing, quantisation, weighted reduction, rank sum, BF16 rounding)
lives here. BF16 values are made by truncating fp32 draws to their top 16
bits, so no rounding rule is shared with either side.

Every function takes a seed and returns numpy arrays on the host. The shapes
and distributions follow the workloads of the pages:

* tiny        N=128, H=1024 BF16 ~N(0,1), E=16, top-2 distinct uniform experts,
              softmax(N(0,1)) weights, R=2.
* decode      N in {1..256}, top-8 of 256 distinct uniform int32 ids,
              |N(0,1)| fp32 weights, an opaque 3584-byte NVFP4 payload plus
              448 e4m3 scale bytes per token (vLLM ds-exp-ag compare view,
              bench_moe_allgather.py: per-token payload of the decode sweep), R=8.
* prefill     N=4096, H=7168 BF16 ~N(0,1), 256 experts in 8 groups,
              sigmoid(N(0,1)) scores, top-4 groups then top-8 experts
              (DeepEP README, performance table setting), R=8.
* rs          BF16 H=8192 ~N(0,1), R=4, 32..512 tokens per rank (vLLM PR
              "Eliminate staging from NCCL symmetric reduce-scatter",
              reduce-scatter latency table), top-8 of 256.
* decode_ll   R=8 ranks x 128 tokens, H=7168 BF16 ~N(0,1), top-8 of 256
              distinct uniform ids, |N(0,1)| weights (DeepEP README,
              "Low-latency kernels with pure RDMA": 128 tokens per batch,
              7168 hidden, top-8, FP8 dispatching and BF16 combining).
* skewed      N=16384, H=7168, 256 experts with Zipf(s=1.2) popularity, top-8
              distinct, R=16, with a few experts of zero popularity so that
              empty experts occur.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng_for",
    "bf16_normal",
    "route_uniform",
    "route_grouped",
    "route_zipf",
    "weights_softmax",
    "weights_abs_normal",
    "raw_bytes_with_marker_words",
    "tiny_case",
    "decode_case",
    "prefill_case",
    "rs_case",
    "skewed_case",
    "decode_ll_case",
    "PAGE_SENTINEL_WORD",
]

# The 32-bit word the Lamport all-gather on the vLLM ds-exp-ag page uses as
# its "not yet written" marker. Payload bytes that contain it must still
# travel through dispatch unchanged, so the decode inputs plant it on purpose.
PAGE_SENTINEL_WORD = 0x80000000


def rng_for(seed: int, stream: int = 0) -> np.random.Generator:
    """A PCG64 generator keyed by (seed, stream)."""
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def bf16_normal(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """BF16 bit patterns (uint16) of N(0, scale^2) draws, truncated from fp32."""
    f = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        f = f * np.float32(scale)
    return (np.ascontiguousarray(f).view(np.uint32) >> 16).astype(np.uint16)


def route_uniform(rng: np.random.Generator, n: int, e: int, k: int) -> np.ndarray:
    """k distinct experts per token, uniform over [0, e); int32 [n, k]."""
    if n == 0:
        return np.zeros((0, k), dtype=np.int32)
    keys = rng.random((n, e), dtype=np.float32)
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def route_grouped(rng: np.random.Generator, n: int, e: int = 256, groups: int = 8,
                  topk_groups: int = 4, k: int = 8):
    """Group-limited routing: sigmoid(N(0,1)) scores, top groups by their max
    score, then the top-k experts inside the chosen groups.

    Returns (topk_idx int32 [n, k], topk_weights fp32 [n, k]); weights are the
    chosen scores divided by their sum. Ties go to the lower index.
    """
    z = rng.standard_normal((n, e), dtype=np.float32).astype(np.float64)
    scores = 1.0 / (1.0 + np.exp(-z))
    per = e // groups
    gscore = scores.reshape(n, groups, per).max(axis=2)
    gsel = np.argsort(-gscore, axis=1, kind="stable")[:, :topk_groups]
    in_sel = np.zeros((n, groups), dtype=bool)
    np.put_along_axis(in_sel, gsel, True, axis=1)
    expert_ok = np.repeat(in_sel, per, axis=1)
    masked = np.where(expert_ok, scores, -1.0)
    idx = np.argsort(-masked, axis=1, kind="stable")[:, :k]
    chosen = np.take_along_axis(scores, idx, axis=1)
    w = chosen / chosen.sum(axis=1, keepdims=True)
    return idx.astype(np.int32), w.astype(np.float32)


def route_zipf(rng: np.random.Generator, n: int, e: int = 256, k: int = 8,
               s: float = 1.2, num_zero: int = 8) -> np.ndarray:
    """k distinct experts per token drawn without replacement with Zipf(s)
    popularity p(x) ~ 1/(pi(x)+1)^s over a seeded permutation pi.

    The num_zero experts with the largest pi get popularity 0, so they are
    never chosen (empty experts). Gumbel-top-k sampling.
    """
    pi = rng.permutation(e)
    logp = -s * np.log(pi.astype(np.float64) + 1.0)
    logp[pi >= e - num_zero] = -np.inf
    u = rng.random((n, e))
    g = -np.log(-np.log(np.clip(u, 1e-300, 1.0 - 1e-16)))
    keys = logp[None, :] + g
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def weights_softmax(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    """softmax of N(0,1) logits per row; fp32 [n, k]."""
    z = rng.standard_normal((n, k)).astype(np.float64)
    z = np.exp(z - z.max(axis=1, keepdims=True)) if n else z
    w = z / z.sum(axis=1, keepdims=True) if n else z
    return w.astype(np.float32)


def weights_abs_normal(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    """|N(0,1)| fp32 [n, k], as the decode benchmark draws them."""
    return np.abs(rng.standard_normal((n, k), dtype=np.float32))


def raw_bytes_with_marker_words(rng: np.random.Generator, n: int, nbytes: int,
                                marker_frac: float = 0.01) -> np.ndarray:
    """Uniform random bytes uint8 [n, nbytes] with about marker_frac of the
    aligned 32-bit words set to PAGE_SENTINEL_WORD (little-endian)."""
    b = rng.integers(0, 256, size=(n, nbytes), dtype=np.uint8)
    if n and nbytes >= 4:
        words = b[:, : (nbytes // 4) * 4].view(np.uint32)
        hit = rng.random(words.shape) < marker_frac
        words[hit] = np.uint32(PAGE_SENTINEL_WORD)
    return b


# ---------------------------------------------------------------------------
# Whole workloads. Each returns a dict of numpy arrays plus the shape scalars.
# ---------------------------------------------------------------------------

def tiny_case(seed: int = 0, n: int = 128, hidden: int = 1024, e: int = 16,
              k: int = 2, r: int = 2) -> dict:
    g = rng_for(seed, 1)
    return dict(
        name="tiny", num_tokens=n, hidden=hidden, num_experts=e, topk=k, num_ranks=r,
        topk_idx=route_uniform(g, n, e, k),
        topk_weights=weights_softmax(g, n, k),
        hidden_bf16=bf16_normal(g, (n, hidden)),
    )


def decode_case(seed: int = 0, n: int = 256, e: int = 256, k: int = 8, r: int = 8,
                payload_bytes: int = 3584, scale_bytes: int = 448) -> dict:
    g = rng_for(seed, 2)
    return dict(
        name="decode", num_tokens=n, hidden=2 * payload_bytes, num_experts=e, topk=k,
        num_ranks=r, raw_payload_bytes=payload_bytes, raw_scale_bytes=scale_bytes,
        topk_idx=route_uniform(g, n, e, k),
        topk_weights=weights_abs_normal(g, n, k),
        payload=raw_bytes_with_marker_words(g, n, payload_bytes),
        scales=raw_bytes_with_marker_words(g, n, scale_bytes),
    )


def prefill_case(seed: int = 0, n: int = 4096, hidden: int = 7168, e: int = 256,
                 k: int = 8, r: int = 8, groups: int = 8, topk_groups: int = 4) -> dict:
    g = rng_for(seed, 3)
    idx, w = route_grouped(g, n, e, groups, topk_groups, k)
    return dict(
        name="prefill", num_tokens=n, hidden=hidden, num_experts=e, topk=k, num_ranks=r,
        topk_idx=idx, topk_weights=w, hidden_bf16=bf16_normal(g, (n, hidden)),
    )


def rs_case(seed: int = 0, tokens_per_rank: int = 32, hidden: int = 8192, r: int = 4,
            e: int = 256, k: int = 8, with_partials: bool = True,
            with_expert_out: bool = True) -> dict:
    """Combine / reduce-scatter workload. Per-rank output is
    tokens_per_rank * hidden * 2 bytes (32 tokens -> 0.5 MiB at H=8192)."""
    g = rng_for(seed, 4)
    n = r * tokens_per_rank
    out = dict(name="rs", num_tokens=n, hidden=hidden, num_experts=e, topk=k, num_ranks=r,
               tokens_per_rank=tokens_per_rank,
               topk_idx=route_uniform(g, n, e, k),
               topk_weights=weights_softmax(g, n, k))
    if with_partials:
        out["partials_bf16"] = bf16_normal(g, (r, n, hidden))
    if with_expert_out:
        out["expert_out_bf16"] = bf16_normal(g, (n * k, hidden))
    return out


def skewed_case(seed: int = 0, n: int = 16384, hidden: int = 7168, e: int = 256,
                k: int = 8, r: int = 16, s: float = 1.2, num_zero: int = 8) -> dict:
    g = rng_for(seed, 5)
    return dict(
        name="skewed", num_tokens=n, hidden=hidden, num_experts=e, topk=k, num_ranks=r,
        topk_idx=route_zipf(g, n, e, k, s, num_zero),
        topk_weights=weights_softmax(g, n, k),
        hidden_bf16=bf16_normal(g, (n, hidden)),
    )


def decode_ll_case(seed: int = 0, tokens_per_rank: int = 128, r: int = 8, hidden: int = 7168,
                   e: int = 256, k: int = 8) -> dict:
    g = rng_for(seed, 6)
    n = tokens_per_rank * r
    return dict(
        name="decode_ll", num_tokens=n, hidden=hidden, num_experts=e, topk=k, num_ranks=r,
        max_tokens_per_rank=tokens_per_rank,
        topk_idx=route_uniform(g, n, e, k),
        topk_weights=weights_abs_normal(g, n, k),
        hidden_bf16=bf16_normal(g, (n, hidden)),
    )
