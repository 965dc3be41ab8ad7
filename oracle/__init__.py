"""Python access to the plain CPU oracle (oracle.c) through ctypes.

TEST INFRASTRUCTURE ONLY. Tests, the package smoke check and the benchmark's
CPU-baseline leg may import this module; the product path (the CUDA library
and its binding) never does. All arrays are numpy arrays on the host.
"""
from __future__ import annotations

import ctypes
import fcntl
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

BF16, FP8_E4M3_B128, NVFP4_B16, RAW, FP8_E4M3_UE8M0 = 0, 1, 2, 3, 4

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fast-math, no FMA
    contraction, no host-specific flags)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))

    def stale():
        return force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest

    if stale():
        # processes of a spawned pool may build at once: one compiles, the
        # others wait on the lock and find the library built
        with open(_LIB + ".lock", "w") as lock:
            fcntl.flock(lock, fcntl.LOCK_EX)
            if stale():
                tmp = f"{_LIB}.{os.getpid()}.tmp"
                cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                       "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
                subprocess.check_call(cmd)
                os.replace(tmp, _LIB)
                force = False
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        f32, u8, u16, i32 = ctypes.c_float, ctypes.c_uint8, ctypes.c_uint16, ctypes.c_int
        _lib.oracle_bf16_to_f32.restype = f32
        _lib.oracle_bf16_to_f32.argtypes = [u16]
        _lib.oracle_f32_to_bf16.restype = u16
        _lib.oracle_f32_to_bf16.argtypes = [f32]
        _lib.oracle_e4m3_value.restype = f32
        _lib.oracle_e4m3_value.argtypes = [u8]
        _lib.oracle_e4m3_encode.restype = u8
        _lib.oracle_e4m3_encode.argtypes = [f32]
        _lib.oracle_e2m1_value.restype = f32
        _lib.oracle_e2m1_value.argtypes = [u8]
        _lib.oracle_e2m1_encode.restype = u8
        _lib.oracle_e2m1_encode.argtypes = [f32]
        _lib.oracle_fp8_group.restype = None
        _lib.oracle_nvfp4_group.restype = None
        _lib.oracle_fp8_ue8m0_group.restype = None
        for name in ("oracle_record_layout", "oracle_layout", "oracle_dispatch",
                     "oracle_identity_expert", "oracle_combine_topk", "oracle_combine_ranks",
                     "oracle_combine_topk_ranks", "oracle_combine_topk_f64"):
            getattr(_lib, name).restype = i32
        for name in ("oracle_slot_layout", "oracle_pack_slots", "oracle_unpack_slots",
                     "oracle_rank_layout", "oracle_dispatch_ranks", "oracle_combine_gather_ranks",
                     "oracle_ll_layout", "oracle_dispatch_ll", "oracle_combine_backward",
                     "oracle_dispatch_backward", "oracle_gather_ranks_backward"):
            getattr(_lib, name).restype = i32
        # routines with 64-bit scalar arguments need their full signatures:
        # ctypes passes a bare Python int as a 32-bit C int
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        _lib.oracle_dispatch_ll.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, i64,
                                            vp, vp]
        _lib.oracle_combine_backward.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, vp, vp]
        _lib.oracle_gather_ranks_backward.argtypes = [vp, vp, i32, i32, i32, i64, vp]
        _lib.oracle_mask_topk_ids.restype = None
        _lib.oracle_combine_norm.restype = i32
        _lib.oracle_combine_norm.argtypes = [i32] + [ctypes.c_void_p] * 4 + [i32] * 5 + \
            [ctypes.c_void_p, ctypes.c_void_p, f32, ctypes.c_void_p, ctypes.c_void_p]
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return ctypes.c_void_p(0)
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


# ---- number formats --------------------------------------------------------

def bf16_to_f32(b: int) -> float:
    return _load().oracle_bf16_to_f32(int(b))


def f32_to_bf16(f: float) -> int:
    return _load().oracle_f32_to_bf16(float(np.float32(f)))


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e4m3_encode(x: float) -> int:
    return _load().oracle_e4m3_encode(float(np.float32(x)))


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e2m1_encode(x: float) -> int:
    return _load().oracle_e2m1_encode(float(np.float32(x)))


def bf16_to_f32_array(b: np.ndarray) -> np.ndarray:
    """Vector form of bf16_to_f32 (an exact widening, used by tests)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_array(f: np.ndarray) -> np.ndarray:
    lib = _load()
    f = np.ascontiguousarray(f, dtype=np.float32)
    return np.array([lib.oracle_f32_to_bf16(float(v)) for v in f.ravel()],
                    dtype=np.uint16).reshape(f.shape)


def fp8_group(x_bf16: np.ndarray):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    q = np.zeros(x.size, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.float32)
    _load().oracle_fp8_group(_p(x), ctypes.c_int(x.size), _p(q), _p(sc))
    return q, float(sc[0])


def nvfp4_group(x_bf16: np.ndarray):
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    assert x.size % 2 == 0
    q = np.zeros(x.size // 2, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.uint8)
    _load().oracle_nvfp4_group(_p(x), ctypes.c_int(x.size), _p(q), _p(sc))
    return q, int(sc[0])


# ---- record layout -----------------------------------------------------------

def fp8_ue8m0_group(x_bf16: np.ndarray):
    """(e4m3 codes uint8 [n], UE8M0 scale byte) of one group."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    q = np.zeros(x.size, np.uint8)
    b = np.zeros(1, np.uint8)
    _load().oracle_fp8_ue8m0_group(_p(x), x.size, _p(q), _p(b))
    return q, int(b[0])


def record_layout(topk: int, hidden: int, in_kind: int, out_kind: int,
                  raw_payload_bytes: int = 0, raw_scale_bytes: int = 0) -> dict:
    out = np.zeros(7, dtype=np.int32)
    rc = _load().oracle_record_layout(topk, hidden, in_kind, out_kind, raw_payload_bytes,
                                      raw_scale_bytes, _p(out))
    _check(rc, "record_layout")
    keys = ("record_bytes", "off_ids", "off_weights", "off_payload", "off_scales",
            "payload_bytes", "scale_bytes")
    return {k: int(v) for k, v in zip(keys, out)}


# ---- layout -------------------------------------------------------------------

def layout(topk_idx: np.ndarray, num_experts: int, num_ranks: int) -> dict:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    n, k = idx.shape
    out = dict(
        tokens_per_expert=np.zeros(num_experts, np.int32),
        tokens_per_rank=np.zeros(num_ranks, np.int32),
        is_token_in_rank=np.zeros((n, num_ranks), np.uint8),
        expert_offset=np.zeros(num_experts + 1, np.int32),
        rank_offset=np.zeros(num_ranks + 1, np.int32),
        slot_of=np.zeros((n, k), np.int32),
        src_of_slot=np.zeros(n * k, np.int32),
    )
    rc = _load().oracle_layout(
        _p(idx), n, k, num_experts, num_ranks, _p(out["tokens_per_expert"]),
        _p(out["tokens_per_rank"]), _p(out["is_token_in_rank"]), _p(out["expert_offset"]),
        _p(out["rank_offset"]), _p(out["slot_of"]), _p(out["src_of_slot"]))
    _check(rc, "layout")
    out["num_pairs"] = int(out["expert_offset"][-1])
    return out


# ---- dispatch -------------------------------------------------------------------

def dispatch(topk_idx, topk_weights, hidden, scales, slot_of, num_records: int,
             in_kind: int, out_kind: int, hidden_size: int,
             raw_payload_bytes: int = 0, raw_scale_bytes: int = 0) -> np.ndarray:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    n, k = idx.shape
    lay = record_layout(k, hidden_size, in_kind, out_kind, raw_payload_bytes, raw_scale_bytes)
    rec = np.zeros((num_records, lay["record_bytes"]), dtype=np.uint8)
    h = np.ascontiguousarray(hidden)
    sc = None if scales is None else np.ascontiguousarray(scales)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    rc = _load().oracle_dispatch(_p(idx), _p(w), _p(h), _p(sc), n, k, hidden_size, in_kind,
                                 out_kind, raw_payload_bytes, raw_scale_bytes, _p(so), _p(rec))
    _check(rc, "dispatch")
    return rec


def identity_expert(records: np.ndarray, topk: int, hidden_size: int, out_kind: int) -> np.ndarray:
    rec = np.ascontiguousarray(records, dtype=np.uint8)
    y = np.zeros((rec.shape[0], hidden_size), dtype=np.uint16)
    rc = _load().oracle_identity_expert(_p(rec), rec.shape[0], topk, hidden_size, out_kind, _p(y))
    _check(rc, "identity_expert")
    return y


# ---- combine ----------------------------------------------------------------------

def combine_topk(y, topk_weights, slot_of, hidden_size: int) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    n, k = so.shape
    out = np.zeros((n, hidden_size), dtype=np.uint16)
    _check(_load().oracle_combine_topk(_p(y), _p(w), _p(so), n, k, hidden_size, _p(out)),
           "combine_topk")
    return out


def combine_ranks(partials) -> np.ndarray:
    p = np.ascontiguousarray(partials, dtype=np.uint16)
    r, n, h = p.shape
    out = np.zeros((n, h), dtype=np.uint16)
    _check(_load().oracle_combine_ranks(_p(p), r, n, h, _p(out)), "combine_ranks")
    return out


def combine_topk_ranks(y, topk_idx, topk_weights, slot_of, num_experts: int, num_ranks: int,
                       hidden_size: int) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    n, k = so.shape
    out = np.zeros((n, hidden_size), dtype=np.uint16)
    _check(_load().oracle_combine_topk_ranks(_p(y), _p(idx), _p(w), _p(so), n, k, num_experts,
                                             num_ranks, hidden_size, _p(out)),
           "combine_topk_ranks")
    return out


def combine_topk_f64(y, topk_weights, slot_of, hidden_size: int) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    n, k = so.shape
    out = np.zeros((n, hidden_size), dtype=np.float64)
    _check(_load().oracle_combine_topk_f64(_p(y), _p(w), _p(so), n, k, hidden_size, _p(out)),
           "combine_topk_f64")
    return out


def combine_norm(mode: int, y, topk_idx, topk_weights, slot_of, residual, gamma, eps: float,
                 num_experts: int, num_ranks: int, hidden_size: int):
    """mode 0 top-k, 1 rank sum (y = partials [R, N, H]), 2 top-k grouped by rank.
    Returns (normed, residual_out), uint16 BF16 patterns [N, H]."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    res = np.ascontiguousarray(residual, dtype=np.uint16)
    g = np.ascontiguousarray(gamma, dtype=np.uint16)
    n = res.shape[0]
    if mode == 1:
        idx = w = so = None
        k = 1
    else:
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        w = np.ascontiguousarray(topk_weights, dtype=np.float32)
        so = np.ascontiguousarray(slot_of, dtype=np.int32)
        k = so.shape[1]
    normed = np.zeros((n, hidden_size), dtype=np.uint16)
    rout = np.zeros((n, hidden_size), dtype=np.uint16)
    rc = _load().oracle_combine_norm(mode, _p(y), _p(idx), _p(w), _p(so), n, k, num_experts,
                                     num_ranks, hidden_size, _p(res), _p(g), float(eps),
                                     _p(normed), _p(rout))
    _check(rc, "combine_norm")
    return normed, rout


def slot_layout(bytes_per_rank):
    b = np.ascontiguousarray(bytes_per_rank, dtype=np.int64)
    off = np.zeros(len(b), np.int64)
    sb = np.zeros(1, np.int64)
    _check(_load().oracle_slot_layout(len(b), _p(b), _p(off), _p(sb)), "slot_layout")
    return off.tolist(), int(sb[0])


def _ptr_array(arrs):
    return (ctypes.c_void_p * 4)(*[a.ctypes.data for a in arrs])


def pack_slots(tensors, num_ranks: int) -> np.ndarray:
    """tensors: rank-major numpy arrays; returns uint8 slots [R, slot_bytes]."""
    ts = [np.ascontiguousarray(t).view(np.uint8).reshape(-1) for t in tensors]
    b = np.array([t.size // num_ranks for t in ts], np.int64)
    _, sb = slot_layout(b)
    slots = np.zeros((num_ranks, sb), np.uint8)
    _check(_load().oracle_pack_slots(len(ts), num_ranks, _p(b), _ptr_array(ts), _p(slots)),
           "pack_slots")
    return slots


def unpack_slots(slots, bytes_per_rank, num_ranks: int):
    s = np.ascontiguousarray(slots, dtype=np.uint8)
    b = np.ascontiguousarray(bytes_per_rank, dtype=np.int64)
    outs = [np.zeros(int(x) * num_ranks, np.uint8) for x in b]
    _check(_load().oracle_unpack_slots(len(b), num_ranks, _p(b), _p(s), _ptr_array(outs)),
           "unpack_slots")
    return outs


def mask_topk_ids(topk_idx, num_actual_tokens: int) -> np.ndarray:
    ids = np.array(topk_idx, dtype=np.int32, copy=True, order="C")
    n, k = ids.shape
    _load().oracle_mask_topk_ids(_p(ids), n, k, int(num_actual_tokens))
    return ids


def rank_layout(is_token_in_rank, tokens_per_expert, expert_alignment: int = 1) -> dict:
    m = np.ascontiguousarray(is_token_in_rank, dtype=np.uint8)
    tpe = np.ascontiguousarray(tokens_per_expert, dtype=np.int32)
    n, r = m.shape
    out = dict(send_head=np.zeros((n, r), np.int32), recv_src_idx=np.zeros(n * r, np.int32),
               recv_offset=np.zeros(r + 1, np.int32), recv_tokens_per_expert=np.zeros(tpe.size, np.int32))
    _check(_load().oracle_rank_layout(_p(m), _p(tpe), n, r, tpe.size, expert_alignment,
                                      _p(out["send_head"]), _p(out["recv_src_idx"]),
                                      _p(out["recv_offset"]), _p(out["recv_tokens_per_expert"])),
           "rank_layout")
    return out


def dispatch_ranks(topk_idx, topk_weights, hidden, scales, send_head, num_records: int,
                   num_experts: int, in_kind: int, out_kind: int, hidden_size: int,
                   raw_payload_bytes: int = 0, raw_scale_bytes: int = 0) -> np.ndarray:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    sh = np.ascontiguousarray(send_head, dtype=np.int32)
    n, k = idx.shape
    lay = record_layout(k, hidden_size, in_kind, out_kind, raw_payload_bytes, raw_scale_bytes)
    rec = np.zeros((num_records, lay["record_bytes"]), dtype=np.uint8)
    h = np.ascontiguousarray(hidden)
    sc = None if scales is None else np.ascontiguousarray(scales)
    _check(_load().oracle_dispatch_ranks(_p(idx), _p(w), _p(h), _p(sc), n, k, num_experts,
                                         sh.shape[1], hidden_size, in_kind, out_kind,
                                         raw_payload_bytes, raw_scale_bytes, _p(sh), _p(rec)),
           "dispatch_ranks")
    return rec


def combine_gather_ranks(recv_out, send_head, hidden_size: int) -> np.ndarray:
    y = np.ascontiguousarray(recv_out, dtype=np.uint16)
    sh = np.ascontiguousarray(send_head, dtype=np.int32)
    n, r = sh.shape
    out = np.zeros((n, hidden_size), np.uint16)
    _check(_load().oracle_combine_gather_ranks(_p(y), _p(sh), n, r, hidden_size, _p(out)),
           "combine_gather_ranks")
    return out


def ll_layout(topk_idx, num_experts: int, num_ranks: int, max_tokens_per_rank: int) -> dict:
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    n, k = idx.shape
    cap = num_ranks * max_tokens_per_rank
    out = dict(ll_slot_of=np.zeros((n, k), np.int32), src_info=np.zeros((num_experts, cap), np.int32),
               layout_range=np.zeros((num_experts, num_ranks), np.int64),
               recv_count=np.zeros(num_experts, np.int32))
    _check(_load().oracle_ll_layout(_p(idx), n, k, num_experts, num_ranks, max_tokens_per_rank,
                                    _p(out["ll_slot_of"]), _p(out["src_info"]),
                                    _p(out["layout_range"]), _p(out["recv_count"])), "ll_layout")
    return out


def dispatch_ll(hidden, scales, ll_slot_of, rows: int, in_kind: int, out_kind: int,
                hidden_size: int, raw_payload_bytes: int = 0, raw_scale_bytes: int = 0):
    so = np.ascontiguousarray(ll_slot_of, dtype=np.int32)
    n, k = so.shape
    lay = record_layout(k, hidden_size, in_kind, out_kind, raw_payload_bytes, raw_scale_bytes)
    x = np.zeros((rows, lay["payload_bytes"]), np.uint8)
    scale_row = (lay["scale_bytes"] + 15) // 16 * 16
    sc = np.zeros((rows, max(scale_row, 1)), np.uint8)
    h = np.ascontiguousarray(hidden)
    s_in = None if scales is None else np.ascontiguousarray(scales)
    _check(_load().oracle_dispatch_ll(_p(h), _p(s_in), n, k, hidden_size, in_kind, out_kind,
                                      raw_payload_bytes, raw_scale_bytes, _p(so), rows, _p(x), _p(sc)),
           "dispatch_ll")
    return x, sc[:, :scale_row]


def combine_backward(grad_out, topk_weights, slot_of, y, rows: int, hidden_size: int,
                     grad_y=None):
    """(grad_y bf16 [rows, H], grad_w fp32 [N, k] or None). Rows of grad_y no
    pair names keep their given values (zeros when grad_y is None)."""
    g = np.ascontiguousarray(grad_out, dtype=np.uint16)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    n, k = so.shape
    gy = np.zeros((rows, hidden_size), np.uint16) if grad_y is None else np.array(grad_y, np.uint16)
    yy = None if y is None else np.ascontiguousarray(y, dtype=np.uint16)
    gw = np.zeros((n, k), np.float32)
    _check(_load().oracle_combine_backward(_p(g), _p(w), _p(so), _p(yy), rows, n, k, hidden_size,
                                           _p(gy), _p(gw)), "combine_backward")
    return gy, (gw if y is not None else None)


def dispatch_backward(grad_in, slot_of, hidden_size: int) -> np.ndarray:
    gi = np.ascontiguousarray(grad_in, dtype=np.uint16)
    so = np.ascontiguousarray(slot_of, dtype=np.int32)
    n, k = so.shape
    out = np.zeros((n, hidden_size), np.uint16)
    _check(_load().oracle_dispatch_backward(_p(gi), _p(so), n, k, hidden_size, _p(out)),
           "dispatch_backward")
    return out


def gather_ranks_backward(grad_out, send_head, rows: int, hidden_size: int, grad_recv=None):
    g = np.ascontiguousarray(grad_out, dtype=np.uint16)
    sh = np.ascontiguousarray(send_head, dtype=np.int32)
    n, r = sh.shape
    gr = np.zeros((rows, hidden_size), np.uint16) if grad_recv is None else np.array(grad_recv, np.uint16)
    _check(_load().oracle_gather_ranks_backward(_p(g), _p(sh), n, r, hidden_size, rows, _p(gr)),
           "gather_ranks_backward")
    return gr
