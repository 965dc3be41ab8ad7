"""Thin Python binding of libmoe.so (include/moe.h) through ctypes.

Argument marshalling only: every step of layout, dispatch and combine runs in
the library's CUDA kernels. PyTorch supplies device memory and the current
stream. There is no fallback: if libmoe.so is missing, importing this module
raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_ALIGNMENT = -2
MOE_ERR_SHAPE = -3
MOE_ERR_CAPACITY = -4
MOE_ERR_CUDA = -5
MOE_ERR_DEVICE_IDS = -6
MOE_ERR_TOO_LARGE = -7
MOE_ERR_TIMEOUT = -8
MOE_NOALLOC_SCRATCH_BYTES = 2 << 20

MOE_PAYLOAD_BF16 = 0
MOE_PAYLOAD_FP8_E4M3_B128 = 1
MOE_PAYLOAD_NVFP4_B16 = 2
MOE_PAYLOAD_RAW = 3
MOE_PAYLOAD_FP8_E4M3_UE8M0 = 4

MOE_COMBINE_TOPK = 0
MOE_COMBINE_RANKS = 1
MOE_COMBINE_TOPK_RANKS = 2

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
        "(there is no CPU fallback)")
_lib = ctypes.CDLL(LIB_PATH)

_i32, _i64, _sz, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p


class _Desc(ctypes.Structure):
    _fields_ = [("num_tokens", _i32), ("topk", _i32), ("num_experts", _i32), ("num_ranks", _i32),
                ("hidden", _i32), ("in_kind", _i32), ("out_kind", _i32),
                ("raw_payload_bytes", _i32), ("raw_scale_bytes", _i32)]


class _Layout(ctypes.Structure):
    _fields_ = [("record_bytes", _i32), ("off_ids", _i32), ("off_weights", _i32),
                ("off_payload", _i32), ("off_scales", _i32), ("payload_bytes", _i32),
                ("scale_bytes", _i32)]


_D = ctypes.POINTER(_Desc)
_lib.moe_strerror.restype = ctypes.c_char_p
_lib.moe_strerror.argtypes = [ctypes.c_int]
_lib.moe_record_layout.restype = ctypes.c_int
_lib.moe_record_layout.argtypes = [_D, ctypes.POINTER(_Layout)]
_lib.moe_workspace_size.restype = _sz
_lib.moe_workspace_size.argtypes = [_D]
_lib.moe_layout.restype = ctypes.c_int
_lib.moe_layout.argtypes = [_D] + [_vp] * 9 + [_sz, _vp]
_lib.moe_layout_noalloc.restype = ctypes.c_int
_lib.moe_layout_noalloc.argtypes = [_D] + [_vp] * 10
_lib.moe_layout_status.restype = ctypes.c_int
_lib.moe_layout_status.argtypes = [_vp, ctypes.POINTER(_i32), _vp]
_lib.moe_dispatch.restype = ctypes.c_int
_lib.moe_dispatch.argtypes = [_D] + [_vp] * 6 + [_sz, _vp]
_lib.moe_layout_dispatch.restype = ctypes.c_int
_lib.moe_layout_dispatch.argtypes = [_D] + [_vp] * 12 + [_sz, _vp, _sz, _vp]
_lib.moe_combine.restype = ctypes.c_int
_lib.moe_combine.argtypes = [_D, ctypes.c_int, _vp, _i64, _vp, _vp, _vp, _vp, _vp]
_lib.moe_combine_norm.restype = ctypes.c_int
_lib.moe_combine_norm.argtypes = [_D, ctypes.c_int, _vp, _i64, _vp, _vp, _vp, _vp, _vp,
                                  ctypes.c_float, _vp, _vp, _vp]


class _SlotDesc(ctypes.Structure):
    _fields_ = [("num_tensors", _i32), ("num_ranks", _i32), ("bytes", _i64 * 4)]


_SD = ctypes.POINTER(_SlotDesc)
_lib.moe_slot_layout.restype = ctypes.c_int
_lib.moe_slot_layout.argtypes = [_SD, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
_lib.moe_pack_slots.restype = ctypes.c_int
_lib.moe_pack_slots.argtypes = [_SD, ctypes.POINTER(_vp), _vp, _vp]
_lib.moe_unpack_slots.restype = ctypes.c_int
_lib.moe_unpack_slots.argtypes = [_SD, _vp, ctypes.POINTER(_vp), _vp]
_lib.moe_rank_layout.restype = ctypes.c_int
_lib.moe_rank_layout.argtypes = [_D, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]
_lib.moe_layout_ll_dispatch.restype = ctypes.c_int
_lib.moe_layout_ll_dispatch.argtypes = [_D] + [_vp] * 10 + [_i32] + [_vp] * 5 + [_sz, _vp, _sz, _vp, _sz, _vp]
_lib.moe_layout_ll.restype = ctypes.c_int
_lib.moe_layout_ll.argtypes = [_D] + [_vp] * 8 + [_i32] + [_vp] * 5 + [_sz, _vp]
_lib.moe_layout_ranks.restype = ctypes.c_int
_lib.moe_layout_ranks.argtypes = [_D] + [_vp] * 8 + [_i32] + [_vp] * 5 + [_sz, _vp]
_lib.moe_dispatch_ranks.restype = ctypes.c_int
_lib.moe_dispatch_ranks.argtypes = [_D] + [_vp] * 6 + [_sz, _vp]
_lib.moe_combine_gather_ranks.restype = ctypes.c_int
_lib.moe_combine_gather_ranks.argtypes = [_D, _vp, _i64, _vp, _vp, _vp]
_lib.moe_ll_layout.restype = ctypes.c_int
_lib.moe_ll_layout.argtypes = [_D, _i32] + [_vp] * 8 + [_vp]
_lib.moe_dispatch_ll.restype = ctypes.c_int
_lib.moe_dispatch_ll.argtypes = [_D, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp]
_lib.moe_combine_backward.restype = ctypes.c_int
_lib.moe_combine_backward.argtypes = [_D, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp]
_lib.moe_dispatch_backward.restype = ctypes.c_int
_lib.moe_dispatch_backward.argtypes = [_D, _vp, _i64, _vp, _vp, _vp]
_lib.moe_combine_gather_ranks_backward.restype = ctypes.c_int
_lib.moe_combine_gather_ranks_backward.argtypes = [_D, _vp, _vp, _vp, _i64, _vp]
_lib.moe_mask_topk_ids.restype = ctypes.c_int
_lib.moe_mask_topk_ids.argtypes = [_vp, _i32, _i32, _vp, _vp]
_lib.moe_device_status.restype = ctypes.c_int
_lib.moe_device_status.argtypes = [_vp, ctypes.c_int]
_lib.moe_set_wait_limit_ns.restype = ctypes.c_int
_lib.moe_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
_lib.moe_pack_record.restype = ctypes.c_int
_lib.moe_pack_record.argtypes = [_D, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]
_lib.moe_unpack_record.restype = ctypes.c_int
_lib.moe_unpack_record.argtypes = [_D, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {moe_strerror(code)} ({code})")
        self.code = code


@dataclass
class MoeDesc:
    """Shape and format of one call (moe_desc_t)."""
    num_tokens: int
    topk: int
    num_experts: int
    num_ranks: int
    hidden: int
    in_kind: int = MOE_PAYLOAD_BF16
    out_kind: int = MOE_PAYLOAD_BF16
    raw_payload_bytes: int = 0
    raw_scale_bytes: int = 0

    def c(self) -> _Desc:
        return _Desc(self.num_tokens, self.topk, self.num_experts, self.num_ranks, self.hidden,
                     self.in_kind, self.out_kind, self.raw_payload_bytes, self.raw_scale_bytes)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr() if t.numel() else None
    return t


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def moe_strerror(code: int) -> str:
    return _lib.moe_strerror(int(code)).decode()


def moe_record_layout(desc: MoeDesc) -> dict:
    lay = _Layout()
    _check(_lib.moe_record_layout(ctypes.byref(desc.c()), ctypes.byref(lay)), "moe_record_layout")
    return {name: getattr(lay, name) for name, _ in _Layout._fields_}


def moe_workspace_size(desc: MoeDesc) -> int:
    return int(_lib.moe_workspace_size(ctypes.byref(desc.c())))


def layout_outputs(desc: MoeDesc, device) -> dict:
    """Allocates the output tensors of moe_layout (torch device memory)."""
    n, k, e, r = desc.num_tokens, desc.topk, desc.num_experts, desc.num_ranks
    i32 = dict(dtype=torch.int32, device=device)
    return dict(
        tokens_per_expert=torch.empty(e, **i32),
        tokens_per_rank=torch.empty(r, **i32),
        is_token_in_rank=torch.empty((n, r), dtype=torch.uint8, device=device),
        expert_offset=torch.empty(e + 1, **i32),
        rank_offset=torch.empty(r + 1, **i32),
        slot_of=torch.empty((n, k), **i32),
        src_of_slot=torch.empty(n * k, **i32),
    )


def moe_layout(desc: MoeDesc, topk_idx: torch.Tensor, out: dict | None = None,
               workspace: torch.Tensor | None = None, stream=None) -> dict:
    """Routing layout (see include/moe.h). Returns the dict of output tensors
    (plus 'workspace')."""
    if out is None:
        out = layout_outputs(desc, topk_idx.device)
    if workspace is None:
        workspace = torch.empty(max(moe_workspace_size(desc), 256), dtype=torch.uint8,
                                device=topk_idx.device)
    rc = _lib.moe_layout(ctypes.byref(desc.c()), _ptr(topk_idx), _ptr(out["tokens_per_expert"]),
                         _ptr(out["tokens_per_rank"]), _ptr(out["is_token_in_rank"]),
                         _ptr(out["expert_offset"]), _ptr(out["rank_offset"]),
                         _ptr(out["slot_of"]), _ptr(out.get("src_of_slot")), _ptr(workspace),
                         workspace.numel(), _stream(stream))
    _check(rc, "moe_layout")
    out["workspace"] = workspace
    return out


def moe_layout_noalloc(desc: MoeDesc, topk_idx: torch.Tensor, out: dict | None = None,
                       status: torch.Tensor | None = None, stream=None) -> dict:
    """Routing layout without a workspace, for callers that cannot provide
    device scratch: the library uses its own fixed 2 MiB device array instead
    (see include/moe.h for the size limit and the rule that calls overlapping
    on the GPU race). `status` (int32 [1] on the device) receives this call's
    status word."""
    if out is None:
        out = layout_outputs(desc, topk_idx.device)
    rc = _lib.moe_layout_noalloc(ctypes.byref(desc.c()), _ptr(topk_idx),
                                 _ptr(out["tokens_per_expert"]), _ptr(out["tokens_per_rank"]),
                                 _ptr(out["is_token_in_rank"]), _ptr(out["expert_offset"]),
                                 _ptr(out["rank_offset"]), _ptr(out["slot_of"]),
                                 _ptr(out.get("src_of_slot")), _ptr(status), _stream(stream))
    _check(rc, "moe_layout_noalloc")
    return out


def moe_device_status(clear: bool = True) -> int:
    """Status of the kernels with bounded waits on this device since the last
    clearing call: MOE_OK or MOE_ERR_TIMEOUT (synchronises the device)."""
    v = _i32(0)
    _check(_lib.moe_device_status(ctypes.byref(v), 1 if clear else 0), "moe_device_status")
    return v.value


def moe_set_wait_limit_ns(ns: int) -> None:
    """Budget of the bounded waits for later launches (0 = the default one
    second; a test hook, see include/moe.h)."""
    _check(_lib.moe_set_wait_limit_ns(int(ns)), "moe_set_wait_limit_ns")


def moe_layout_status(workspace: torch.Tensor, stream=None) -> int:
    """Status word of the last moe_layout on this workspace (synchronises)."""
    v = _i32(0)
    _check(_lib.moe_layout_status(_ptr(workspace), ctypes.byref(v), _stream(stream)),
           "moe_layout_status")
    return v.value


def moe_dispatch(desc: MoeDesc, topk_idx: torch.Tensor, topk_weights: torch.Tensor,
                 hidden: torch.Tensor, scales: torch.Tensor | None, slot_of: torch.Tensor,
                 records: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Permute and pack: writes one record per routed pair into `records`
    (uint8 [N*k, record_bytes] when allocated here)."""
    lay = moe_record_layout(desc)
    if records is None:
        records = torch.empty((desc.num_tokens * desc.topk, lay["record_bytes"]),
                              dtype=torch.uint8, device=topk_idx.device)
    nbytes = records.numel() * records.element_size()
    rc = _lib.moe_dispatch(ctypes.byref(desc.c()), _ptr(topk_idx), _ptr(topk_weights),
                           _ptr(hidden), _ptr(scales), _ptr(slot_of), _ptr(records), nbytes,
                           _stream(stream))
    _check(rc, "moe_dispatch")
    return records


def moe_combine(desc: MoeDesc, mode: int, expert_out: torch.Tensor,
                topk_idx: torch.Tensor | None, topk_weights: torch.Tensor | None,
                slot_of: torch.Tensor | None, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Combine (see include/moe.h): returns bf16 [N, H]."""
    if out is None:
        out = torch.empty((desc.num_tokens, desc.hidden), dtype=torch.bfloat16,
                          device=expert_out.device)
    rows = expert_out.numel() // max(desc.hidden, 1)
    rc = _lib.moe_combine(ctypes.byref(desc.c()), int(mode), _ptr(expert_out), rows,
                          _ptr(topk_idx), _ptr(topk_weights), _ptr(slot_of), _ptr(out),
                          _stream(stream))
    _check(rc, "moe_combine")
    return out


def moe_combine_norm(desc: MoeDesc, mode: int, expert_out: torch.Tensor,
                     topk_idx: torch.Tensor | None, topk_weights: torch.Tensor | None,
                     slot_of: torch.Tensor | None, residual_in: torch.Tensor,
                     gamma: torch.Tensor, eps: float, normed_out: torch.Tensor | None = None,
                     residual_out: torch.Tensor | None = None, stream=None):
    """Combine fused with residual add and RMSNorm (see include/moe.h).
    Returns (normed_out, residual_out), both bf16 [N, H]."""
    shape = (desc.num_tokens, desc.hidden)
    if normed_out is None:
        normed_out = torch.empty(shape, dtype=torch.bfloat16, device=expert_out.device)
    if residual_out is None:
        residual_out = torch.empty(shape, dtype=torch.bfloat16, device=expert_out.device)
    rows = expert_out.numel() // max(desc.hidden, 1)
    rc = _lib.moe_combine_norm(ctypes.byref(desc.c()), int(mode), _ptr(expert_out), rows,
                               _ptr(topk_idx), _ptr(topk_weights), _ptr(slot_of),
                               _ptr(residual_in), _ptr(gamma), float(eps), _ptr(normed_out),
                               _ptr(residual_out), _stream(stream))
    _check(rc, "moe_combine_norm")
    return normed_out, residual_out


def moe_rank_layout(desc: MoeDesc, lay: dict, expert_alignment: int = 1, out: dict | None = None,
                    stream=None) -> dict:
    """Per-rank receive layout from moe_layout's outputs (see include/moe.h)."""
    n, r, e = desc.num_tokens, desc.num_ranks, desc.num_experts
    dev = lay["tokens_per_rank"].device
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = dict(send_head=torch.empty((n, r), **i32), recv_src_idx=torch.empty(n * r, **i32),
                   recv_offset=torch.empty(r + 1, **i32),
                   recv_tokens_per_expert=torch.empty(e, **i32))
    rc = _lib.moe_rank_layout(ctypes.byref(desc.c()), _ptr(lay["is_token_in_rank"]),
                              _ptr(lay["tokens_per_rank"]), _ptr(lay["tokens_per_expert"]),
                              int(expert_alignment), _ptr(out["send_head"]),
                              _ptr(out.get("recv_src_idx")), _ptr(out["recv_offset"]),
                              _ptr(out["recv_tokens_per_expert"]), _stream(stream))
    _check(rc, "moe_rank_layout")
    return out


def rank_layout_outputs(desc: MoeDesc, device) -> dict:
    """Fresh receive-layout output tensors of one call (int32, on device)."""
    n, r, e = desc.num_tokens, desc.num_ranks, desc.num_experts
    i32 = dict(dtype=torch.int32, device=device)
    return dict(send_head=torch.empty((n, r), **i32), recv_src_idx=torch.empty(n * r, **i32),
                recv_offset=torch.empty(r + 1, **i32), recv_tokens_per_expert=torch.empty(e, **i32))


def moe_layout_ranks(desc: MoeDesc, topk_idx: torch.Tensor, expert_alignment: int = 1,
                     out: dict | None = None, rank_out: dict | None = None, workspace=None,
                     stream=None) -> tuple[dict, dict]:
    """moe_layout and moe_rank_layout in one call (see include/moe.h).
    Returns (layout outputs with the workspace, receive-layout outputs)."""
    if out is None:
        out = layout_outputs(desc, topk_idx.device)
    if rank_out is None:
        rank_out = rank_layout_outputs(desc, topk_idx.device)
    if workspace is None:
        workspace = torch.empty(max(moe_workspace_size(desc), 256), dtype=torch.uint8, device=topk_idx.device)
    prepare_layout_ranks(desc, topk_idx, expert_alignment, out, rank_out, workspace, stream)()
    out["workspace"] = workspace
    return out, rank_out


def prepare_layout_ranks(desc: MoeDesc, topk_idx, expert_alignment: int, out: dict, rank_out: dict,
                         workspace, stream=None) -> Prepared:
    d = desc.c()
    args = (ctypes.byref(d),
            *_vps(topk_idx, out["tokens_per_expert"], out["tokens_per_rank"], out["is_token_in_rank"],
                  out["expert_offset"], out["rank_offset"], out["slot_of"], out.get("src_of_slot")),
            ctypes.c_int32(expert_alignment),
            *_vps(rank_out["send_head"], rank_out.get("recv_src_idx"), rank_out["recv_offset"],
                  rank_out["recv_tokens_per_expert"], workspace),
            ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_layout_ranks", args, (d, topk_idx, out, rank_out, workspace))


def moe_dispatch_ranks(desc: MoeDesc, topk_idx, topk_weights, hidden, scales, send_head,
                       records=None, stream=None) -> torch.Tensor:
    """One record per (token, rank) at send_head; records uint8 [N*R, record_bytes]
    when allocated here."""
    lay = moe_record_layout(desc)
    if records is None:
        records = torch.empty((desc.num_tokens * desc.num_ranks, lay["record_bytes"]),
                              dtype=torch.uint8, device=topk_idx.device)
    rc = _lib.moe_dispatch_ranks(ctypes.byref(desc.c()), _ptr(topk_idx), _ptr(topk_weights),
                                 _ptr(hidden), _ptr(scales), _ptr(send_head), _ptr(records),
                                 records.numel() * records.element_size(), _stream(stream))
    _check(rc, "moe_dispatch_ranks")
    return records


def moe_combine_gather_ranks(desc: MoeDesc, recv_out: torch.Tensor, send_head: torch.Tensor,
                             out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[t] = bf16(sum over ranks of recv_out[send_head[t, r]]), bf16 [N, H]."""
    if out is None:
        out = torch.empty((desc.num_tokens, desc.hidden), dtype=torch.bfloat16,
                          device=recv_out.device)
    rows = recv_out.numel() // max(desc.hidden, 1)
    rc = _lib.moe_combine_gather_ranks(ctypes.byref(desc.c()), _ptr(recv_out), rows,
                                       _ptr(send_head), _ptr(out), _stream(stream))
    _check(rc, "moe_combine_gather_ranks")
    return out


def moe_combine_backward(desc: MoeDesc, grad_out, topk_weights, slot_of, expert_out=None,
                         rows: int | None = None, grad_expert_out=None, grad_weights=None,
                         stream=None):
    """Backward of the top-k weighted combine (see include/moe.h). Returns
    (grad_expert_out bf16 [rows, H], grad_weights fp32 [N, k] or None)."""
    h = desc.hidden
    if rows is None:
        rows = expert_out.numel() // h if expert_out is not None else grad_expert_out.numel() // h
    dev = grad_out.device
    if grad_expert_out is None:
        grad_expert_out = torch.zeros((rows, h), dtype=torch.bfloat16, device=dev)
    if expert_out is not None and grad_weights is None:
        grad_weights = torch.empty((desc.num_tokens, desc.topk), dtype=torch.float32, device=dev)
    rc = _lib.moe_combine_backward(ctypes.byref(desc.c()), _ptr(grad_out), _ptr(topk_weights),
                                   _ptr(slot_of), _ptr(expert_out), int(rows), _ptr(grad_expert_out),
                                   _ptr(grad_weights) if expert_out is not None else None,
                                   _stream(stream))
    _check(rc, "moe_combine_backward")
    return grad_expert_out, grad_weights if expert_out is not None else None


def moe_dispatch_backward(desc: MoeDesc, grad_in, slot_of, grad_hidden=None, stream=None):
    """Backward of dispatch: grad_hidden[t] = bf16(sum_j grad_in[slot_of[t, j]])."""
    if grad_hidden is None:
        grad_hidden = torch.empty((desc.num_tokens, desc.hidden), dtype=torch.bfloat16,
                                  device=grad_in.device)
    rows = grad_in.numel() // max(desc.hidden, 1)
    rc = _lib.moe_dispatch_backward(ctypes.byref(desc.c()), _ptr(grad_in), rows, _ptr(slot_of),
                                    _ptr(grad_hidden), _stream(stream))
    _check(rc, "moe_dispatch_backward")
    return grad_hidden


def moe_combine_gather_ranks_backward(desc: MoeDesc, grad_out, send_head, grad_recv, stream=None):
    """grad_recv[send_head[t, r]] = grad_out[t] for every rank row the token read."""
    rows = grad_recv.numel() // max(desc.hidden, 1)
    rc = _lib.moe_combine_gather_ranks_backward(ctypes.byref(desc.c()), _ptr(grad_out),
                                                _ptr(send_head), _ptr(grad_recv), rows,
                                                _stream(stream))
    _check(rc, "moe_combine_gather_ranks_backward")
    return grad_recv


def moe_ll_layout(desc: MoeDesc, max_tokens_per_rank: int, topk_idx, lay: dict,
                  out: dict | None = None, stream=None) -> dict:
    """Fixed-capacity, expert-major receive layout (see include/moe.h)."""
    n, k, e, r = desc.num_tokens, desc.topk, desc.num_experts, desc.num_ranks
    cap = r * max_tokens_per_rank
    dev = topk_idx.device
    if out is None:
        out = dict(ll_slot_of=torch.empty((n, k), dtype=torch.int32, device=dev),
                   src_info=torch.empty((e, cap), dtype=torch.int32, device=dev),
                   layout_range=torch.empty((e, r), dtype=torch.int64, device=dev),
                   recv_count=torch.empty(e, dtype=torch.int32, device=dev))
    rc = _lib.moe_ll_layout(ctypes.byref(desc.c()), int(max_tokens_per_rank), _ptr(topk_idx),
                            _ptr(lay["slot_of"]), _ptr(lay["expert_offset"]),
                            _ptr(lay["src_of_slot"]), _ptr(out["ll_slot_of"]),
                            _ptr(out["src_info"]), _ptr(out["layout_range"]),
                            _ptr(out["recv_count"]), _stream(stream))
    _check(rc, "moe_ll_layout")
    out["capacity"] = cap
    return out


def ll_layout_outputs(desc: MoeDesc, max_tokens_per_rank: int, device) -> dict:
    """Fresh fixed-capacity layout output tensors of one call (on device)."""
    n, k, e, r = desc.num_tokens, desc.topk, desc.num_experts, desc.num_ranks
    cap = r * max_tokens_per_rank
    return dict(ll_slot_of=torch.empty((n, k), dtype=torch.int32, device=device),
                src_info=torch.empty((e, cap), dtype=torch.int32, device=device),
                layout_range=torch.empty((e, r), dtype=torch.int64, device=device),
                recv_count=torch.empty(e, dtype=torch.int32, device=device), capacity=cap)


def moe_layout_ll(desc: MoeDesc, max_tokens_per_rank: int, topk_idx: torch.Tensor, out: dict | None = None,
                  ll_out: dict | None = None, workspace=None, stream=None) -> tuple[dict, dict]:
    """moe_layout and moe_ll_layout in one call (see include/moe.h).
    Returns (layout outputs with the workspace, fixed-capacity outputs)."""
    if out is None:
        out = layout_outputs(desc, topk_idx.device)
    if ll_out is None:
        ll_out = ll_layout_outputs(desc, max_tokens_per_rank, topk_idx.device)
    if workspace is None:
        workspace = torch.empty(max(moe_workspace_size(desc), 256), dtype=torch.uint8, device=topk_idx.device)
    prepare_layout_ll(desc, max_tokens_per_rank, topk_idx, out, ll_out, workspace, stream)()
    out["workspace"] = workspace
    return out, ll_out


def prepare_layout_ll(desc: MoeDesc, max_tokens_per_rank: int, topk_idx, out: dict, ll_out: dict, workspace,
                      stream=None) -> Prepared:
    d = desc.c()
    args = (ctypes.byref(d),
            *_vps(topk_idx, out["tokens_per_expert"], out["tokens_per_rank"], out["is_token_in_rank"],
                  out["expert_offset"], out["rank_offset"], out["slot_of"], out.get("src_of_slot")),
            ctypes.c_int32(max_tokens_per_rank),
            *_vps(ll_out["ll_slot_of"], ll_out["src_info"], ll_out["layout_range"], ll_out["recv_count"],
                  workspace),
            ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_layout_ll", args, (d, topk_idx, out, ll_out, workspace))


def moe_dispatch_ll(desc: MoeDesc, hidden, scales, ll_slot_of, capacity: int,
                    x_out=None, scales_out=None, stream=None):
    """Payload and scales into [E * capacity, ...] buffers; returns (x_out, scales_out)."""
    lay = moe_record_layout(desc)
    rows = desc.num_experts * capacity
    dev = hidden.device
    if x_out is None:
        x_out = torch.empty((rows, lay["payload_bytes"]), dtype=torch.uint8, device=dev)
    if scales_out is None and lay["scale_bytes"]:
        scale_row = (lay["scale_bytes"] + 15) // 16 * 16
        scales_out = torch.empty((rows, scale_row), dtype=torch.uint8, device=dev)
    sb = scales_out.numel() * scales_out.element_size() if scales_out is not None else 0
    rc = _lib.moe_dispatch_ll(ctypes.byref(desc.c()), _ptr(hidden), _ptr(scales), _ptr(ll_slot_of),
                              _ptr(x_out), x_out.numel() * x_out.element_size(), _ptr(scales_out),
                              sb, _stream(stream))
    _check(rc, "moe_dispatch_ll")
    return x_out, scales_out


def _slot_desc(num_ranks: int, sizes) -> _SlotDesc:
    d = _SlotDesc()
    d.num_tensors = len(sizes)
    d.num_ranks = num_ranks
    for i, b in enumerate(sizes):
        d.bytes[i] = int(b)
    return d


def moe_slot_layout(num_ranks: int, bytes_per_rank) -> tuple[list[int], int]:
    """Offsets of the tensors in a rank slot and the slot size (host only)."""
    d = _slot_desc(num_ranks, bytes_per_rank)
    off = (_i64 * 4)()
    sb = _i64(0)
    _check(_lib.moe_slot_layout(ctypes.byref(d), off, ctypes.byref(sb)), "moe_slot_layout")
    return [off[i] for i in range(len(bytes_per_rank))], sb.value


def moe_pack_slots(tensors: list, num_ranks: int, slots: torch.Tensor | None = None, stream=None):
    """Packs tensors (each rank-major, numel divisible by num_ranks) into
    slots uint8 [R, slot_bytes]."""
    sizes = [t.numel() * t.element_size() // num_ranks for t in tensors]
    _, sb = moe_slot_layout(num_ranks, sizes)
    if slots is None:
        slots = torch.empty((num_ranks, sb), dtype=torch.uint8, device=tensors[0].device)
    d = _slot_desc(num_ranks, sizes)
    arr = (_vp * 4)(*[_ptr(t) for t in tensors])
    _check(_lib.moe_pack_slots(ctypes.byref(d), arr, _ptr(slots), _stream(stream)), "moe_pack_slots")
    return slots


def moe_unpack_slots(slots: torch.Tensor, outputs: list, num_ranks: int, stream=None):
    """Fills outputs (rank-major) from slots [R, slot_bytes]."""
    sizes = [t.numel() * t.element_size() // num_ranks for t in outputs]
    d = _slot_desc(num_ranks, sizes)
    arr = (_vp * 4)(*[_ptr(t) for t in outputs])
    _check(_lib.moe_unpack_slots(ctypes.byref(d), _ptr(slots), arr, _stream(stream)),
           "moe_unpack_slots")
    return outputs


def moe_mask_topk_ids(topk_idx: torch.Tensor, num_actual_tokens: torch.Tensor, stream=None):
    """Sets ids of tokens at or past the device scalar num_actual_tokens to -1."""
    n, k = topk_idx.shape
    _check(_lib.moe_mask_topk_ids(_ptr(topk_idx), n, k, _ptr(num_actual_tokens), _stream(stream)),
           "moe_mask_topk_ids")
    return topk_idx


def moe_pack_record(desc: MoeDesc, src_token: int, slot_j: int, expert: int, ids_row, w_row,
                    payload_row, scales_row):
    """Host-only: builds one record (numpy uint8) from host numpy rows."""
    import numpy as np
    lay = moe_record_layout(desc)
    rec = np.zeros(lay["record_bytes"], dtype=np.uint8)
    arrs = [np.ascontiguousarray(a) if a is not None else None
            for a in (ids_row, w_row, payload_row, scales_row)]
    p = [a.ctypes.data if a is not None else None for a in arrs]
    _check(_lib.moe_pack_record(ctypes.byref(desc.c()), src_token, slot_j, expert, p[0], p[1],
                                p[2], p[3], rec.ctypes.data), "moe_pack_record")
    return rec


def moe_unpack_record(desc: MoeDesc, record):
    """Host-only: splits one record (numpy uint8) into its fields."""
    import numpy as np
    lay = moe_record_layout(desc)
    rec = np.ascontiguousarray(record, dtype=np.uint8)
    t, j, e = _i32(), _i32(), _i32()
    ids = np.zeros(desc.topk, np.int32)
    w = np.zeros(desc.topk, np.float32)
    pay = np.zeros(lay["payload_bytes"], np.uint8)
    sc = np.zeros(lay["scale_bytes"], np.uint8)
    _check(_lib.moe_unpack_record(ctypes.byref(desc.c()), rec.ctypes.data, ctypes.byref(t),
                                  ctypes.byref(j), ctypes.byref(e), ids.ctypes.data,
                                  w.ctypes.data, pay.ctypes.data,
                                  sc.ctypes.data if sc.size else None),
           "moe_unpack_record")
    return dict(src_token=t.value, slot_j=j.value, expert=e.value, ids=ids, weights=w,
                payload=pay, scales=sc)


class Prepared:
    """One libmoe call with its arguments marshalled once, for repeated
    launches on the same buffers and stream (argument marshalling only; each
    call of the object enqueues the library's kernels again)."""

    def __init__(self, name: str, args: tuple, keep: tuple):
        self._fn = getattr(_lib, name)
        self._name = name
        self._args = args
        self._keep = keep  # ctypes structs and tensors the arguments point into

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != MOE_OK:
            raise MoeError(rc, self._name)


def _vps(*ts):
    return tuple(ctypes.c_void_p(_ptr(t)) for t in ts)


def prepare_layout(desc: MoeDesc, topk_idx, out: dict, workspace, stream=None) -> Prepared:
    d = desc.c()
    ptrs = _vps(topk_idx, out["tokens_per_expert"], out["tokens_per_rank"],
                out["is_token_in_rank"], out["expert_offset"], out["rank_offset"], out["slot_of"],
                out.get("src_of_slot"), workspace)
    args = (ctypes.byref(d), *ptrs, ctypes.c_size_t(workspace.numel()),
            ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_layout", args, (d, topk_idx, out, workspace))


def moe_layout_dispatch(desc: MoeDesc, topk_idx, topk_weights, hidden, scales, out: dict | None = None,
                        workspace=None, records=None, stream=None):
    """moe_layout then moe_dispatch in one call (see include/moe.h); the
    dispatch overlaps the layout. Returns (layout outputs dict, records)."""
    dev = topk_idx.device
    if out is None:
        out = layout_outputs(desc, dev)
    if workspace is None:
        workspace = torch.empty(max(moe_workspace_size(desc), 256), dtype=torch.uint8, device=dev)
    if records is None:
        rb = moe_record_layout(desc)["record_bytes"]
        records = torch.empty((max(desc.num_tokens * desc.topk, 1), rb), dtype=torch.uint8, device=dev)
    prepare_layout_dispatch(desc, topk_idx, topk_weights, hidden, scales, out, workspace, records,
                            stream)()
    out["workspace"] = workspace
    return out, records


def prepare_layout_dispatch(desc: MoeDesc, topk_idx, topk_weights, hidden, scales, out: dict,
                            workspace, records, stream=None) -> Prepared:
    d = desc.c()
    ptrs = _vps(topk_idx, topk_weights, hidden, scales, out["tokens_per_expert"],
                out["tokens_per_rank"], out["is_token_in_rank"], out["expert_offset"],
                out["rank_offset"], out["slot_of"], out.get("src_of_slot"), workspace)
    args = (ctypes.byref(d), *ptrs, ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(_ptr(records)),
            ctypes.c_size_t(records.numel() * records.element_size()), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_layout_dispatch", args, (d, topk_idx, topk_weights, hidden, scales, out,
                                                  workspace, records))


def prepare_dispatch(desc: MoeDesc, topk_idx, topk_weights, hidden, scales, slot_of, records,
                     stream=None) -> Prepared:
    d = desc.c()
    ptrs = _vps(topk_idx, topk_weights, hidden, scales, slot_of, records)
    args = (ctypes.byref(d), *ptrs, ctypes.c_size_t(records.numel() * records.element_size()),
            ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_dispatch", args, (d, topk_idx, topk_weights, hidden, scales, slot_of,
                                           records))


def prepare_ll_layout(desc: MoeDesc, max_tokens_per_rank: int, topk_idx, lay: dict, out: dict,
                      stream=None) -> Prepared:
    d = desc.c()
    ptrs = _vps(topk_idx, lay["slot_of"], lay["expert_offset"], lay["src_of_slot"],
                out["ll_slot_of"], out["src_info"], out["layout_range"], out["recv_count"])
    args = (ctypes.byref(d), ctypes.c_int32(max_tokens_per_rank), *ptrs,
            ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_ll_layout", args, (d, topk_idx, lay, out))


def prepare_dispatch_ll(desc: MoeDesc, hidden, scales, ll_slot_of, x_out, scales_out,
                        stream=None) -> Prepared:
    d = desc.c()
    sb = scales_out.numel() * scales_out.element_size() if scales_out is not None else 0
    args = (ctypes.byref(d), *_vps(hidden, scales, ll_slot_of, x_out),
            ctypes.c_size_t(x_out.numel() * x_out.element_size()), ctypes.c_void_p(_ptr(scales_out)),
            ctypes.c_size_t(sb), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_dispatch_ll", args, (d, hidden, scales, ll_slot_of, x_out, scales_out))


def prepare_rank_layout(desc: MoeDesc, lay: dict, expert_alignment: int, out: dict,
                        stream=None) -> Prepared:
    d = desc.c()
    args = (ctypes.byref(d), *_vps(lay["is_token_in_rank"], lay["tokens_per_rank"],
                                   lay["tokens_per_expert"]),
            ctypes.c_int32(expert_alignment),
            *_vps(out["send_head"], out.get("recv_src_idx"), out["recv_offset"],
                  out["recv_tokens_per_expert"]),
            ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_rank_layout", args, (d, lay, out))


def prepare_dispatch_ranks(desc: MoeDesc, topk_idx, topk_weights, hidden, scales, send_head,
                           records, stream=None) -> Prepared:
    d = desc.c()
    args = (ctypes.byref(d), *_vps(topk_idx, topk_weights, hidden, scales, send_head, records),
            ctypes.c_size_t(records.numel() * records.element_size()),
            ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_dispatch_ranks", args, (d, topk_idx, topk_weights, hidden, scales,
                                                 send_head, records))


def prepare_layout_ll_dispatch(desc: MoeDesc, max_tokens_per_rank: int, topk_idx, hidden, scales, out: dict,
                               ll_out: dict, workspace, x_out, scales_out, stream=None) -> Prepared:
    """moe_layout_ll and moe_dispatch_ll in one call (see include/moe.h)."""
    d = desc.c()
    sb = scales_out.numel() * scales_out.element_size() if scales_out is not None else 0
    args = (ctypes.byref(d),
            *_vps(topk_idx, hidden, scales, out["tokens_per_expert"], out["tokens_per_rank"],
                  out["is_token_in_rank"], out["expert_offset"], out["rank_offset"], out["slot_of"],
                  out.get("src_of_slot")),
            ctypes.c_int32(max_tokens_per_rank),
            *_vps(ll_out["ll_slot_of"], ll_out["src_info"], ll_out["layout_range"], ll_out["recv_count"],
                  workspace),
            ctypes.c_size_t(workspace.numel()), ctypes.c_void_p(_ptr(x_out)),
            ctypes.c_size_t(x_out.numel() * x_out.element_size()), ctypes.c_void_p(_ptr(scales_out)),
            ctypes.c_size_t(sb), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_layout_ll_dispatch", args, (d, topk_idx, hidden, scales, out, ll_out, workspace,
                                                     x_out, scales_out))


def prepare_combine_gather_ranks(desc: MoeDesc, recv_out, send_head, out, stream=None) -> Prepared:
    d = desc.c()
    rows = recv_out.numel() // max(desc.hidden, 1)
    args = (ctypes.byref(d), ctypes.c_void_p(_ptr(recv_out)), ctypes.c_int64(rows),
            *_vps(send_head, out), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_combine_gather_ranks", args, (d, recv_out, send_head, out))


def prepare_combine(desc: MoeDesc, mode: int, expert_out, topk_idx, topk_weights, slot_of, out,
                    stream=None) -> Prepared:
    d = desc.c()
    rows = expert_out.numel() // max(desc.hidden, 1)
    ptrs = _vps(topk_idx, topk_weights, slot_of, out)
    args = (ctypes.byref(d), ctypes.c_int(mode), ctypes.c_void_p(_ptr(expert_out)),
            ctypes.c_int64(rows), *ptrs, ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_combine", args, (d, expert_out, topk_idx, topk_weights, slot_of, out))


def prepare_combine_backward(desc: MoeDesc, grad_out, topk_weights, slot_of, expert_out, rows: int,
                             grad_expert_out, grad_weights, stream=None) -> Prepared:
    d = desc.c()
    args = (ctypes.byref(d), *_vps(grad_out, topk_weights, slot_of, expert_out),
            ctypes.c_int64(rows), *_vps(grad_expert_out, grad_weights),
            ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_combine_backward", args, (d, grad_out, topk_weights, slot_of, expert_out,
                                                   grad_expert_out, grad_weights))


def prepare_dispatch_backward(desc: MoeDesc, grad_in, slot_of, grad_hidden, stream=None) -> Prepared:
    d = desc.c()
    rows = grad_in.numel() // max(desc.hidden, 1)
    args = (ctypes.byref(d), ctypes.c_void_p(_ptr(grad_in)), ctypes.c_int64(rows),
            *_vps(slot_of, grad_hidden), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_dispatch_backward", args, (d, grad_in, slot_of, grad_hidden))


def prepare_combine_norm(desc: MoeDesc, mode: int, expert_out, topk_idx, topk_weights, slot_of,
                         residual_in, gamma, eps: float, normed_out, residual_out,
                         stream=None) -> Prepared:
    d = desc.c()
    rows = expert_out.numel() // max(desc.hidden, 1)
    args = (ctypes.byref(d), ctypes.c_int(mode), ctypes.c_void_p(_ptr(expert_out)),
            ctypes.c_int64(rows), *_vps(topk_idx, topk_weights, slot_of, residual_in, gamma),
            ctypes.c_float(eps), *_vps(normed_out, residual_out), ctypes.c_void_p(_stream(stream)))
    return Prepared("moe_combine_norm", args, (d, expert_out, topk_idx, topk_weights, slot_of,
                                               residual_in, gamma, normed_out, residual_out))


def exported_symbols() -> list[str]:
    return ["moe_strerror", "moe_record_layout", "moe_workspace_size", "moe_layout",
            "moe_layout_status", "moe_dispatch", "moe_combine", "moe_pack_record",
            "moe_unpack_record", "moe_layout_noalloc", "moe_combine_norm", "moe_slot_layout",
            "moe_pack_slots", "moe_unpack_slots", "moe_mask_topk_ids", "moe_rank_layout",
            "moe_dispatch_ranks", "moe_combine_gather_ranks", "moe_ll_layout",
            "moe_dispatch_ll", "moe_combine_backward", "moe_dispatch_backward",
            "moe_combine_gather_ranks_backward", "moe_layout_dispatch", "moe_device_status",
            "moe_layout_ranks", "moe_layout_ll", "moe_layout_ll_dispatch", "moe_set_wait_limit_ns"]
