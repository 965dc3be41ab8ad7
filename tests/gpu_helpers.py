"""Host <-> device conversions shared by the GPU tests (no method arithmetic)."""
import numpy as np
import torch

DEV = torch.device("cuda:0")


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def dev_bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16, dtype=np.uint16).view(np.int16)).to(DEV).view(torch.bfloat16)


def host_bf16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    return t.cpu().numpy()


def bf16_f64(u16):
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_combine_close(got_u16, ref_u16, what=""):
    """The contract tolerance |gpu - ref| <= 1e-2 * max(1, |ref|)."""
    g, r = bf16_f64(got_u16), bf16_f64(ref_u16)
    bad = np.abs(g - r) > 1e-2 * np.maximum(1.0, np.abs(r))
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of tolerance"
