"""Constructed inputs and per-row expectations shared by the format tests.

Test infrastructure: builds input groups from the format definitions and asks
the oracle's group quantisers for one row's payload bytes; it holds no part
of the CUDA path."""
import numpy as np

import oracle

# e4m3 codes with mantissa 7: d = 1.875 * 2^e, whose fp32 reciprocal is inexact
NVFP4_MIDPOINT_SCALES = [0x17, 0x2F, 0x37, 0x3F, 0x4F, 0x67]


def nvfp4_midpoint_group(scale_code: int) -> tuple[np.ndarray, dict]:
    """A group of 16 whose e4m3 scale is d = value(scale_code) and whose
    elements sit exactly on e2m1 midpoints after division by d.

    Element 0 is 6d (so amax / 6 = d exactly); the others are m*d for the
    midpoints m in {1.25, 2.5, 5} (both signs) and a few grid values. Returns
    the BF16 patterns and {element index: the expected e2m1 code}."""
    d = oracle.e4m3_value(scale_code)
    # the midpoint between two e2m1 magnitudes goes to the code with an even
    # index (round half to even on the code grid {0,.5,1,1.5,2,3,4,6}):
    # 1.25 -> 1 (code 2), 2.5 -> 2 (code 4), 5 -> 4 (code 6)
    elems = [(6.0, 7), (1.25, 2), (2.5, 4), (5.0, 6), (-1.25, 8 | 2), (-2.5, 8 | 4), (-5.0, 8 | 6),
             (0.75, 2), (1.75, 4), (3.5, 6), (-0.25, 8 | 0), (1.0, 2), (3.0, 5), (0.0, 0),
             (5.0, 6), (2.5, 4)]
    xf = np.array([m * d for m, _ in elems], np.float32)
    bits = xf.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "every element must be an exact BF16 value"
    return (bits >> 16).astype(np.uint16), {i: c for i, (_, c) in enumerate(elems)}


def quantised_row(x_bf16: np.ndarray, out_kind: int):
    """The payload and scale bytes of one BF16 row, group by group, from the
    oracle's group quantisers (not from its dispatch). Scales are None for
    BF16 pass-through."""
    if out_kind == oracle.BF16:
        return x_bf16.view(np.uint8).copy(), None
    pay, sc = [], []
    if out_kind == oracle.FP8_E4M3_B128:
        for g in range(0, x_bf16.size, 128):
            q, s = oracle.fp8_group(x_bf16[g:g + 128])
            pay.append(q)
            sc.append(np.frombuffer(np.float32(s).tobytes(), np.uint8))
    elif out_kind == oracle.NVFP4_B16:
        for g in range(0, x_bf16.size, 16):
            q, s = oracle.nvfp4_group(x_bf16[g:g + 16])
            pay.append(q)
            sc.append(np.uint8([s]))
    elif out_kind == oracle.FP8_E4M3_UE8M0:
        for g in range(0, x_bf16.size, 128):
            q, s = oracle.fp8_ue8m0_group(x_bf16[g:g + 128])
            pay.append(q)
            sc.append(np.uint8([s]))
    else:
        raise ValueError(out_kind)
    return np.concatenate(pay), np.concatenate(sc)
