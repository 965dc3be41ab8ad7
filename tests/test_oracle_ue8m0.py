"""Pins of the oracle's FP8 e4m3 quantiser with power-of-two UE8M0 scales:
the scale is the least power of two >= max(amax, 1e-4)/448 (checked against
an exact rational comparison), no value saturates, the codes equal torch's
float8_e4m3fn cast of the exactly scaled values, the byte is the biased
exponent, decoding stays within half an e4m3 step, and the record layout,
dispatch and identity expert carry it through."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth


def _f(b):
    return oracle.bf16_to_f32_array(np.asarray(b, np.uint16)).astype(np.float64)


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("seed,scale", [(1, 1.0), (2, 1e-3), (3, 300.0), (4, 1e-6), (5, 3e30)])
def test_scale_is_the_least_power_of_two_at_or_above_a_over_448(seed, scale):
    g = np.random.default_rng(seed)
    for _ in range(20):
        x = synth.bf16_normal(g, (128,), scale=scale)
        q, byte = oracle.fp8_ue8m0_group(x)
        e = byte - 127
        amax = float(np.abs(_f(x)).max())
        a = max(np.float32(amax), np.float32(1e-4))
        v = Fraction(float(np.float32(a) / np.float32(448.0)))  # the fp32 quotient, exactly
        assert Fraction(2) ** e >= v and Fraction(2) ** (e - 1) < v
        # codes: torch's cast of x * 2^-e (exact scaling), no saturation needed
        scaled = (_f(x) * 2.0 ** -e).astype(np.float32)
        assert np.abs(scaled).max() <= 448.0 * (1 + 2 ** -23)
        np.testing.assert_array_equal(q, _torch_e4m3(scaled))


def test_decode_error_bound_and_exact_powers():
    g = np.random.default_rng(6)
    x = synth.bf16_normal(g, (128,), scale=5.0)
    q, byte = oracle.fp8_ue8m0_group(x)
    deq = np.array([oracle.e4m3_value(int(c)) for c in q]) * 2.0 ** (byte - 127)
    xf = _f(x)
    # e4m3 keeps 3 mantissa bits: relative step 2^-3 for normals, absolute
    # 2^-9 * scale below 2^-6 * scale
    tol = np.maximum(np.abs(xf) * 2.0 ** -4, 2.0 ** -10 * 2.0 ** (byte - 127)) * 1.0001
    assert np.all(np.abs(deq - xf) <= tol)
    # a group whose amax/448 is itself a power of two keeps that exponent
    y = np.zeros(128, np.uint16)
    y[0] = 0x43E0  # 448.0 -> v = 1 -> e = 0
    q2, b2 = oracle.fp8_ue8m0_group(y)
    assert b2 == 127 and q2[0] == 0x7E  # e4m3 448 = 0b0_1111_110
    # all zeros: a = 1e-4, v = 1e-4/448 in [2^-23, 2^-22) -> e = -22
    q3, b3 = oracle.fp8_ue8m0_group(np.zeros(128, np.uint16))
    assert b3 == 127 - 22 and not q3.any()


def test_record_dispatch_and_identity_expert_carry_ue8m0():
    k, h = 8, 512
    lay = oracle.record_layout(k, h, oracle.BF16, oracle.FP8_E4M3_UE8M0)
    assert lay["payload_bytes"] == h and lay["scale_bytes"] == h // 128
    assert lay["record_bytes"] == 16 + 32 + 32 + 512 + 16  # 4 scale bytes padded to 16
    c = synth.prefill_case(seed=7, n=12, hidden=h)
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    L = oracle.layout(ids, 256, 8)
    P = L["num_pairs"]
    rec = oracle.dispatch(ids, w, x, None, L["slot_of"], P, oracle.BF16, oracle.FP8_E4M3_UE8M0, h)
    y = oracle.identity_expert(rec, k, h, oracle.FP8_E4M3_UE8M0)
    for s in range(P):
        t = int(rec[s, :4].view(np.int32)[0])
        for g in range(h // 128):
            q, byte = oracle.fp8_ue8m0_group(x[t, g * 128:(g + 1) * 128])
            np.testing.assert_array_equal(rec[s, lay["off_payload"] + g * 128:lay["off_payload"] + (g + 1) * 128], q)
            assert rec[s, lay["off_scales"] + g] == byte
        assert not rec[s, lay["off_scales"] + h // 128:].any()  # padding zero
        want = [oracle.e4m3_value(int(cq)) * 2.0 ** (int(rec[s, lay["off_scales"] + i // 128]) - 127)
                for i, cq in enumerate(rec[s, lay["off_payload"]:lay["off_payload"] + h])]
        want16 = torch.tensor(want, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(y[s], want16)
