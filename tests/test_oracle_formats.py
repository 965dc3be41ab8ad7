"""Pins of the oracle's number formats and quantisers against things other
than the oracle itself: torch's own conversions (independent library code),
values fixed by the format definitions (OCP FP8 e4m3fn, FP4 e2m1), closed-form
error bounds and special cases."""
import numpy as np
import pytest
import torch

import oracle
from format_cases import NVFP4_MIDPOINT_SCALES, nvfp4_midpoint_group

# ---------------------------------------------------------------- BF16 -----


def _bf16_torch(f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(f32.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_round_matches_torch_on_random_and_ties():
    g = np.random.default_rng(0)
    vals = [g.standard_normal(2000).astype(np.float32),
            (g.standard_normal(500) * 1e30).astype(np.float32),
            (g.standard_normal(500) * 1e-38).astype(np.float32)]  # subnormals
    # exact midpoints between consecutive BF16 values, both parities
    base = g.integers(0x0080, 0x7f00, size=500).astype(np.uint32)
    mids = ((base << 16) | 0x8000).view(np.float32)
    vals += [mids, -mids, np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, 1e-45], np.float32)]
    f = np.concatenate(vals)
    got = oracle.f32_to_bf16_array(f)
    np.testing.assert_array_equal(got, _bf16_torch(f))


def test_bf16_widen_is_exact():
    codes = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    got = np.array([oracle.bf16_to_f32(int(c)) for c in codes], np.float32)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]) == np.isnan(ref[~finite]))


# ---------------------------------------------------------------- e4m3 -----


def test_e4m3_decode_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)], np.float32)
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.all(np.isnan(got[nan]))
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_in_range():
    # torch converts with round-to-nearest-even but turns |x| >= 464 into NaN
    # instead of saturating, so compare inside (-464, 464) and check the
    # saturation separately.
    finite = [oracle.e4m3_value(c) for c in range(256) if c not in (0x7F, 0xFF)]
    finite = np.unique(np.array(finite, np.float32))
    mids = ((finite[1:].astype(np.float64) + finite[:-1]) / 2).astype(np.float32)
    g = np.random.default_rng(1)
    rnd = np.concatenate([g.uniform(-460, 460, 3000), g.standard_normal(3000) * 2.0 ** -8,
                          g.standard_normal(2000)]).astype(np.float32)
    x = np.concatenate([finite, mids, np.nextafter(mids, np.float32(np.inf)),
                        np.nextafter(mids, np.float32(-np.inf)), rnd]).astype(np.float32)
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], np.uint8)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("x,code", [(1.0, 0x38), (448.0, 0x7E), (449.0, 0x7E), (1e6, 0x7E),
                                    (-1e6, 0xFE), (float("inf"), 0x7E), (2.0 ** -9, 0x01),
                                    (2.0 ** -10, 0x00), (1.5 * 2.0 ** -10, 0x01),
                                    (1.0625, 0x38), (1.1875, 0x3A), (-0.0, 0x80)])
def test_e4m3_encode_special_values(x, code):
    # 1.0 = 0.0111.000 (bias 7); 448 = 0.1111.110 is the largest finite value,
    # beyond it the encoder saturates; 2^-9 is the smallest subnormal; 2^-10 is
    # a tie between 0 and 2^-9 and goes to the even code 0; 1.0625 is a tie
    # between 1.0 (even) and 1.125; 1.1875 between 1.125 and 1.25 (even).
    assert oracle.e4m3_encode(x) == code


# ---------------------------------------------------------------- e2m1 -----

E2M1_SPEC = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX FP4 E2M1 magnitudes


def test_e2m1_decode_matches_spec_table():
    for c in range(16):
        v = E2M1_SPEC[c & 7]
        got = oracle.e2m1_value(c)
        assert got == (-v if c & 8 else v)
        assert np.signbit(got) == bool(c & 8)


@pytest.mark.parametrize("x,code", [
    (0.0, 0), (0.25, 0), (0.2500001, 1), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4),
    (3.5, 6), (5.0, 6), (5.0001, 7), (6.0, 7), (7.0, 7), (1e9, 7), (-0.25, 8), (-0.1, 8),
    (-0.75, 10), (-5.0, 14), (-100.0, 15), (0.5, 1), (1.5, 3), (3.0, 5), (4.0, 6)])
def test_e2m1_encode_midpoints_and_saturation(x, code):
    # Midpoints between neighbouring magnitudes go to the even code; beyond 6
    # the encoder saturates; the sign bit is kept for values that round to 0.
    assert oracle.e2m1_encode(x) == code


def test_e2m1_encode_is_monotone_and_idempotent():
    xs = np.linspace(-8, 8, 4001).astype(np.float32)
    vals = np.array([oracle.e2m1_value(oracle.e2m1_encode(float(x))) for x in xs])
    assert np.all(np.diff(vals) >= 0)
    for c in range(16):
        if c == 8:
            continue
        assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c


# ------------------------------------------------------------- FP8 group ----

def _bf16(f):
    return (np.asarray(f, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_fp8_group_matches_torch_cast_and_bound():
    g = np.random.default_rng(2)
    for trial in range(50):
        x = _bf16(g.standard_normal(128) * (10.0 ** g.uniform(-3, 3)))
        q, scale = oracle.fp8_group(x)
        xf = oracle.bf16_to_f32_array(x)
        amax = np.float32(np.max(np.abs(xf)))
        a = max(amax, np.float32(1e-4))
        assert np.float32(scale) == np.float32(a) / np.float32(448.0)
        inv = np.float32(448.0) / np.float32(a)
        ref = torch.from_numpy((xf * inv).astype(np.float32)).to(torch.float8_e4m3fn)
        np.testing.assert_array_equal(q, ref.view(torch.uint8).numpy())
        deq = np.array([oracle.e4m3_value(c) for c in q], np.float64) * scale
        # half a step of e4m3: 2^-4 relative for normals, 2^-10 * scale below
        bound = np.maximum(np.abs(xf) * 2.0 ** -4, scale * 2.0 ** -10) * (1 + 2.0 ** -18)
        assert np.all(np.abs(deq - xf) <= bound)


def test_fp8_group_special_cases():
    q, scale = oracle.fp8_group(np.zeros(128, np.uint16))
    assert np.all(q == 0) and np.float32(scale) == np.float32(1e-4) / np.float32(448)
    x = np.zeros(128, np.float32)
    x[5], x[77] = 3.0, -3.0
    q, scale = oracle.fp8_group(_bf16(x))
    assert q[5] == 0x7E and q[77] == 0xFE and np.all(np.delete(q, [5, 77]) == 0)


# ----------------------------------------------------------- NVFP4 group ----

def test_nvfp4_group_bound_and_packing():
    g = np.random.default_rng(3)
    for trial in range(200):
        xf = (g.standard_normal(16) * (10.0 ** g.uniform(-2, 2))).astype(np.float32)
        x = _bf16(xf)
        xf = oracle.bf16_to_f32_array(x).astype(np.float64)
        q, sc = oracle.nvfp4_group(x)
        d = oracle.e4m3_value(sc)
        amax = np.max(np.abs(xf))
        # the scale is e4m3(amax/6): within half an e4m3 step of amax/6
        assert abs(d - amax / 6) <= max(amax / 6 * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
        codes = np.empty(16, np.uint8)
        codes[0::2], codes[1::2] = q & 15, q >> 4
        deq = np.array([oracle.e2m1_value(c) for c in codes]) * d
        # Inside the grid the worst half-step is 1 (between 4 and 6), so the
        # error is at most d; beyond 6*d the code saturates at 6 and the error
        # is |x| - 6d <= amax - 6d. That happens when e4m3 rounded the scale
        # down (by at most 2^-4 for normal scales, more for subnormal ones).
        bound = max(d, amax - 6 * d) * (1 + 1e-6)
        assert np.all(np.abs(deq - xf) <= bound)
        if d >= 2.0 ** -6:  # normal e4m3 scale: amax/d lies in [5.6, 6.4]
            assert 5.6 <= amax / d <= 6.4
            i = int(np.argmax(np.abs(xf)))
            assert (codes[i] & 7) in (6, 7)


def test_nvfp4_group_special_cases():
    q, sc = oracle.nvfp4_group(np.zeros(16, np.uint16))
    assert sc == 0 and np.all(q == 0)
    x = np.zeros(16, np.float32)
    x[0], x[3] = 6.0, -1.5  # amax/6 = 1 -> scale code 0x38, d = 1
    q, sc = oracle.nvfp4_group(_bf16(x))
    assert sc == 0x38
    assert q[0] == 0x07            # element 0 in the low nibble, element 1 (0) high
    assert q[1] == (0xB << 4)      # element 3 = -1.5 -> code 8|3 in the high nibble
    assert np.all(q[2:] == 0)


@pytest.mark.parametrize("scale_code", NVFP4_MIDPOINT_SCALES)
def test_nvfp4_divides_by_the_scale(scale_code):
    """The NVFP4 reading quantises x / d, one IEEE division. With d = 1.875 *
    2^e the quotient of m*d is exactly the midpoint m, which must go to the
    even code; multiplying by an fp32 reciprocal 1/d instead lands just off
    the midpoint and picks the other neighbour for some of these elements,
    so this group tells the two forms apart."""
    x, want = nvfp4_midpoint_group(scale_code)
    q, sc = oracle.nvfp4_group(x)
    assert sc == scale_code
    codes = np.empty(16, np.uint8)
    codes[0::2], codes[1::2] = q & 15, q >> 4
    for i, c in want.items():
        assert codes[i] == c, (i, codes[i], c)
    # the group discriminates: x * fl(1/d) rounds differently at >= 1 midpoint
    d = np.float32(oracle.e4m3_value(scale_code))
    inv = np.float32(1.0) / d
    xf = oracle.bf16_to_f32_array(x)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    differs = 0
    for i in range(16):
        v = float(np.float32(xf[i]) * inv)
        a = abs(v)
        dist = np.abs(grid - a)
        nearest = np.flatnonzero(dist == dist.min())
        code = int(nearest[0] if len(nearest) == 1 else nearest[nearest % 2 == 0][0])
        if a >= 6.0:
            code = 7
        code |= 8 if v < 0 or (v == 0 and np.signbit(v)) else 0
        differs += code != want[i]
    assert differs >= 1
