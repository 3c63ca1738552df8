"""Pins for the oracle's number formats: E4M3 (float8_e4m3fn), E8M0, the rceil
scale exponent and BF16 rounding.

Each check compares the oracle with something other than itself: PyTorch's
float8_e4m3fn / bfloat16 conversions (library routines), exact rational
arithmetic with Python's Fraction (brute force), or closed-form invariants
of the formats.  E4M3 is the element type the MindSpeed RFC fixes
(section 3.3.1, "dtype 统一为 E4M3"; section 3.5.2.3, float8_e4m3fn); the
E8M0 power-of-two scale and the rceil rule come from the torchtitan-npu
tutorial ("每32个元素共享一个 e8m0 scale"; log keyword "mxfp8_rceil").
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _torch_e4m3_value(code: int) -> float:
    t = torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn)
    return float(t.to(torch.float32).item())


def test_e4m3_decode_all_codes_match_torch(orc):
    vals = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    for c in range(256):
        ref = _torch_e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert math.isnan(vals[c]) and math.isnan(ref)
        else:
            assert vals[c] == ref, (c, vals[c], ref)
            assert math.copysign(1.0, vals[c]) == math.copysign(1.0, ref)


def test_e4m3_closed_form_extremes(orc):
    d = orc.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x00, 0x80], dtype=np.uint8))
    assert d[0] == 448.0            # largest finite, S.1111.110
    assert d[1] == 2.0 ** -6        # smallest normal
    assert d[2] == 2.0 ** -9        # smallest subnormal
    assert d[3] == 0.0 and math.copysign(1, d[4]) == -1.0


def test_e4m3_roundtrip_every_finite_code(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = orc.e4m3_encode(orc.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def _finite_pos_table(orc):
    return [float(v) for v in orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))]


def _brute_nearest_code(a: float, table) -> int:
    """Nearest non-negative finite code by exhaustive search; ties -> even code."""
    best = None
    for c, v in enumerate(table):
        d = abs(Fraction(a) - Fraction(v))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_e4m3_midpoints_round_to_even(orc):
    table = _finite_pos_table(orc)
    mids, expect = [], []
    for c in range(0x7E):
        mid = (table[c] + table[c + 1]) / 2.0          # exact in double
        mids += [mid, -mid]
        even = c if c % 2 == 0 else c + 1
        expect += [even, even | 0x80]
    got = orc.e4m3_encode(np.array(mids))
    assert np.array_equal(got, np.array(expect, dtype=np.uint8))


def test_e4m3_encode_matches_brute_force_and_torch(orc):
    table = _finite_pos_table(orc)
    rng = random.Random(7)
    vals = []
    for _ in range(3000):
        e = rng.uniform(-12, 9)
        vals.append(float(np.float32(rng.choice([-1, 1]) * min(448.0, 2.0 ** e))))
    vals += [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -12]
    got = orc.e4m3_encode(np.array(vals))
    for v, g in zip(vals, got):
        want = _brute_nearest_code(abs(v), table) | (0x80 if math.copysign(1, v) < 0 else 0)
        assert g == want, (v, g, want)
    # PyTorch's float32 -> float8_e4m3fn conversion rounds to nearest even
    # (it does not saturate above 448, so only in-range values are compared).
    f32 = np.array(vals, dtype=np.float32)
    assert np.all(f32.astype(np.float64) == np.array(vals))
    ref = torch.from_numpy(f32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e4m3_saturates(orc):
    big = np.array([448.0000001, 464.0, 480.0, 1e6, 1e300, math.inf])
    assert np.all(orc.e4m3_encode(big) == 0x7E)
    assert np.all(orc.e4m3_encode(-big) == 0xFE)
    n = orc.e4m3_encode(np.array([math.nan]))
    assert n[0] & 0x7F == 0x7F


def test_e8m0_decode(orc):
    assert orc.e8m0_decode(127) == 1.0
    assert orc.e8m0_decode(0) == 2.0 ** -127
    assert orc.e8m0_decode(254) == 2.0 ** 127
    assert math.isnan(orc.e8m0_decode(255))


def _bf16_exact(bits: int) -> Fraction:
    E, m = (bits >> 7) & 0xFF, bits & 0x7F
    if E == 0:
        return Fraction(m) * Fraction(2) ** -133
    return Fraction(128 + m) * Fraction(2) ** (E - 134)


def _rceil_exact(v: Fraction) -> int:
    """Smallest integer e with 448 * 2^e >= v, clamped to [-127, 127]."""
    if v == 0:
        return -127
    e = math.floor(math.log2(float(v) / 448.0)) - 2
    while Fraction(448) * Fraction(2) ** e < v:
        e += 1
    assert Fraction(448) * Fraction(2) ** (e - 1) < v
    return max(-127, min(127, e))


def test_rceil_every_positive_bf16(orc):
    """The frexp rule equals ceil(log2(amax/448)) evaluated exactly, for every
    positive finite BF16 value used as amax."""
    for bits in range(1, 0x7F80):
        v = _bf16_exact(bits)
        assert orc.rceil_exponent(float(v)) == _rceil_exact(v), hex(bits)
    assert orc.rceil_exponent(0.0) == -127


def test_rceil_boundaries(orc):
    # amax = 448 * 2^j is exactly representable: e = j (no overflow, minimal).
    for j in range(-100, 100):
        assert orc.rceil_exponent(448.0 * 2.0 ** j) == j
        # just above 448*2^j the exponent must step up
        assert orc.rceil_exponent(450.0 * 2.0 ** j) == j + 1


def _bf16_rne_exact(x: float) -> int:
    """BF16 bits of the value nearest to x, ties to even, by exact arithmetic."""
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(Fraction(x))
    if a == 0:
        return sign
    p = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** p > a:
        p -= 1
    lead = max(p, -126)
    q = Fraction(2) ** (lead - 7)
    r = round(a / q) * q                # Fraction.__round__ is half-to-even
    if r > Fraction(255) * Fraction(2) ** 120:
        return sign | 0x7F80
    f = np.array([float(r)], dtype=np.float32)
    assert Fraction(float(f[0])) == r
    return sign | int(f.view(np.uint32)[0] >> 16)


def test_bf16_rounding_matches_exact_and_torch(orc):
    rng = random.Random(11)
    vals = []
    for _ in range(4000):
        vals.append(rng.choice([-1, 1]) * rng.uniform(0.5, 1.0) * 2.0 ** rng.randint(-140, 127))
    # double-rounding traps: exactly-representable midpoint plus a tiny bit
    vals += [1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8 + 2 ** -40),
             2.0 ** -134, 2.0 ** -134 * 1.0000001, 3.3e38, 3.4e38, 0.0, -0.0]
    got = orc.bf16_from_double(np.array(vals))
    for v, g in zip(vals, got):
        assert g == _bf16_rne_exact(v), (v, hex(g))
    assert got[-10] == 0x3F81          # 1 + 2^-8 + 2^-30 rounds up in one step
    # float32-representable inputs: PyTorch's float32 -> bfloat16 (RNE) agrees
    f32 = np.array(vals[:4000], dtype=np.float32)
    f32 = f32[np.isfinite(f32)]
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_from_double(f32.astype(np.float64)), ref)
