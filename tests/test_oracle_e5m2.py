"""Pins for the oracle's E5M2 destination type (MindSpeed RFC section 3.5.2.3:
dst_type E4M3 or E5M2).  E5M2 is OCP float8_e5m2: bias 15, Inf and NaN at
exponent 31, largest finite 57344; conversion rounds to nearest even and
saturates; the rceil rule uses 57344 in place of 448.

Checked against PyTorch's float8_e5m2 (decode of every code, RNE encode of
in-range values), exhaustive nearest-code search, exact rationals for rceil
on every positive BF16 value, and the invariants rceil implies.
"""
import math
from fractions import Fraction

import numpy as np
import torch


def _torch_e5m2(code):
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e5m2).float().item())


def test_e5m2_decode_all_codes_match_torch(orc):
    vals = orc.e5m2_decode(np.arange(256, dtype=np.uint8))
    for c in range(256):
        ref = _torch_e5m2(c)
        if math.isnan(ref):
            assert math.isnan(vals[c])
        else:
            assert vals[c] == ref and math.copysign(1, vals[c]) == math.copysign(1, ref), c


def _finite_codes():
    return [c for c in range(256) if ((c >> 2) & 0x1F) != 0x1F]


def test_e5m2_roundtrip_midpoints_and_saturation(orc):
    codes = np.array(_finite_codes(), dtype=np.uint8)
    assert np.array_equal(orc.e5m2_encode(orc.e5m2_decode(codes)), codes)
    pos = [float(v) for v in orc.e5m2_decode(np.arange(0x7C, dtype=np.uint8))]  # 0 .. 57344
    mids = np.array([(pos[c] + pos[c + 1]) / 2 for c in range(0x7B)])
    even = np.array([c if c % 2 == 0 else c + 1 for c in range(0x7B)], dtype=np.uint8)
    assert np.array_equal(orc.e5m2_encode(mids), even)
    assert np.array_equal(orc.e5m2_encode(-mids), even | 0x80)
    big = np.array([57344.5, 61440.0, 1e9, math.inf])
    assert np.all(orc.e5m2_encode(big) == 0x7B) and np.all(orc.e5m2_encode(-big) == 0xFB)


def test_e5m2_encode_matches_brute_force_and_torch(orc):
    rng = np.random.default_rng(3)
    v = (rng.choice([-1.0, 1.0], 3000) * np.exp2(rng.uniform(-18, 15.8, 3000))).astype(np.float32)
    v = v.astype(np.float64)
    got = orc.e5m2_encode(v)
    table = [float(x) for x in orc.e5m2_decode(np.arange(0x7C, dtype=np.uint8))]
    for x, g in zip(v[:600], got[:600]):
        a = Fraction(abs(float(x)))
        best = min(range(len(table)), key=lambda c: (abs(a - Fraction(table[c])), c % 2))
        assert g == (best | (0x80 if x < 0 else 0)), x
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def _bf16_exact(bits):
    E, m = (bits >> 7) & 0xFF, bits & 0x7F
    return Fraction(m) * Fraction(2) ** -133 if E == 0 else Fraction(128 + m) * Fraction(2) ** (E - 134)


def test_rceil_e5m2_every_positive_bf16(orc):
    for bits in range(1, 0x7F80, 3):
        v = _bf16_exact(bits)
        e = math.floor(math.log2(float(v) / 57344.0)) - 2
        while Fraction(57344) * Fraction(2) ** e < v:
            e += 1
        assert orc.rceil_exponent_fmt(float(v), 1) == max(-127, min(127, e)), hex(bits)
    assert orc.rceil_exponent_fmt(0.0, 1) == -127
    assert orc.rceil_exponent_fmt(448.0, 0) == 0 and orc.rceil_exponent_fmt(57344.0, 1) == 0


def test_quant_rows_e5m2_invariants(orc):
    g = torch.Generator().manual_seed(9)
    x = torch.randn(64, 256, generator=g, dtype=torch.float64)
    x = x * torch.pow(2.0, torch.randint(-60, 60, (64, 8, 1), generator=g).double()).repeat_interleave(32, 2).view(64, 256)
    xb = x.float().to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.quant_rows_fmt(bits, 1)
    xv = orc.bf16_to_double(bits).reshape(64, 8, 32)
    e = s.astype(np.int64) - 127
    scaled = xv * np.power(2.0, -e)[..., None]
    assert np.all(np.abs(scaled) <= 57344.0)
    qv = orc.e5m2_decode(q).reshape(64, 8, 32)
    qmax = np.abs(qv).max(axis=2)
    assert np.all((qmax >= 28672.0) & (qmax <= 57344.0))
    ref = torch.from_numpy(scaled.reshape(64, 256).astype(np.float32)).to(torch.float8_e5m2).view(torch.uint8)
    assert np.array_equal(ref.numpy(), q)
    # E4M3 path of the same entry point is the pinned default quantizer
    q4, s4 = orc.quant_rows_fmt(bits, 0)
    q0, s0 = orc.quant_rows(bits)
    assert np.array_equal(q4, q0) and np.array_equal(s4, s0)
