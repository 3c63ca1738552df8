"""Pins for the oracle's block-scaled GEMM and grouped GEMM.

The FP8 matmul consumes the E4M3 payloads and their E8M0 scales and returns
BF16 (torchtitan-npu tutorial, "MXFP8 与 HiF8 架构原理速览": "输出恢复为 BF16";
the MoE expert layers use the grouped matmul).  The oracle sums exact
dequantized products in FP64 and rounds once to BF16.  Checked here against
exact rational arithmetic (Python Fraction) on tiny shapes, against a plain
float64 matmul in the special case where every sum is exactly representable,
and, for the grouped GEMM, against per-expert slices.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch


def _e4m3_exact(codes: np.ndarray):
    """Exact values of E4M3 codes through PyTorch's float8_e4m3fn decode."""
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)
    return t.numpy()


def _rand_operand(rng, rows, K, spread):
    codes = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C     # no NaN codes in the payload
    scales = rng.integers(127 - spread, 127 + spread + 1, size=(rows, K // 32), dtype=np.uint8)
    return codes, scales


def _bf16_rne_exact(v: Fraction) -> int:
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return 0
    p = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** p > a:
        p -= 1
    q = Fraction(2) ** (max(p, -126) - 7)
    r = round(a / q) * q
    if r > Fraction(255) * Fraction(2) ** 120:
        return sign | 0x7F80
    f = np.array([float(r)], dtype=np.float32)
    return sign | int(f.view(np.uint32)[0] >> 16)


@pytest.mark.parametrize("M,N,K,spread,seed", [(5, 7, 64, 4, 0), (8, 3, 128, 20, 1),
                                               (3, 8, 256, 60, 2), (1, 1, 32, 0, 3)])
def test_gemm_matches_exact_rational(orc, M, N, K, spread, seed):
    rng = np.random.default_rng(seed)
    qa, sa = _rand_operand(rng, M, K, spread)
    qb, sb = _rand_operand(rng, N, K, spread)
    a = orc.dequant_rows(qa, sa)
    b = orc.dequant_rows(qb, sb)
    va, vb = _e4m3_exact(qa), _e4m3_exact(qb)
    # dequantization is exact: code value times 2^(scale-127)
    for i in range(M):
        for k in range(K):
            assert Fraction(a[i, k]) == Fraction(va[i, k]) * Fraction(2) ** (int(sa[i, k // 32]) - 127)
    y = orc.gemm(a, b)
    logged = 0
    for i in range(M):
        for j in range(N):
            exact = sum((Fraction(a[i, k]) * Fraction(b[j, k]) for k in range(K)), Fraction(0))
            want = _bf16_rne_exact(exact)
            if y[i, j] != want:
                # FP64 accumulation rounded before the BF16 rounding: the result
                # must then be the BF16 rounding of the sequential FP64 sum.
                acc = 0.0
                for k in range(K):
                    acc += float(a[i, k]) * float(b[j, k])
                assert Fraction(acc) != exact
                assert y[i, j] == _bf16_rne_exact(Fraction(acc))
                logged += 1
    assert logged <= max(1, (M * N) // 10)


def test_gemm_plain_matmul_special_case(orc):
    """Scales of 2^0 and small integer payloads: every sum is an integer far
    below 2^8, so the BF16 result equals an ordinary float64 matmul."""
    rng = np.random.default_rng(9)
    ints = np.array([0, 1, 2, 3, 4, -1, -2, -3, -4])
    codes = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48, -1: 0xB8, -2: 0xC0, -3: 0xC4, -4: 0xC8}
    av = rng.choice(ints, size=(16, 32))
    bv = rng.choice(ints, size=(12, 32))
    enc = np.vectorize(codes.get)
    qa, qb = enc(av).astype(np.uint8), enc(bv).astype(np.uint8)
    one = np.full((16, 1), 127, np.uint8)
    a = orc.dequant_rows(qa, one)
    b = orc.dequant_rows(qb, np.full((12, 1), 127, np.uint8))
    assert np.array_equal(a, av) and np.array_equal(b, bv)
    ref = av.astype(np.float64) @ bv.T.astype(np.float64)
    assert np.all(np.abs(ref) < 256)
    want = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.gemm(a, b), want)


def test_gemm_row_sampling_matches_full(orc):
    rng = np.random.default_rng(4)
    a = orc.dequant_rows(*_rand_operand(rng, 40, 96, 6))
    b = orc.dequant_rows(*_rand_operand(rng, 24, 96, 6))
    full = orc.gemm(a, b)
    rows = np.array([39, 0, 17, 17, 5])
    assert np.array_equal(orc.gemm(a, b, rows=rows), full[rows])


def test_gemm_transposed_operands(orc):
    """(A B^T)^T = B A^T: the oracle is symmetric in its operands."""
    rng = np.random.default_rng(5)
    a = orc.dequant_rows(*_rand_operand(rng, 9, 64, 5))
    b = orc.dequant_rows(*_rand_operand(rng, 11, 64, 5))
    assert np.array_equal(orc.gemm(a, b).T, orc.gemm(b, a))


def test_grouped_gemm_matches_per_expert_slices(orc):
    rng = np.random.default_rng(6)
    K, N, G = 64, 16, 6
    sizes = np.array([0, 5, 0, 33, 1, 0])               # includes empty experts
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    a = orc.dequant_rows(*_rand_operand(rng, int(off[-1]), K, 5))
    b = np.stack([orc.dequant_rows(*_rand_operand(rng, N, K, 5)) for _ in range(G)])
    y = orc.grouped_gemm(a, b, off)
    assert y.shape == (off[-1], N)
    for g in range(G):
        lo, hi = off[g], off[g + 1]
        if hi > lo:
            assert np.array_equal(y[lo:hi], orc.gemm(a[lo:hi], b[g]))
    rows = np.array([38, 5, 6, 0])
    assert np.array_equal(orc.grouped_gemm(a, b, off, rows=rows), y[rows])


def test_grouped_gemm_exact_tiny(orc):
    rng = np.random.default_rng(8)
    K, N = 32, 3
    off = np.array([0, 2, 2, 3], dtype=np.int64)
    qa, sa = _rand_operand(rng, 3, K, 3)
    a = orc.dequant_rows(qa, sa)
    b = np.stack([orc.dequant_rows(*_rand_operand(rng, N, K, 3)) for _ in range(3)])
    y = orc.grouped_gemm(a, b, off)
    owner = [0, 0, 2]
    for r in range(3):
        for n in range(N):
            exact = sum((Fraction(a[r, k]) * Fraction(b[owner[r], n, k]) for k in range(K)), Fraction(0))
            assert y[r, n] == _bf16_rne_exact(exact)
