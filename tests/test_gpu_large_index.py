"""GPU parity past 2^31 elements: operands and outputs whose element offsets
exceed the range of a 32-bit index, checked against the oracle at both ends of
the index range (the first and last 32-row blocks of a quantized tensor, output
rows whose offsets lie beyond 2^31 in a GEMM).  The quantization is the 1x32
rceil rule of the torchtitan-npu tutorial ("MXFP8 与 HiF8 架构原理速览"); the
GEMM tolerance is |gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref) on the oracle's
product of its own quantization of the same BF16 rows.
"""
import numpy as np
import pytest
import torch

from _util import assert_gemm_close, bits, gpu_or_skip, u8

pytestmark = pytest.mark.gpu

BIG = 1 << 31


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _mods():
    from mxfp8_microscaled_precision_gb300 import mxq, workloads
    from oracle import oracle
    return mxq, workloads, oracle


def test_dual_quant_past_2_31_elements():
    """X [65632, 32768] BF16 (2.15e9 elements), row and column copies with
    plain row-major scales; blocks at row 0 and at the last 32 rows (whose
    payload offsets in both copies pass 2^31) equal the oracle's dual
    quantization of the same 32 rows byte for byte."""
    mxq, workloads, oracle = _mods()
    R, C = 65632, 32768
    assert R * C > BIG and R % 32 == 0
    x = workloads.normal((R, C), 1.0, seed=2031, device="cuda")
    # a few hard groups in the last block: an outlier, a zero group, a NaN
    x[R - 1, 7] = 3.0e4
    x[R - 2, 64:96] = 0.0
    x[R - 3, C - 1] = float("nan")
    qr, sr, qc, sc = mxq.quant_1x32_dual(x, layout="rowmajor")
    torch.cuda.synchronize()
    assert mxq.get_device_status() == 0
    for r0 in (0, R - 32):
        blk = x[r0:r0 + 32]
        oqr, osr, oqc, osc = oracle.quant_dual(bits(blk))
        assert np.array_equal(u8(qr[r0:r0 + 32]), oqr), f"row payload at row {r0}"
        assert np.array_equal(u8(sr[r0:r0 + 32]), osr), f"row scales at row {r0}"
        assert np.array_equal(u8(qc[:, r0:r0 + 32]), oqc), f"column payload at row {r0}"
        assert np.array_equal(u8(sc[:, r0 // 32:r0 // 32 + 1]), osc), f"column scales at row {r0}"


def test_gemm_output_past_2_31_elements():
    """Y [2^21 + 77, 1056] = X W^T with K = 64 (2.2e9 output elements, a ragged
    last row tile and a ragged last column tile): 48 sampled rows, most of them
    past the 2^31-element offset, plus the first and last rows, against the
    oracle."""
    mxq, workloads, oracle = _mods()
    M, N, K = (1 << 21) + 77, 1056, 64
    assert M * N > BIG
    X = workloads.normal_with_outliers((M, K), seed=2032, device="cuda")
    W = workloads.normal((N, K), 0.02, seed=2033)
    xq, xs, _, _ = mxq.quant_1x32_dual(X, col=False)
    wq, ws, _, _ = mxq.quant_1x32_dual(W.cuda(), col=False)
    y = mxq.gemm(xq, xs, wq, ws, M, N, K)
    torch.cuda.synchronize()
    assert mxq.get_device_status() == 0
    first_big = BIG // N + 1
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, M - 1, M - 2], rng.integers(first_big, M, 45)])).astype(np.int64)
    rt = torch.from_numpy(rows).cuda()
    deq = lambda t: oracle.dequant_rows(*oracle.quant_rows(bits(t)))
    ref = oracle.gemm(deq(X[rt]), deq(W), rows=None)
    assert_gemm_close(y[rt], ref, "gemm rows past 2^31 elements")
