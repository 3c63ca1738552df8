"""GPU parity of the E5M2 destination type (MindSpeed RFC section 3.5.2.3:
dst_type E4M3 or E5M2): 1x32 row / column quantization bit-exact against the
oracle, and block-scaled GEMMs with E5M2 x E5M2 and mixed E5M2 x E4M3
operands within the GEMM tolerance."""
import numpy as np
import pytest
import torch

from _util import assert_gemm_close, bits, gpu_or_skip, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _mods():
    from mxfp8_microscaled_precision_gb300 import mxq, workloads
    from oracle import oracle
    return mxq, workloads, oracle


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
@pytest.mark.parametrize("shape,col", [((256, 512), True), ((130, 96), False), ((1, 4096), False), ((96, 160), True)])
def test_e5m2_quant_matches_oracle(shape, col, layout):
    mxq, workloads, oracle = _mods()
    g = torch.Generator().manual_seed(shape[0] + shape[1])
    x = torch.randn(shape, generator=g, dtype=torch.float64)
    x = (x * torch.pow(2.0, torch.randint(-40, 40, (shape[0], 1), generator=g).double())).float().to(torch.bfloat16)
    x[0, 3] = float("nan") if shape[1] >= 64 else x[0, 3]
    qr, sr, qc, sc = mxq.quant_1x32_dual_batched(x.cuda(), col=col, layout=layout, fmt="e5m2")
    torch.cuda.synchronize()
    conv = oracle.scale_tiled if layout == "tiled" else (lambda s: s.reshape(-1))
    oq, os_ = oracle.quant_rows_fmt(bits(x), 1)
    assert np.array_equal(u8(qr[0]), oq) and np.array_equal(u8(sr[0]).reshape(-1), conv(os_).reshape(-1))
    if col:
        oqc, osc = oracle.quant_rows_fmt(np.ascontiguousarray(bits(x).T), 1)
        assert np.array_equal(u8(qc[0]), oqc) and np.array_equal(u8(sc[0]).reshape(-1), conv(osc).reshape(-1))


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e5m2", "e4m3"), ("e4m3", "e5m2")])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (300, 272, 416)])
def test_e5m2_gemm(a_fmt, b_fmt, M, N, K):
    mxq, workloads, oracle = _mods()
    X = workloads.normal((M, K), 1e-3, seed=M + N)             # gradient-like operand
    W = workloads.normal((N, K), 0.02, seed=N + K)
    fa, fb = (1 if a_fmt == "e5m2" else 0), (1 if b_fmt == "e5m2" else 0)
    xq, xs, _, _ = mxq.quant_1x32_dual_batched(X.cuda(), col=False, fmt=a_fmt)
    wq, ws, _, _ = mxq.quant_1x32_dual_batched(W.cuda(), col=False, fmt=b_fmt)
    y = mxq.gemm_fmt(xq[0], xs[0], a_fmt, wq[0], ws[0], b_fmt, M, N, K)
    torch.cuda.synchronize()
    a = oracle.dequant_rows_fmt(*oracle.quant_rows_fmt(bits(X), fa), fa)
    b = oracle.dequant_rows_fmt(*oracle.quant_rows_fmt(bits(W), fb), fb)
    assert_gemm_close(y, oracle.gemm(a, b), f"{a_fmt} x {b_fmt}")
