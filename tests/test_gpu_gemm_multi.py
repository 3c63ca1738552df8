"""GPU parity of mxq_gemm_bf16out_multi: several GEMMs in one persistent launch.

Each result must equal, bit for bit, the single-GEMM call on the same operands
(the tile computation is the same; only the assignment of tiles to SMs
differs), and the single-GEMM path is held to the oracle here as well:
|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref) on the oracle's FP64 product of its
own quantization of the BF16 inputs.  The backward pass of a linear layer
runs its dgrad and wgrad matmuls on the row and column copies of the 1x32
quantization (torchtitan-npu tutorial, "MXFP8 与 HiF8 架构原理速览").
"""
import numpy as np
import pytest
import torch

from _util import assert_gemm_close, bits, gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _mods():
    from mxfp8_microscaled_precision_gb300 import mxq, workloads
    from oracle import oracle
    return mxq, workloads, oracle


def _same(a, b, what):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), what


def _desc(aq, as_, bq, bs, M, N, K, **kw):
    return dict(a_q=aq, a_s=as_, b_q=bq, b_s=bs, M=M, N=N, K=K, **kw)


@pytest.mark.parametrize("M,N,K", [(8192, 4096, 4096), (320, 288, 416), (1024, 160, 2048)])
def test_backward_pair_equals_separate_calls(M, N, K):
    """dX = dY W (dY row copy x W column copy) and dW = dY^T X (column copies);
    the layer is X [M, K] -> Y [M, N] with W [N, K]."""
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=M + 1, device="cuda")
    W = workloads.normal((N, K), 0.02, seed=N + 2, device="cuda")
    dY = workloads.normal((M, N), 1e-3, seed=K + 3, device="cuda")
    _, _, xq_t, xs_t = mxq.quant_1x32_dual(X)
    _, _, wq_t, ws_t = mxq.quant_1x32_dual(W)
    gq, gs, gq_t, gs_t = mxq.quant_1x32_dual(dY)
    dx, dw = mxq.gemm_multi([_desc(gq, gs, wq_t, ws_t, M, K, N), _desc(gq_t, gs_t, xq_t, xs_t, N, K, M)])
    dx1 = mxq.gemm(gq, gs, wq_t, ws_t, M, K, N)
    dw1 = mxq.gemm(gq_t, gs_t, xq_t, xs_t, N, K, M)
    torch.cuda.synchronize()
    _same(dx, dx1, "dgrad")
    _same(dw, dw1, "wgrad")
    if M * N * K <= 1 << 30:   # the oracle on the whole output
        ogq, ogs, ogq_t, ogs_t = oracle.quant_dual(bits(dY))
        _, _, owq_t, ows_t = oracle.quant_dual(bits(W))
        _, _, oxq_t, oxs_t = oracle.quant_dual(bits(X))
        assert_gemm_close(dx, oracle.gemm(oracle.dequant_rows(ogq, ogs), oracle.dequant_rows(owq_t, ows_t)), "dgrad")
        assert_gemm_close(dw, oracle.gemm(oracle.dequant_rows(ogq_t, ogs_t), oracle.dequant_rows(oxq_t, oxs_t)),
                          "wgrad")


def test_four_mixed_gemms_with_formats_and_tails():
    """Four GEMMs of different shapes (ragged M, N not a multiple of the tile,
    K with a 32-tail), one with an E5M2 operand: each equals its own call and
    the oracle."""
    mxq, workloads, oracle = _mods()
    shapes = [(300, 272, 416, "e4m3"), (129, 384, 2048, "e5m2"), (1, 128, 32, "e4m3"), (640, 1040, 160, "e4m3")]
    descs, refs, singles = [], [], []
    for i, (M, N, K, afmt) in enumerate(shapes):
        A = workloads.normal_with_outliers((M, K), seed=10 + i)
        B = workloads.normal((N, K), 0.02, seed=20 + i)
        fa = 1 if afmt == "e5m2" else 0
        aq, as_, _, _ = mxq.quant_1x32_dual_batched(A.cuda(), col=False, fmt=afmt)
        bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
        descs.append(_desc(aq[0], as_[0], bq, bs, M, N, K, a_fmt=afmt))
        singles.append(mxq.gemm_fmt(aq[0], as_[0], afmt, bq, bs, "e4m3", M, N, K))
        a_ref = oracle.dequant_rows_fmt(*oracle.quant_rows_fmt(bits(A), fa), fa)
        refs.append(oracle.gemm(a_ref, oracle.dequant_rows(*oracle.quant_rows(bits(B)))))
    outs = mxq.gemm_multi(descs)
    torch.cuda.synchronize()
    for i, (y, y1, ref) in enumerate(zip(outs, singles, refs)):
        _same(y, y1, f"gemm {i}")
        assert_gemm_close(y, ref, f"gemm {i} {shapes[i]}")


def test_empty_and_zero_k_members():
    """M == 0 members are skipped, K == 0 members are zero-filled, and the
    others are computed; strided outputs keep the bytes between rows."""
    mxq, workloads, oracle = _mods()
    M, N, K = 256, 512, 512
    X = workloads.normal((M, K), 1.0, seed=5)
    W = workloads.normal((N, K), 0.02, seed=6)
    xq, xs, _, _ = mxq.quant_1x32_dual(X.cuda(), col=False)
    wq, ws, _, _ = mxq.quant_1x32_dual(W.cuda(), col=False)
    big = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    zero_k = torch.full((64, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    empty = torch.full((4, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    mxq.gemm_multi([_desc(xq, xs, wq, ws, M, N, K, out=big[:, :N]),
                    _desc(xq, xs, wq, ws, 64, 128, 0, out=zero_k),
                    _desc(xq, xs, wq, ws, 0, 128, K, out=empty)])
    y1 = mxq.gemm(xq, xs, wq, ws, M, N, K)
    torch.cuda.synchronize()
    _same(big[:, :N], y1, "member")
    assert torch.all(big[:, N:] == 7.0), "bytes past N in each row were written"
    assert torch.all(zero_k == 0), "K == 0 member must be zero"
    assert torch.all(empty == 3.0), "M == 0 member must not be touched"


def test_mn_major_pair():
    """Two 32x32-recipe dgrads (B = the single payload read MN-major)."""
    mxq, workloads, oracle = _mods()
    descs, singles = [], []
    for i, (M, n, k) in enumerate([(512, 1024, 768), (300, 384, 256)]):
        dY = workloads.normal((M, n), 1e-3, seed=30 + i)
        Wt = workloads.normal((n, k), 0.02, seed=40 + i)
        gq, gs, _, _ = mxq.quant_1x32_dual(dY.cuda(), col=False)
        wq, _, ws_bwd = mxq.quant_32x32(Wt.cuda())
        descs.append(_desc(gq, gs, wq, ws_bwd, M, k, n))
        singles.append(mxq.gemm(gq, gs, wq, ws_bwd, M, k, n, b_mn_major=True))
    outs = mxq.gemm_multi(descs, b_mn_major=True)
    torch.cuda.synchronize()
    for i, (y, y1) in enumerate(zip(outs, singles)):
        _same(y, y1, f"mn-major gemm {i}")


def test_device_status_clean_after_multi():
    mxq, _, _ = _mods()
    assert mxq.get_device_status() == 0
