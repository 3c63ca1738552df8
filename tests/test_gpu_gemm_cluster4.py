"""GPU parity of the dense GEMMs on clusters of two CTA pairs (MXQ_GEMM_CLUSTER=4).

In that schedule the two pairs of a cluster compute vertically adjacent
256 x 256 tiles and share each B tile through multicast loads.  Every pair
still issues the same MMAs over the same K order as on clusters of one pair,
so each result must equal the one-pair result bit for bit.  The outputs are
also held to the oracle: |gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref) on the
oracle's FP64 product of its own quantization of the BF16 inputs (the FP8
matmul with BF16 output of the torchtitan-npu tutorial, "MXFP8 与 HiF8 架构原理速览";
the 32x32 single payload read N-major by the dgrad, MindSpeed RFC "Add
MXFP8-32x32 quantization support to FSDP", section 3.1).
"""
import os

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


def _with_cluster(value, fn):
    old = os.environ.get("MXQ_GEMM_CLUSTER")
    os.environ["MXQ_GEMM_CLUSTER"] = value
    try:
        out = fn()
        torch.cuda.synchronize()
        return out
    finally:
        if old is None:
            del os.environ["MXQ_GEMM_CLUSTER"]
        else:
            os.environ["MXQ_GEMM_CLUSTER"] = old


def _both(fn):
    """fn() on clusters of two pairs, then on single pairs."""
    return _with_cluster("4", fn), _with_cluster("2", fn)


def _same(a, b, what):
    assert a.shape == b.shape, what
    assert torch.equal(a.view(torch.uint8) if a.dtype == torch.uint8 else a.view(torch.int16),
                       b.view(torch.uint8) if b.dtype == torch.uint8 else b.view(torch.int16)), what


@pytest.mark.parametrize("M,N,K", [
    (300, 272, 416),     # one cluster row: the second pair holds rows 256..299 only
    (1, 128, 32),        # the second pair entirely past the rows
    (129, 384, 256),
    (600, 528, 384),     # two cluster rows, the second one partly filled; N ragged
    (1100, 1056, 1024),  # several clusters, ragged in M and N
    (2048, 2048, 2048),
])
def test_forward_equals_pairs_and_oracle(M, N, K):
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=M + 7 * N + K)
    W = workloads.normal((N, K), 0.02, seed=3 * M + N + K)
    xq, xs, _, _ = mxq.quant_1x32_dual(X.cuda(), col=False)
    wq, ws, _, _ = mxq.quant_1x32_dual(W.cuda(), col=False)
    y4, y2 = _both(lambda: mxq.gemm(xq, xs, wq, ws, M, N, K))
    _same(y4, y2, f"forward {M}x{N}x{K}")
    if M * N * K <= 1 << 28:
        oxq, oxs = oracle.quant_rows(bits(X))
        owq, ows = oracle.quant_rows(bits(W))
        assert_gemm_close(y4, oracle.gemm(oracle.dequant_rows(oxq, oxs), oracle.dequant_rows(owq, ows)),
                          f"forward {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(320, 288, 416), (1024, 640, 768)])
def test_dgrad_wgrad_n_major_equal_pairs_and_oracle(M, N, K):
    """dX = dY W reads W's column copy N-major; dW = dY^T X contracts over M;
    both in one launch and as separate launches."""
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=M + 11)
    W = workloads.normal((N, K), 0.02, seed=N + 12)
    dY = workloads.normal((M, N), 1e-3, seed=K + 13)
    _, _, xq_t, xs_t = mxq.quant_1x32_dual(X.cuda())
    _, _, wq_t, ws_t = mxq.quant_1x32_dual(W.cuda())
    gq, gs, gq_t, gs_t = mxq.quant_1x32_dual(dY.cuda())

    def run():
        dx = mxq.gemm(gq, gs, wq_t, ws_t, M, K, N)
        dw = mxq.gemm(gq_t, gs_t, xq_t, xs_t, N, K, M)
        pair = mxq.gemm_multi([dict(a_q=gq, a_s=gs, b_q=wq_t, b_s=ws_t, M=M, N=K, K=N),
                               dict(a_q=gq_t, a_s=gs_t, b_q=xq_t, b_s=xs_t, M=N, N=K, K=M)])
        return dx, dw, pair[0], pair[1]

    r4, r2 = _both(run)
    for a, b, what in zip(r4, r2, ["dgrad", "wgrad", "dgrad in the multi launch", "wgrad in the multi launch"]):
        _same(a, b, what)
    _same(r4[0], r4[2], "dgrad: multi launch vs single")
    _same(r4[1], r4[3], "wgrad: multi launch vs single")
    ogq, ogs, ogq_t, ogs_t = oracle.quant_dual(bits(dY))
    _, _, owq_t, ows_t = oracle.quant_dual(bits(W))
    _, _, oxq_t, oxs_t = oracle.quant_dual(bits(X))
    assert_gemm_close(r4[0], oracle.gemm(oracle.dequant_rows(ogq, ogs), oracle.dequant_rows(owq_t, ows_t)), "dgrad")
    assert_gemm_close(r4[1], oracle.gemm(oracle.dequant_rows(ogq_t, ogs_t), oracle.dequant_rows(oxq_t, oxs_t)),
                      "wgrad")


def test_32x32_payload_read_n_major():
    """The 32x32 recipe's dgrad: the one weight payload read N-major with the
    backward scales."""
    mxq, workloads, oracle = _mods()
    M, n, k = 700, 512, 384
    W = workloads.normal((n, k), 0.02, seed=21)
    dY = workloads.normal((M, n), 1e-3, seed=22)
    q, _, sb = mxq.quant_32x32(W.cuda())
    gq, gs, _, _ = mxq.quant_1x32_dual(dY.cuda(), col=False)
    dx4, dx2 = _both(lambda: mxq.gemm(gq, gs, q, sb, M, k, n, b_mn_major=True))
    _same(dx4, dx2, "32x32 dgrad")
    oq, osf, _ = oracle.quant_32x32(bits(W))
    ogq, ogs = oracle.quant_rows(bits(dY))
    w_deq = oracle.dequant_rows(oq, osf)
    assert_gemm_close(dx4, oracle.gemm(oracle.dequant_rows(ogq, ogs), np.ascontiguousarray(w_deq.T)),
                      "32x32 dgrad")


@pytest.mark.parametrize("M,N,K,mn", [(576, 512, 384, False), (1300, 768, 256, True)])
def test_quantizing_epilogue_equals_pairs(M, N, K, mn):
    """The quantizing epilogue's BF16 output, E4M3 payload and scales on
    clusters of two pairs equal the single-pair bytes, and the payload and
    scales equal the oracle's 1x32 quantization of that BF16 output."""
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=M + 31)
    W = workloads.normal((N, K), 0.02, seed=N + 32)
    xq, xs, _, _ = mxq.quant_1x32_dual(X.cuda(), col=False)
    if mn:   # dgrad-style: the 32x32 payload of W^T [K, N] read N-major
        wq, _, ws = mxq.quant_32x32(W.t().contiguous().cuda())
    else:
        wq, ws, _, _ = mxq.quant_1x32_dual(W.cuda(), col=False)
    r4, r2 = _both(lambda: mxq.gemm_mxfp8out(xq, xs, wq, ws, M, N, K, b_mn_major=mn))
    for a, b, what in zip(r4, r2, ["y", "y_q", "y_s"]):
        _same(a, b, what)
    q_ref, s_ref = oracle.quant_rows(bits(r4[0]))
    assert np.array_equal(u8(r4[1]), q_ref), "payload vs the oracle's quantization of y"
    assert np.array_equal(u8(r4[2]), oracle.scale_tiled(s_ref)), "tiled scales vs the oracle's"
