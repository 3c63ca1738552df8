"""GPU parity of the grouped GEMMs with more experts than the CTA-pair kernel's
schedule tables hold (512 < G <= 1024): those launches run on the single-CTA
kernel, and the results must meet the same bar against the oracle,
|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref).  G = 512 (the largest count the pair
kernel takes) is checked beside them.

The MoE expert layers run the quantized grouped matmul (torchtitan-npu
tutorial, "MoE 专家层 (Grouped MM)"; MindSpeed RFC section 2.2, gate_up_proj
and down_proj) and its weight gradient over each expert's tokens.
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


def _sizes(G, seed):
    """Expert sizes 0..40 (a quarter of the experts empty), seeded."""
    rng = np.random.default_rng(seed)
    s = rng.integers(0, 41, G)
    s[rng.random(G) < 0.25] = 0
    return s.astype(np.int64)


@pytest.mark.parametrize("G", [512, 513, 700, 1024])
def test_grouped_rows_many_experts(G):
    mxq, workloads, oracle = _mods()
    sizes = _sizes(G, seed=G)
    N, K = 128, 96
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    A = workloads.normal_with_outliers((M, K), seed=G + 1)
    B = workloads.normal((G * N, K), 0.02, seed=G + 2)
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    y = mxq.grouped_gemm(aq, as_, bq, bs, torch.from_numpy(off).cuda(), N, K)
    torch.cuda.synchronize()
    oa, osa = oracle.quant_rows(bits(A))
    ob, osb = oracle.quant_rows(bits(B))
    ref = oracle.grouped_gemm(oracle.dequant_rows(oa, osa), oracle.dequant_rows(ob, osb).reshape(G, N, K), off)
    assert_gemm_close(y, ref, f"grouped rows, {G} experts")


@pytest.mark.parametrize("G", [512, 600, 1024])
def test_grouped_wgrad_many_experts(G):
    """dW_g = dY_g^T X_g for every expert (empty experts give zeros)."""
    mxq, workloads, oracle = _mods()
    sizes = _sizes(G, seed=3 * G)
    N, K = 128, 64
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    dY = workloads.normal((M, N), 1e-3, seed=G + 3)
    X = workloads.normal_with_outliers((M, K), seed=G + 4)
    offd = torch.from_numpy(off).cuda()
    cap = mxq.grouped_capacity(M, G)
    aq, as_ = mxq.quant_cols_grouped(dY.cuda(), offd, cap)
    bq, bs = mxq.quant_cols_grouped(X.cuda(), offd, cap)
    dw = mxq.grouped_gemm_wgrad(aq, as_, bq, bs, offd, M)
    torch.cuda.synchronize()
    assert dw.shape == (G, N, K)
    oaq, oas = oracle.quant_cols_grouped(bits(dY), off, cap)
    obq, obs = oracle.quant_cols_grouped(bits(X), off, cap)
    P, L = oracle.padded_slots(off)
    empty = np.flatnonzero(L == 0)
    assert empty.size > 0 and torch.all(dw[torch.from_numpy(empty).cuda()] == 0), "empty experts must be zero"
    live = np.flatnonzero(L > 0)
    got, ref = [], []
    for g in live:
        sl = slice(int(P[g]), int(P[g] + L[g]))
        a = oracle.dequant_rows(np.ascontiguousarray(oaq[:, sl]), np.ascontiguousarray(oas[:, sl.start // 32:sl.stop // 32]))
        b = oracle.dequant_rows(np.ascontiguousarray(obq[:, sl]), np.ascontiguousarray(obs[:, sl.start // 32:sl.stop // 32]))
        ref.append(oracle.bf16_to_double(oracle.gemm(a, b)))
    got = dw[torch.from_numpy(live).cuda()].float().cpu().numpy().astype(np.float64)
    ref = np.stack(ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    bad = np.abs(got - ref) > 1e-2 * np.abs(ref) + 1e-3 * rms
    assert not bad.any(), f"{int(bad.sum())} weight-gradient outputs outside the bar, {G} experts"
