"""GPU parity of the MoE backward pieces against the oracle.

- dgrad: the stacked expert weights [G, N, K] are quantized per expert in one
  batched call; their column copies [G, K, N] feed the grouped GEMM
  (dX_r = dY_r W_g for the rows r of expert g).
- wgrad: token-axis quantization inside each expert (groups of 32 tokens from
  the expert's first token, zero-padded at its end, 128-aligned slots) and the
  grouped-contraction GEMM (dW_g = dY_g^T X_g).

The MoE expert layers (gate_up_proj / down_proj) run quantized grouped
matmuls (torchtitan-npu tutorial, "MoE 专家层 (Grouped MM)"; MindSpeed RFC
section 2.2); the token-padding rule is the reading stated in the oracle.
"""
import numpy as np
import pytest
import torch

from _util import assert_gemm_close, bits, gpu_or_skip, tiled_to_plain, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _mods():
    from mxfp8_microscaled_precision_gb300 import mxq, workloads
    from oracle import oracle
    return mxq, workloads, oracle


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
@pytest.mark.parametrize("B,R,C,pad", [(3, 256, 384, 0), (5, 96, 160, 64), (1, 128, 128, 0)])
def test_batched_dual_quant_matches_oracle(B, R, C, pad, layout):
    mxq, workloads, oracle = _mods()
    full = workloads.normal((B, R + pad, C), 0.02, seed=B * R + C)
    x = full.cuda()[:, :R, :]                      # matrix stride (R+pad)*C, not R*C
    qr, sr, qc, sc = mxq.quant_1x32_dual_batched(x, layout=layout)
    torch.cuda.synchronize()
    conv = oracle.scale_tiled if layout == "tiled" else (lambda s: s.reshape(-1))
    for b in range(B):
        oqr, osr, oqc, osc = oracle.quant_dual(bits(full[b, :R]))
        assert np.array_equal(u8(qr[b]), oqr) and np.array_equal(u8(sr[b]), conv(osr))
        assert np.array_equal(u8(qc[b]), oqc) and np.array_equal(u8(sc[b]), conv(osc))


@pytest.mark.parametrize("sizes", [[0, 5, 0, 300, 1, 130], [128, 256], [33, 31, 129, 127, 0, 1], [1000]])
def test_grouped_cols_quant_matches_oracle(sizes):
    mxq, workloads, oracle = _mods()
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M, C = int(off[-1]), 192
    x = workloads.normal_with_outliers((M, C), seed=M + len(sizes))
    cap = mxq.grouped_capacity(M, len(sizes))
    P, L = oracle.padded_slots(off)
    used = int(P[-1] + L[-1])
    oq, os_ = oracle.quant_cols_grouped(bits(x), off, cap)
    for layout in ("rowmajor", "tiled"):
        q, s = mxq.quant_cols_grouped(x.cuda(), torch.from_numpy(off).cuda(), cap, layout=layout)
        torch.cuda.synchronize()
        assert np.array_equal(u8(q)[:, :used], oq[:, :used])
        sp = u8(s) if layout == "rowmajor" else tiled_to_plain(u8(s), C, cap // 32)
        assert np.array_equal(sp[:, :used // 32], os_[:, :used // 32])


def _moe_case(sizes, N, K, seed):
    mxq, workloads, oracle = _mods()
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    dY = workloads.normal((M, N), 1e-3, seed=seed)
    X = workloads.normal_with_outliers((M, K), seed=seed + 1)
    W = workloads.normal((G, N, K), 0.02, seed=seed + 2)
    return mxq, oracle, off, dY, X, W


@pytest.mark.parametrize("sizes,N,K", [([0, 5, 0, 300, 1, 130], 256, 384), ([64] * 8, 128, 256),
                                        ([33, 0, 129, 127], 384, 128)])
def test_moe_dgrad_via_batched_column_copies(sizes, N, K):
    mxq, oracle, off, dY, X, W = _moe_case(sizes, N, K, seed=sum(sizes) + N)
    G = len(sizes)
    offd = torch.from_numpy(off).cuda()
    gq, gs, _, _ = mxq.quant_1x32_dual(dY.cuda(), col=False)
    _, _, wq_col, ws_col = mxq.quant_1x32_dual_batched(W.cuda(), row=False)        # [G, K, N]
    dx = mxq.grouped_gemm(gq, gs, wq_col.reshape(G * K, N), ws_col.reshape(-1), offd, K, N)
    torch.cuda.synchronize()
    og, ogs = oracle.quant_rows(bits(dY))
    wt = np.stack([oracle.dequant_rows(*oracle.quant_dual(bits(W[g]), want_row=False)[2:]) for g in range(G)])
    ref = oracle.grouped_gemm(oracle.dequant_rows(og, ogs), wt, off)
    assert_gemm_close(dx, ref, "moe dgrad")


@pytest.mark.parametrize("sizes,N,K", [([0, 5, 0, 300, 1, 130], 256, 384), ([64] * 8, 128, 256),
                                        ([33, 0, 129, 127], 384, 128), ([0, 0, 0], 128, 128)])
def test_moe_wgrad_matches_oracle(sizes, N, K):
    mxq, oracle, off, dY, X, W = _moe_case(sizes, N, K, seed=3 * sum(sizes) + K)
    G = len(sizes)
    M = int(off[-1])
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
    for g in range(G):
        if L[g] == 0:
            assert torch.all(dw[g] == 0), f"expert {g} is empty and must be zero"
            continue
        sl = slice(int(P[g]), int(P[g] + L[g]))
        a = oracle.dequant_rows(np.ascontiguousarray(oaq[:, sl]), np.ascontiguousarray(oas[:, sl.start // 32:sl.stop // 32]))
        b = oracle.dequant_rows(np.ascontiguousarray(obq[:, sl]), np.ascontiguousarray(obs[:, sl.start // 32:sl.stop // 32]))
        assert_gemm_close(dw[g], oracle.gemm(a, b), f"moe wgrad expert {g}")


def test_moe_wgrad_full_size_sampled():
    """128 experts, 131072 routed rows (Zipf loads, empty experts): down-proj
    wgrad dW_g [4096, 2048] = dY_g^T H_g on sampled output rows of selected experts."""
    mxq, workloads, oracle = _mods()
    d = workloads.moe_grouped(weights=False)
    off = d["routing"].offsets.numpy()
    G, M = off.size - 1, int(off[-1])
    offd = torch.from_numpy(off).cuda()
    H = d["H"]                                                   # [M, 2048]
    dY = workloads.normal((M, 4096), 1e-3, seed=4711, device="cuda")
    cap = mxq.grouped_capacity(M, G)
    aq, as_ = mxq.quant_cols_grouped(dY, offd, cap)
    bq, bs = mxq.quant_cols_grouped(H.cuda(), offd, cap)
    dw = mxq.grouped_gemm_wgrad(aq, as_, bq, bs, offd, M)
    torch.cuda.synchronize()
    sizes = np.diff(off)
    nz = np.flatnonzero(sizes)
    experts = sorted({int(nz[np.argmax(sizes[nz])]), int(nz[np.argmin(sizes[nz])]), int(nz[len(nz) // 2])})
    rng = np.random.default_rng(5)
    dY_h = dY.cpu()
    for g in experts:
        lo, hi = int(off[g]), int(off[g + 1])
        sub = np.array([0, lo, hi - lo])                          # one expert, on its own
        oaq, oas = oracle.quant_cols_grouped(bits(dY_h[lo:hi]), np.array([0, hi - lo]), cap)
        obq, obs = oracle.quant_cols_grouped(bits(H[lo:hi]), np.array([0, hi - lo]), cap)
        L = (hi - lo + 127) // 128 * 128
        a = oracle.dequant_rows(np.ascontiguousarray(oaq[:, :L]), np.ascontiguousarray(oas[:, :L // 32]))
        b = oracle.dequant_rows(np.ascontiguousarray(obq[:, :L]), np.ascontiguousarray(obs[:, :L // 32]))
        rows = np.unique(np.concatenate([[0, 4095], rng.integers(0, 4096, 16)]))
        assert_gemm_close(dw[g][torch.from_numpy(rows).cuda()], oracle.gemm(a, b, rows=rows), f"expert {g}")
        del sub
