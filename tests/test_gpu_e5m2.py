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


# ---- MoE backward with E5M2 gradients: the token-axis quantizer inside each
# expert and both grouped GEMMs take the E5M2 payload of dY.

def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


@pytest.mark.parametrize("sizes", [[0, 5, 0, 300, 1, 130], [33, 31, 129, 127, 0, 1], [1000]])
def test_e5m2_grouped_cols_quant_matches_oracle(sizes):
    mxq, workloads, oracle = _mods()
    from _util import tiled_to_plain
    off = _offsets(sizes)
    M, C = int(off[-1]), 160
    g = torch.Generator().manual_seed(M + 7)
    x = torch.randn((M, C), generator=g, dtype=torch.float64)
    x = (x * torch.pow(2.0, torch.randint(-60, 60, (M, 1), generator=g).double())).float().to(torch.bfloat16)
    cap = mxq.grouped_capacity(M, len(sizes))
    P, L = oracle.padded_slots(off)
    used = int(P[-1] + L[-1])
    oq, os_ = oracle.quant_cols_grouped(bits(x), off, cap, fmt=1)
    for layout in ("rowmajor", "tiled"):
        q, s = mxq.quant_cols_grouped(x.cuda(), torch.from_numpy(off).cuda(), cap, layout=layout, fmt="e5m2")
        torch.cuda.synchronize()
        assert np.array_equal(u8(q)[:, :used], oq[:, :used]), layout
        sp = u8(s) if layout == "rowmajor" else tiled_to_plain(u8(s), C, cap // 32)
        assert np.array_equal(sp[:, :used // 32], os_[:, :used // 32]), layout


@pytest.mark.parametrize("sizes,N,K", [([0, 5, 0, 300, 1, 130], 256, 384), ([33, 0, 129, 127], 384, 128)])
def test_e5m2_moe_dgrad(sizes, N, K):
    """dX_r = dY_r W_g with dY in E5M2 and the expert weights' column copies in E4M3."""
    mxq, workloads, oracle = _mods()
    G, off = len(sizes), _offsets(sizes)
    M = int(off[-1])
    dY = workloads.normal((M, N), 1e-3, seed=M + N)
    W = workloads.normal((G, N, K), 0.02, seed=K + G)
    gq, gs, _, _ = mxq.quant_1x32_dual_batched(dY.cuda(), col=False, fmt="e5m2")
    _, _, wq_col, ws_col = mxq.quant_1x32_dual_batched(W.cuda(), row=False)            # [G, K, N]
    dx = mxq.grouped_gemm(gq[0], gs[0], wq_col.reshape(G * K, N), ws_col.reshape(-1),
                          torch.from_numpy(off).cuda(), K, N, a_fmt="e5m2")
    torch.cuda.synchronize()
    a = oracle.dequant_rows_fmt(*oracle.quant_rows_fmt(bits(dY), 1), 1)
    wt = np.stack([oracle.dequant_rows(*oracle.quant_dual(bits(W[g]), want_row=False)[2:]) for g in range(G)])
    assert_gemm_close(dx, oracle.grouped_gemm(a, wt, off), "e5m2 moe dgrad")


@pytest.mark.parametrize("sizes,N,K", [([0, 5, 0, 300, 1, 130], 256, 384), ([64] * 8, 128, 256)])
def test_e5m2_moe_wgrad(sizes, N, K):
    """dW_g = dY_g^T X_g with dY_g's token-axis copy in E5M2 and X_g's in E4M3."""
    mxq, workloads, oracle = _mods()
    G, off = len(sizes), _offsets(sizes)
    M = int(off[-1])
    offd = torch.from_numpy(off).cuda()
    dY = workloads.normal((M, N), 1e-3, seed=2 * M + N)
    X = workloads.normal_with_outliers((M, K), seed=M + K)
    cap = mxq.grouped_capacity(M, G)
    aq, as_ = mxq.quant_cols_grouped(dY.cuda(), offd, cap, fmt="e5m2")
    bq, bs = mxq.quant_cols_grouped(X.cuda(), offd, cap)
    dw = mxq.grouped_gemm_wgrad(aq, as_, bq, bs, offd, M, a_fmt="e5m2")
    torch.cuda.synchronize()
    oaq, oas = oracle.quant_cols_grouped(bits(dY), off, cap, fmt=1)
    obq, obs = oracle.quant_cols_grouped(bits(X), off, cap)
    P, L = oracle.padded_slots(off)
    for g in range(G):
        if L[g] == 0:
            assert torch.all(dw[g] == 0), f"expert {g} is empty and must be zero"
            continue
        sl = slice(int(P[g]), int(P[g] + L[g]))
        ss = slice(sl.start // 32, sl.stop // 32)
        a = oracle.dequant_rows_fmt(np.ascontiguousarray(oaq[:, sl]), np.ascontiguousarray(oas[:, ss]), 1)
        b = oracle.dequant_rows(np.ascontiguousarray(obq[:, sl]), np.ascontiguousarray(obs[:, ss]))
        assert_gemm_close(dw[g], oracle.gemm(a, b), f"e5m2 moe wgrad expert {g}")
