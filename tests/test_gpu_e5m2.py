"""GPU parity of the E5M2 destination type (MindSpeed RFC section 3.5.2.3:
dst_type E4M3 or E5M2 for the quantizer of both recipes): 1x32 row / column
and 32x32 block quantization bit-exact against the oracle, and block-scaled
GEMMs with E5M2 x E5M2 and mixed E5M2 x E4M3 operands (including the 32x32
payload read forward and N-major) within the GEMM tolerance."""
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


# ---- 32x32 blocks with the E5M2 payload ---------------------------------------------------

def _spread32(n, k, seed, nonfinite=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, k, generator=g, dtype=torch.float64)
    e = torch.randint(-60, 60, (n // 32, k // 32), generator=g).double()
    x = x * torch.pow(2.0, e).repeat_interleave(32, 0).repeat_interleave(32, 1)
    xb = x.float().to(torch.bfloat16)
    if n >= 64 and k >= 64:
        xb[:32, 32:64] = 0.0
        xb[33, 1] = -0.0
    if nonfinite and n >= 64 and k >= 96:
        xb[40, 70] = float("nan")
        xb[5, 3] = float("-inf")
    return xb


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
@pytest.mark.parametrize("shape", [(64, 96), (128, 128), (384, 256), (96, 4096), (4096, 160)])
def test_e5m2_32x32_matches_oracle(shape, layout):
    mxq, _, oracle = _mods()
    w = _spread32(*shape, seed=shape[0] + 5 * shape[1], nonfinite=shape == (384, 256))
    q, sf, sb = mxq.quant_32x32(w.cuda(), layout=layout, fmt="e5m2")
    torch.cuda.synchronize()
    oq, osf, osb = oracle.quant_32x32(bits(w), fmt=1)
    conv = oracle.scale_tiled if layout == "tiled" else (lambda s: s)
    assert np.array_equal(u8(q), oq), "payload"
    assert np.array_equal(u8(sf), conv(osf)), "s_fwd"
    assert np.array_equal(u8(sb), conv(osb)), "s_bwd"


def test_e5m2_32x32_full_weight():
    """The 7168 x 7168 weight of the 32x32 path, E5M2 payload, tiled scales."""
    mxq, workloads, oracle = _mods()
    w = workloads.normal((7168, 7168), 0.02, seed=workloads.seed_for("weight_32x32", "W"))
    q, sf, sb = mxq.quant_32x32(w.cuda(), fmt="e5m2")
    torch.cuda.synchronize()
    oq, osf, osb = oracle.quant_32x32(bits(w), fmt=1)
    assert np.array_equal(u8(q), oq)
    assert np.array_equal(u8(sf), oracle.scale_tiled(osf)) and np.array_equal(u8(sb), oracle.scale_tiled(osb))


@pytest.mark.parametrize("M,n,k", [(300, 384, 256), (256, 512, 1024)])
def test_e5m2_32x32_forward_and_mn_major_dgrad(M, n, k):
    """The single E5M2 32x32 payload of W [n, k] read K-major with s_fwd
    (forward, X in E4M3) and N-major with s_bwd (dgrad, dY in E5M2)."""
    mxq, workloads, oracle = _mods()
    W = workloads.normal((n, k), 0.02, seed=n + k + 1)
    X = workloads.normal_with_outliers((M, k), seed=M + k)
    dY = workloads.normal((M, n), 1e-3, seed=M + n)
    q, sf, sb = mxq.quant_32x32(W.cuda(), fmt="e5m2")
    xq, xs, _, _ = mxq.quant_1x32_dual(X.cuda(), col=False)
    gq, gs, _, _ = mxq.quant_1x32_dual_batched(dY.cuda(), col=False, fmt="e5m2")
    y = mxq.gemm_fmt(xq, xs, "e4m3", q, sf, "e5m2", M, n, k)
    dx = mxq.gemm_fmt(gq[0], gs[0], "e5m2", q, sb, "e5m2", M, k, n, b_mn_major=True)
    torch.cuda.synchronize()
    oq, osf, _ = oracle.quant_32x32(bits(W), fmt=1)
    w_deq = oracle.dequant_rows_fmt(oq, osf, 1)
    x_deq = oracle.dequant_rows(*oracle.quant_rows(bits(X)))
    g_deq = oracle.dequant_rows_fmt(*oracle.quant_rows_fmt(bits(dY), 1), 1)
    assert_gemm_close(y, oracle.gemm(x_deq, w_deq), "e5m2 32x32 forward")
    assert_gemm_close(dx, oracle.gemm(g_deq, np.ascontiguousarray(w_deq.T)), "e5m2 32x32 dgrad")
