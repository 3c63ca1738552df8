"""GPU parity of the block-scaled GEMM (forward, dgrad, wgrad; 1x32 and the
32x32 single-payload dgrad) against the oracle, within
|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref).

The FP8 matmul returns BF16 (torchtitan-npu tutorial, "MXFP8 与 HiF8 架构原理速览");
under the 32x32 recipe forward and backward read one weight payload and
differ only in the scales (MindSpeed RFC, sections 3.1 and 3.3.3).  The
oracle quantizes the same BF16 inputs itself; nothing it uses comes from
the GPU.
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


def _rows_operand(x_cpu):
    """GPU row quantization (tiled scales) and the oracle's dequantized copy."""
    mxq, _, oracle = _mods()
    q, s, _, _ = mxq.quant_1x32_dual(x_cpu.cuda(), col=False)
    oq, os_ = oracle.quant_rows(bits(x_cpu))
    return q, s, oracle.dequant_rows(oq, os_)


def _dual_operand(x_cpu):
    mxq, _, oracle = _mods()
    qr, sr, qc, sc = mxq.quant_1x32_dual(x_cpu.cuda())
    oqr, osr, oqc, osc = oracle.quant_dual(bits(x_cpu))
    return (qr, sr, oracle.dequant_rows(oqr, osr)), (qc, sc, oracle.dequant_rows(oqc, osc))


@pytest.mark.parametrize("M,N,K", [
    (256, 512, 512),     # the small linear layer
    (300, 272, 416),     # ragged M, N not a multiple of 128, K tail of 32
    (1, 128, 32),        # single row, single 32-group
    (129, 384, 256),
    (200, 144, 96),
    (512, 1024, 2048),   # several tiles in each direction
    (1000, 48, 160),     # N smaller than one tile
])
def test_forward_shapes(M, N, K):
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=M + N + K)
    W = workloads.normal((N, K), 0.02, seed=M * N + K)
    xq, xs, xd = _rows_operand(X)
    wq, ws, wd = _rows_operand(W)
    y = mxq.gemm(xq, xs, wq, ws, M, N, K)
    torch.cuda.synchronize()
    assert_gemm_close(y, oracle.gemm(xd, wd), f"forward {M}x{N}x{K}")


def test_wide_scale_spread():
    """Every 32-group of both operands at its own power of two (2^-20..2^20)."""
    mxq, _, oracle = _mods()
    g = torch.Generator().manual_seed(3)
    M, N, K = 192, 256, 640

    def spread(r, c):
        x = torch.randn(r, c, generator=g, dtype=torch.float64)
        e = torch.randint(-20, 21, (r, c // 32, 1), generator=g).double()
        return (x.view(r, c // 32, 32) * torch.pow(2.0, e)).view(r, c).float().to(torch.bfloat16)

    xq, xs, xd = _rows_operand(spread(M, K))
    wq, ws, wd = _rows_operand(spread(N, K))
    y = mxq.gemm(xq, xs, wq, ws, M, N, K)
    torch.cuda.synchronize()
    assert_gemm_close(y, oracle.gemm(xd, wd), "wide scales")


def test_forward_dgrad_wgrad_small():
    mxq, workloads, oracle = _mods()
    M, N, K = 384, 256, 640
    X = workloads.normal_with_outliers((M, K), seed=21)
    W = workloads.normal((N, K), 0.02, seed=22)
    dY = workloads.normal((M, N), 1e-3, seed=23)
    (xr, xrs, xrd), (xc, xcs, xcd) = _dual_operand(X)
    (wr, wrs, wrd), (wc, wcs, wcd) = _dual_operand(W)
    (gr, grs, grd), (gc, gcs, gcd) = _dual_operand(dY)
    y = mxq.gemm(xr, xrs, wr, wrs, M, N, K)
    dx = mxq.gemm(gr, grs, wc, wcs, M, K, N)
    dw = mxq.gemm(gc, gcs, xc, xcs, N, K, M)
    torch.cuda.synchronize()
    assert_gemm_close(y, oracle.gemm(xrd, wrd), "forward")
    assert_gemm_close(dx, oracle.gemm(grd, wcd), "dgrad")
    assert_gemm_close(dw, oracle.gemm(gcd, xcd), "wgrad")


@pytest.mark.parametrize("M,n,k", [(200, 384, 256), (128, 256, 1024), (65, 1024, 384)])
def test_32x32_forward_and_mn_major_dgrad(M, n, k):
    """One payload W [n, k]: forward Y = X W^T with s_fwd, dgrad dX = dY W with
    the payload read N-major and s_bwd."""
    mxq, workloads, oracle = _mods()
    W = workloads.normal((n, k), 0.02, seed=n + k)
    X = workloads.normal_with_outliers((M, k), seed=M + 1)
    dY = workloads.normal((M, n), 1e-3, seed=M + 2)
    q, sf, sb = mxq.quant_32x32(W.cuda())
    oq, osf, _ = oracle.quant_32x32(bits(W))
    w_deq = oracle.dequant_rows(oq, osf)
    xq, xs, xd = _rows_operand(X)
    gq, gs, gd = _rows_operand(dY)
    y = mxq.gemm(xq, xs, q, sf, M, n, k)
    dx = mxq.gemm(gq, gs, q, sb, M, k, n, b_mn_major=True)
    torch.cuda.synchronize()
    assert_gemm_close(y, oracle.gemm(xd, w_deq), "32x32 forward")
    assert_gemm_close(dx, oracle.gemm(gd, np.ascontiguousarray(w_deq.T)), "32x32 dgrad")


def test_strided_output_and_repeat_calls():
    mxq, workloads, oracle = _mods()
    M, N, K = 260, 256, 384
    xq, xs, xd = _rows_operand(workloads.normal((M, K), 1.0, seed=31))
    wq, ws, wd = _rows_operand(workloads.normal((N, K), 0.02, seed=32))
    big = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:, 32:32 + N]
    ref = oracle.gemm(xd, wd)
    for _ in range(3):
        mxq.gemm(xq, xs, wq, ws, M, N, K, out=out)
    torch.cuda.synchronize()
    assert_gemm_close(out, ref, "strided out")
    assert torch.all(big[:, :32] == 7.0) and torch.all(big[:, 32 + N:] == 7.0)


def test_empty_contraction_writes_zeros():
    mxq, _, _ = _mods()
    y = torch.full((5, 32), 3.0, dtype=torch.bfloat16, device="cuda")
    dummy = torch.zeros(512, dtype=torch.uint8, device="cuda")
    mxq.gemm(dummy, dummy, dummy, dummy, 5, 32, 0, out=y)
    torch.cuda.synchronize()
    assert torch.all(y == 0)


def test_device_status_clean():
    mxq, _, _ = _mods()
    assert mxq.get_device_status() == 0


# ---- full sizes of the workloads (sampled rows) ---------------------------------------

def _sample_rows(M, n=192, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, M // 2, M - 129, M - 1]
    rows = np.unique(np.concatenate([rng.choice(M, size=min(n, M), replace=False), [r for r in fixed if 0 <= r < M]]))
    return rows.astype(np.int64)


def test_full_linear_train_three_gemms():
    """X [8192, 4096], W [4096, 4096], dY [8192, 4096]: forward, dgrad, wgrad."""
    mxq, workloads, oracle = _mods()
    d = workloads.linear_train()
    M, N, K = 8192, 4096, 4096
    (xr, xrs, xrd), (xc, xcs, xcd) = _dual_operand(d["X"])
    (wr, wrs, wrd), (wc, wcs, wcd) = _dual_operand(d["W"])
    (gr, grs, grd), (gc, gcs, gcd) = _dual_operand(d["dY"])
    y = mxq.gemm(xr, xrs, wr, wrs, M, N, K)
    dx = mxq.gemm(gr, grs, wc, wcs, M, K, N)
    dw = mxq.gemm(gc, gcs, xc, xcs, N, K, M)
    torch.cuda.synchronize()
    r = _sample_rows(M, seed=1)
    assert_gemm_close(y[torch.from_numpy(r).cuda()], oracle.gemm(xrd, wrd, rows=r), "forward")
    assert_gemm_close(dx[torch.from_numpy(r).cuda()], oracle.gemm(grd, wcd, rows=r), "dgrad")
    r2 = _sample_rows(N, seed=2)
    assert_gemm_close(dw[torch.from_numpy(r2).cuda()], oracle.gemm(gcd, xcd, rows=r2), "wgrad")


def test_full_weight_32x32_path():
    """W [7168, 7168] 32x32-quantized; X, dY [4096, 7168]: forward and N-major dgrad."""
    mxq, workloads, oracle = _mods()
    d = workloads.weight_32x32()
    M, n, k = 4096, 7168, 7168
    q, sf, sb = mxq.quant_32x32(d["W"].cuda())
    oq, osf, _ = oracle.quant_32x32(bits(d["W"]))
    w_deq = oracle.dequant_rows(oq, osf)
    xq, xs, xd = _rows_operand(d["X"])
    gq, gs, gd = _rows_operand(d["dY"])
    y = mxq.gemm(xq, xs, q, sf, M, n, k)
    dx = mxq.gemm(gq, gs, q, sb, M, k, n, b_mn_major=True)
    torch.cuda.synchronize()
    r = _sample_rows(M, seed=3)
    rt = torch.from_numpy(r).cuda()
    assert_gemm_close(y[rt], oracle.gemm(xd, w_deq, rows=r), "32x32 forward")
    assert_gemm_close(dx[rt], oracle.gemm(gd, np.ascontiguousarray(w_deq.T), rows=r), "32x32 dgrad")


def _sweep_three_gemms(K, n_rows, seed):
    """The sweep layer M = 16384, K = N: dual quantization of X, W, dY checked
    byte for byte against the oracle, then the forward by the single-GEMM call
    and dgrad + wgrad by the one-launch pair the benchmark times, on sampled
    output rows (operand rows quantized by the oracle where the product needs
    only those rows)."""
    mxq, workloads, oracle = _mods()
    from _util import u8
    d = workloads.sweep(K)
    M = 16384
    N = K
    X, W, dY = d["X"], d["W"], d["dY"]
    q = {}
    for name, t in (("X", X), ("W", W), ("dY", dY)):
        qr, sr, qc, sc = mxq.quant_1x32_dual(t.cuda())
        torch.cuda.synchronize()
        oqr, osr, oqc, osc = oracle.quant_dual(bits(t))
        assert np.array_equal(u8(qr), oqr) and np.array_equal(u8(sr), oracle.scale_tiled(osr)), f"{name} row copy"
        assert np.array_equal(u8(qc), oqc) and np.array_equal(u8(sc), oracle.scale_tiled(osc)), f"{name} col copy"
        del oqr, osr, oqc, osc
        q[name] = (qr, sr, qc, sc)
    xr, xrs, xc, xcs = q["X"]
    wr, wrs, wc, wcs = q["W"]
    gr, grs, gc, gcs = q["dY"]
    y = mxq.gemm(xr, xrs, wr, wrs, M, N, K)
    dx, dw = mxq.gemm_multi([dict(a_q=gr, a_s=grs, b_q=wc, b_s=wcs, M=M, N=K, K=N),
                             dict(a_q=gc, a_s=gcs, b_q=xc, b_s=xcs, M=N, N=K, K=M)])
    torch.cuda.synchronize()
    del q, xr, xrs, wr, wrs, gr, grs, wc, wcs, gc, gcs, xc, xcs
    deq_rows = lambda t: oracle.dequant_rows(*oracle.quant_rows(bits(t)))
    r = _sample_rows(M, n=n_rows, seed=seed)
    rt = torch.from_numpy(r).cuda()
    assert_gemm_close(y[rt], oracle.gemm(deq_rows(X[r]), deq_rows(W)), f"forward sweep {K}")
    assert_gemm_close(dx[rt], oracle.gemm(deq_rows(dY[r]), deq_rows(W.t().contiguous())), f"dgrad sweep {K}")
    r2 = _sample_rows(N, n=n_rows, seed=seed + 1)
    gt_rows = deq_rows(dY.t()[r2].contiguous())
    assert_gemm_close(dw[torch.from_numpy(r2).cuda()], oracle.gemm(gt_rows, deq_rows(X.t().contiguous())),
                      f"wgrad sweep {K}")


def test_full_sweep_4096_forward():
    mxq, workloads, oracle = _mods()
    d = workloads.sweep(4096)
    M, K = 16384, 4096
    xq, xs, xd = _rows_operand(d["X"])
    wq, ws, wd = _rows_operand(d["W"])
    y = mxq.gemm(xq, xs, wq, ws, M, K, K)
    torch.cuda.synchronize()
    r = _sample_rows(M, seed=4)
    assert_gemm_close(y[torch.from_numpy(r).cuda()], oracle.gemm(xd, wd, rows=r), "sweep 4096")


def test_full_sweep_4096_three_gemms():
    _sweep_three_gemms(4096, n_rows=128, seed=41)


def test_full_sweep_7168_three_gemms():
    _sweep_three_gemms(7168, n_rows=96, seed=71)


def test_full_sweep_16384_three_gemms():
    """The largest linear layer, X, dY [16384, 16384], W [16384, 16384]: forward by the
    single-GEMM call, dgrad and wgrad by the one-launch pair the benchmark times;
    64 sampled output rows of each against the oracle (operand rows quantized by the
    oracle one by one where the product needs only those rows)."""
    mxq, workloads, oracle = _mods()
    d = workloads.sweep(16384)
    M = N = K = 16384
    X, W, dY = d["X"], d["W"], d["dY"]
    xr, xrs, xc, xcs = mxq.quant_1x32_dual(X.cuda())
    wr, wrs, wc, wcs = mxq.quant_1x32_dual(W.cuda())
    gr, grs, gc, gcs = mxq.quant_1x32_dual(dY.cuda())
    y = mxq.gemm(xr, xrs, wr, wrs, M, N, K)
    dx, dw = mxq.gemm_multi([dict(a_q=gr, a_s=grs, b_q=wc, b_s=wcs, M=M, N=K, K=N),
                             dict(a_q=gc, a_s=gcs, b_q=xc, b_s=xcs, M=N, N=K, K=M)])
    torch.cuda.synchronize()
    del xr, xrs, wr, wrs, gr, grs, wc, wcs, gc, gcs, xc, xcs
    r = _sample_rows(M, n=64, seed=5)
    rt = torch.from_numpy(r).cuda()
    deq_rows = lambda t: oracle.dequant_rows(*oracle.quant_rows(bits(t)))
    w_deq = deq_rows(W)                                        # forward B: W's row copy
    assert_gemm_close(y[rt], oracle.gemm(deq_rows(X[r]), w_deq, rows=None), "forward 16384")
    del w_deq
    wt_deq = deq_rows(W.t().contiguous())                      # dgrad B: W's column copy
    assert_gemm_close(dx[rt], oracle.gemm(deq_rows(dY[r]), wt_deq, rows=None), "dgrad 16384")
    del wt_deq
    xt_deq = deq_rows(X.t().contiguous())                      # wgrad B: X's column copy
    gt_rows = deq_rows(dY.t()[r].contiguous())                 # wgrad A: sampled rows of dY's column copy
    assert_gemm_close(dw[rt], oracle.gemm(gt_rows, xt_deq, rows=None), "wgrad 16384")


def test_c_abi_gemm_layout_argument():
    """mxq_gemm_bf16out through the C ABI: MMA-tiled scales compute, row-major
    scales are refused before anything is launched (output untouched)."""
    import ctypes
    mxq, workloads, oracle = _mods()
    M, N, K = 200, 256, 320
    xq, xs, xd = _rows_operand(workloads.normal_with_outliers((M, K), seed=21))
    wq, ws, wd = _rows_operand(workloads.normal((N, K), 0.02, seed=22))
    y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    L = mxq.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.mxq_gemm_bf16out(p(xq), p(xs), p(wq), p(ws), M, N, K, 0, p(y), N, mxq.ROWMAJOR, mxq._stream())
    torch.cuda.synchronize()
    assert st == 1 and torch.all(y == 3.0)
    st = L.mxq_gemm_bf16out(p(xq), p(xs), p(wq), p(ws), M, N, K, 0, p(y), N, mxq.TILED, mxq._stream())
    torch.cuda.synchronize()
    assert st == 0
    assert_gemm_close(y, oracle.gemm(xd, wd), "C ABI forward")


def test_small_linear_exhaustive():
    """The 256 x 512 x 512 linear forward, every output compared."""
    mxq, workloads, oracle = _mods()
    d = workloads.linear_fwd_small()
    xq, xs, xd = _rows_operand(d["X"])
    wq, ws, wd = _rows_operand(d["W"])
    y = mxq.gemm(xq, xs, wq, ws, 256, 512, 512)
    torch.cuda.synchronize()
    assert_gemm_close(y, oracle.gemm(xd, wd), "small linear")


@pytest.mark.parametrize("M,N,K,pad", [(300, 272, 256, 8), (1000, 4112, 512, 24), (129, 528, 128, 40)])
def test_strided_output_clipped_stores(M, N, K, pad):
    """Output rows ldy = N + pad apart (pad not a multiple of 32 columns), N with a
    last 32-column chunk partly past N, ragged M: equal to the contiguous call bit
    for bit and to the oracle; the padding columns of every row keep their bytes
    (whole chunks leave as tiled stores clipped at N, the rest row by row)."""
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=M + 7)
    W = workloads.normal((N, K), 0.02, seed=N + 8)
    xq, xs, xd = _rows_operand(X)
    wq, ws, wd = _rows_operand(W)
    big = torch.full((M, N + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    y = mxq.gemm(xq, xs, wq, ws, M, N, K, out=big[:, :N])
    y1 = mxq.gemm(xq, xs, wq, ws, M, N, K)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y1.view(torch.int16)), "strided output differs"
    assert torch.all(big[:, N:] == 7.0), "bytes past N in a row were written"
    r = _sample_rows(M, n=min(M, 96), seed=3)
    assert_gemm_close(y1[torch.from_numpy(r).cuda()], oracle.gemm(xd, wd, rows=r), f"strided {M}x{N}x{K}")
