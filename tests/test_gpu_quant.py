"""GPU parity of the quantizers: payload and scale bytes must equal the
oracle's exactly, in the plain and the MMA-tiled scale layouts.

1x32 groups: one E8M0 scale per 32 elements (torchtitan-npu tutorial,
"MXFP8 与 HiF8 架构原理速览"); dual-axis forward/backward copies and the
32x32 single payload (MindSpeed RFC, sections 3.1, 3.3.3).
"""
import numpy as np
import pytest
import torch

from _util import bits, gpu_or_skip, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _mxq():
    from mxfp8_microscaled_precision_gb300 import mxq
    return mxq


def _hard(rows, cols, seed, nonfinite=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float64)
    ge = torch.randint(-126, 110, (rows, cols // 32, 1), generator=g).double()
    x = (x.view(rows, cols // 32, 32) * torch.pow(2.0, ge)).view(rows, cols)
    x = torch.where(torch.rand(rows, cols, generator=g) < 0.01, x * 100, x)
    xb = x.float().to(torch.bfloat16)
    xb[0, :32] = 0.0
    if rows > 1 and cols >= 64:
        xb[1, 32:64] = -0.0
        xb[1, :32] = 1e-39
    if rows > 2 and cols >= 64:
        xb[2, :64] = 3.0
        xb[2, 0] = 1.75 * 2.0 ** 20
        xb[2, 32] = -1.7578125 * 2.0 ** 20
    if nonfinite and rows > 4 and cols >= 64:
        xb[3, 5] = float("nan")
        xb[4, 40] = float("-inf")
    return xb


def _check_dual(x_cpu, layout, row=True, col=True):
    from oracle import oracle
    mxq = _mxq()
    xd = x_cpu.cuda()
    qr, sr, qc, sc = mxq.quant_1x32_dual(xd, row=row, col=col, layout=layout)
    torch.cuda.synchronize()
    oqr, osr, oqc, osc = oracle.quant_dual(bits(x_cpu), want_row=row, want_col=col)
    conv = oracle.scale_tiled if layout == "tiled" else (lambda s: s)
    if row:
        assert np.array_equal(u8(qr), oqr), "row payload"
        assert np.array_equal(u8(sr), conv(osr)), "row scales"
    if col:
        assert np.array_equal(u8(qc), oqc), "col payload"
        assert np.array_equal(u8(sc), conv(osc)), "col scales"


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
@pytest.mark.parametrize("shape", [(256, 512), (96, 160), (32, 32), (160, 4096), (4096, 96), (416, 288)])
def test_dual_matches_oracle(shape, layout):
    from mxfp8_microscaled_precision_gb300 import workloads
    x = workloads.normal_with_outliers(shape, seed=shape[0] * 7 + shape[1])
    _check_dual(x, layout)


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
@pytest.mark.parametrize("shape", [(1, 32), (130, 96), (257, 544), (3, 4096)])
def test_row_only_ragged_rows(shape, layout):
    from mxfp8_microscaled_precision_gb300 import workloads
    x = workloads.normal(shape, 1.0, seed=shape[0] + shape[1])
    _check_dual(x, layout, row=True, col=False)


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
def test_col_only(layout):
    from mxfp8_microscaled_precision_gb300 import workloads
    _check_dual(workloads.student_t((192, 320), seed=5), layout, row=False, col=True)


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
def test_dual_hard_inputs(layout):
    """Huge dynamic range, outliers, zeros, -0, BF16 subnormals, rceil
    boundary amaxes, NaN and Inf groups."""
    _check_dual(_hard(224, 352, seed=11), layout)


def test_strided_input():
    from oracle import oracle
    mxq = _mxq()
    big = torch.randn(160, 512).to(torch.bfloat16)
    x = big[:, 64:64 + 384]
    xd = big.cuda()[:, 64:64 + 384]               # row stride 512, not 384
    assert xd.stride(0) == 512
    qr, sr, qc, sc = mxq.quant_1x32_dual(xd)
    torch.cuda.synchronize()
    oqr, osr, oqc, osc = oracle.quant_dual(bits(x.contiguous()))
    assert np.array_equal(u8(qr), oqr) and np.array_equal(u8(sr), oracle.scale_tiled(osr))
    assert np.array_equal(u8(qc), oqc) and np.array_equal(u8(sc), oracle.scale_tiled(osc))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_column_copy_at_16_byte_alignment(fmt):
    """The column copy into a buffer 16 (not 32) bytes past an aligned address
    (the ABI's minimum alignment, where 256-bit stores are not allowed): the
    same bytes as into an aligned buffer and as the oracle."""
    from oracle import oracle
    mxq = _mxq()
    R, C = 192, 320
    x = torch.randn(R, C).to(torch.bfloat16)
    xd = x.cuda()
    base = torch.full((C * R + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    off = (32 - base.data_ptr() % 32) % 32 + 16            # 16 bytes past a 32-byte boundary
    qc_odd = base[off:off + C * R].view(C, R)
    assert qc_odd.data_ptr() % 32 == 16
    sc = torch.empty(mxq.scale_bytes(C, R), dtype=torch.uint8, device="cuda")
    _, _, qc_al, sc_al, = mxq.quant_1x32_dual_batched(xd, row=False, fmt=fmt)
    q_b = qc_odd.view(1, C, R)
    mxq.quant_1x32_dual_batched(xd, row=False, fmt=fmt, out=(None, None, q_b, sc.view(1, -1)))
    torch.cuda.synchronize()
    assert torch.equal(qc_odd, qc_al[0]) and torch.equal(sc, sc_al[0].reshape(-1))
    assert torch.all(base[:off] == 0xEE) and torch.all(base[off + C * R:] == 0xEE), "bytes outside were written"
    oq, _ = oracle.quant_rows_fmt(np.ascontiguousarray(bits(x).T), 1 if fmt == "e5m2" else 0)
    assert np.array_equal(u8(qc_odd), oq)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_dual_row_copy_at_16_byte_alignment(fmt):
    """The dual kernel's row copy into a buffer 16 (not 32) bytes past an
    aligned address (its 32-byte runs then leave as two 16-byte stores), on a
    ragged shape (rows and columns past the last full tile): the same bytes as
    into an aligned buffer and as the oracle, nothing written outside."""
    from oracle import oracle
    mxq = _mxq()
    R, C = 224, 352                 # multiples of 32 (the column copy's groups), not of the 128-row tile
    x = torch.randn(R, C).to(torch.bfloat16)
    xd = x.cuda()
    base = torch.full((R * C + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    off = (32 - base.data_ptr() % 32) % 32 + 16
    qr_odd = base[off:off + R * C].view(1, R, C)
    assert qr_odd.data_ptr() % 32 == 16
    sr = torch.empty(mxq.scale_bytes(R, C), dtype=torch.uint8, device="cuda")
    qc = torch.empty((1, C, R), dtype=torch.uint8, device="cuda")
    sc = torch.empty(mxq.scale_bytes(C, R), dtype=torch.uint8, device="cuda")
    qr_al, sr_al, qc_al, sc_al = mxq.quant_1x32_dual_batched(xd, fmt=fmt)
    mxq.quant_1x32_dual_batched(xd, fmt=fmt, out=(qr_odd, sr.view(1, -1), qc, sc.view(1, -1)))
    torch.cuda.synchronize()
    assert torch.equal(qr_odd, qr_al) and torch.equal(sr, sr_al[0].reshape(-1))
    assert torch.equal(qc, qc_al) and torch.equal(sc, sc_al[0].reshape(-1))
    assert torch.all(base[:off] == 0xEE) and torch.all(base[off + R * C:] == 0xEE), "bytes outside were written"
    oq, os_ = oracle.quant_rows_fmt(bits(x), 1 if fmt == "e5m2" else 0)
    assert np.array_equal(u8(qr_odd[0]), oq)
    assert np.array_equal(u8(sr), oracle.scale_tiled(os_).reshape(-1))


def test_tiled_padding_is_zero():
    """Scale bytes outside the matrix in the tiled layout are written as 0."""
    mxq = _mxq()
    x = torch.randn(130, 96).to(torch.bfloat16).cuda()
    qr, sr, _, _ = mxq.quant_1x32_dual(x, col=False)
    s = u8(sr).reshape(-1)
    assert s.size == 256 * 4
    # rows 130..255 of every atom, and group 3 of every row, are padding
    atoms = s.reshape(2, 32, 4, 4)                   # [band][r%32][(r%128)/32][g%4]
    assert np.all(atoms[..., 3] == 0)
    band1 = atoms[1]
    rows_in_band1 = np.arange(128).reshape(4, 32).T  # [r%32][(r%128)/32] -> r%128
    assert np.all(band1[rows_in_band1 >= 2] == 0)


def _check_32x32(w_cpu, layout):
    from oracle import oracle
    mxq = _mxq()
    q, sf, sb = mxq.quant_32x32(w_cpu.cuda(), layout=layout)
    torch.cuda.synchronize()
    oq, osf, osb = oracle.quant_32x32(bits(w_cpu))
    conv = oracle.scale_tiled if layout == "tiled" else (lambda s: s)
    assert np.array_equal(u8(q), oq), "payload"
    assert np.array_equal(u8(sf), conv(osf)), "s_fwd"
    assert np.array_equal(u8(sb), conv(osb)), "s_bwd"


@pytest.mark.parametrize("layout", ["tiled", "rowmajor"])
@pytest.mark.parametrize("shape", [(64, 96), (128, 128), (384, 256), (96, 4096), (4096, 160)])
def test_32x32_matches_oracle(shape, layout):
    from mxfp8_microscaled_precision_gb300 import workloads
    _check_32x32(workloads.normal(shape, 0.02, seed=shape[0] + 3 * shape[1]), layout)


def test_32x32_hard_inputs():
    _check_32x32(_hard(192, 320, seed=12), "tiled")
    _check_32x32(_hard(192, 320, seed=13), "rowmajor")


# ---- full sizes of the workloads -------------------------------------------------

def test_full_linear_train_dual():
    """X, W, dY of the 8192 x 4096 x 4096 linear layer, dual-axis, tiled scales."""
    from mxfp8_microscaled_precision_gb300 import workloads
    d = workloads.linear_train()
    for name in ("X", "W", "dY"):
        _check_dual(d[name], "tiled")


def test_full_weight_32x32():
    from mxfp8_microscaled_precision_gb300 import workloads
    _check_32x32(workloads.normal((7168, 7168), 0.02, seed=workloads.seed_for("weight_32x32", "W")), "tiled")


def test_full_moe_row_quant():
    """The routed expert inputs: A [131072, 4096] and H [131072, 2048], row copy."""
    from mxfp8_microscaled_precision_gb300 import workloads
    d = workloads.moe_grouped(weights=False)
    _check_dual(d["A"], "tiled", row=True, col=False)
    _check_dual(d["H"], "tiled", row=True, col=False)


def test_full_sweep_16384_dual():
    from mxfp8_microscaled_precision_gb300 import workloads
    x = workloads.student_t((16384, 16384), seed=workloads.seed_for("sweep_16384", "X"))
    _check_dual(x, "tiled")
