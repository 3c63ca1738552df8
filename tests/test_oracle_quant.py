"""Pins for the oracle's quantizers (1x32 rows, dual-axis, 32x32 blocks) and
for the MMA-tiled scale layout.

Sources: MXFP8 shares one E8M0 scale per 32 consecutive elements (torchtitan-npu
tutorial, "MXFP8 与 HiF8 架构原理速览"); the dual-axis quantizer emits a forward
and a backward copy and the 32x32 variant one payload whose forward and
backward scales differ only in layout (MindSpeed RFC, sections 3.1, 3.3.2,
3.3.3).  The checks use invariants that follow from the rceil rule and the
E4M3 format, a library reduction (PyTorch's float8_e4m3fn conversion of the
exactly scaled values) and structural identities (transposes).
"""
import numpy as np
import pytest
import torch


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _hard_input(rows, cols, seed):
    """BF16 data whose 32-groups span huge dynamic ranges, with outliers,
    exact zeros, negative zeros, subnormals and rceil boundary amaxes."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float64)
    grp_exp = torch.randint(-120, 110, (rows, cols // 32, 1), generator=g).to(torch.float64)
    x = (x.view(rows, cols // 32, 32) * torch.pow(2.0, grp_exp)).view(rows, cols)
    out = torch.rand(rows, cols, generator=g) < 0.01
    x = torch.where(out, x * 100, x)
    xb = x.to(torch.float32).to(torch.bfloat16)
    xb[0, :32] = 0.0
    xb[0, 32:64] = -0.0
    xb[1, :32] = torch.tensor(1e-39).to(torch.bfloat16)   # bf16 subnormal
    xb[1, 32:64] = 0.5
    xb[1, 32] = 448.0                                      # amax exactly 448 -> e = 0
    xb[2, 0:64] = 3.0
    xb[2, 0] = 1.75 * 2.0 ** 20                             # f == 0.875 boundary
    xb[2, 32] = -1.7578125 * 2.0 ** 20                      # just above the boundary
    return xb


def _deq(orc, q, s):
    return orc.dequant_rows(q, s)


def _check_group_invariants(orc, x_bits, q, s):
    """Per 32-group along the last axis: rceil minimality, no overflow,
    amax element lands in [224, 448], error bound, and payload equal to
    PyTorch's float8_e4m3fn conversion of x * 2^-e."""
    R, C = x_bits.shape
    x = orc.bf16_to_double(x_bits)
    e = s.astype(np.int64) - 127
    xg = x.reshape(R, C // 32, 32)
    amax = np.abs(xg).max(axis=2)
    scaled = xg * np.power(2.0, -e)[..., None]
    assert np.all(np.abs(scaled) <= 448.0)
    nz = amax > 0
    # minimal exponent: one step smaller would overflow (unless clamped)
    clamped = e == -127
    assert np.all((amax * np.power(2.0, -(e - 1)) > 448.0) | clamped | ~nz)
    qv = orc.e4m3_decode(q).reshape(R, C // 32, 32)
    qmax = np.abs(qv).max(axis=2)
    sel = nz & ~clamped
    assert np.all((qmax[sel] >= 224.0) & (qmax[sel] <= 448.0))
    assert np.all(s[~nz] == 0) and np.all(np.abs(qv[~nz]) == 0)
    deq = qv * np.power(2.0, e)[..., None]
    err = np.abs(deq - xg)
    big = np.abs(scaled) >= 2.0 ** -6
    assert np.all(err[big] <= 2.0 ** -4 * np.abs(xg[big]))
    small_bound = np.broadcast_to(np.power(2.0, e - 10)[..., None], xg.shape)
    assert np.all(err[~big] <= small_bound[~big])
    # library reduction: the payload is torch's RNE cast of the exactly scaled
    # value (float32 holds it exactly unless it is far below E4M3's range,
    # where the code must be a signed zero)
    sc = scaled.reshape(R, C)
    tiny = np.abs(sc) < 2.0 ** -100
    assert np.all(q[tiny] & 0x7F == 0)
    assert np.all(np.signbit(sc[tiny]) == (q[tiny] >> 7).astype(bool))
    f32 = np.where(tiny, 0.0, sc).astype(np.float32)
    assert np.all(f32[~tiny].astype(np.float64) == sc[~tiny])
    ref = torch.from_numpy(f32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref[~tiny], q[~tiny])


def test_quant_rows_invariants(orc):
    xb = _hard_input(96, 256, seed=1)
    q, s = orc.quant_rows(_bf16_bits(xb))
    _check_group_invariants(orc, _bf16_bits(xb), q, s)
    assert s[0, 0] == 0 and np.all(q[0, :32] == 0x00)
    assert s[0, 1] == 0 and np.all(q[0, 32:64] == 0x80)   # -0 keeps its sign
    assert s[1, 1] == 127 and q[1, 32] == 0x7E             # 448 -> scale 2^0, code 448
    assert s[2, 0] == 127 + 12 and q[2, 0] == 0x7E         # 1.75*2^20 = 448*2^12
    assert s[2, 1] == 127 + 13 and q[2, 32] == 0xF6        # 450*2^12 / 2^13 = 225 -> 224


def test_quant_nonfinite_groups(orc):
    xb = torch.ones(2, 64, dtype=torch.bfloat16)
    xb[0, 3] = float("nan")
    xb[1, 40] = float("-inf")
    xb[1, 41] = -2.0
    q, s = orc.quant_rows(_bf16_bits(xb))
    assert s[0, 0] == 0xFF and np.all(q[0, :32] & 0x7F == 0x7F)
    assert s[0, 1] == 127 - 8 and s[1, 0] == 127 - 8       # amax 1 -> e = -8
    assert s[1, 1] == 0xFF and q[1, 41] == 0xFF and q[1, 40] == 0xFF and q[1, 32] == 0x7F


def test_quant_dual_col_is_row_of_transpose(orc):
    xb = _hard_input(64, 96, seed=2)
    bits = _bf16_bits(xb)
    q_row, s_row, q_col, s_col = orc.quant_dual(bits)
    qr2, sr2 = orc.quant_rows(bits)
    assert np.array_equal(q_row, qr2) and np.array_equal(s_row, sr2)
    qt, st = orc.quant_rows(np.ascontiguousarray(bits.T))
    assert np.array_equal(q_col, qt) and np.array_equal(s_col, st)
    assert q_col.shape == (96, 64) and s_col.shape == (96, 2)
    _check_group_invariants(orc, np.ascontiguousarray(bits.T), q_col, s_col)


def test_quant_32x32_transpose_consistency(orc):
    xb = _hard_input(96, 160, seed=3)
    bits = _bf16_bits(xb)
    q, s_fwd, s_bwd = orc.quant_32x32(bits)
    qt, sft, sbt = orc.quant_32x32(np.ascontiguousarray(bits.T))
    assert np.array_equal(qt, q.T)
    assert np.array_equal(sft, s_bwd) and np.array_equal(sbt, s_fwd)
    # one exponent per tile, repeated along the 32 rows (fwd) / 32 cols (bwd)
    t = s_fwd[::32, :]
    assert np.array_equal(np.repeat(t, 32, axis=0), s_fwd)
    assert np.array_equal(np.repeat(t.T, 32, axis=0), s_bwd)


def test_quant_32x32_tile_invariants(orc):
    xb = _hard_input(64, 128, seed=4)
    bits = _bf16_bits(xb)
    q, s_fwd, _ = orc.quant_32x32(bits)
    x = orc.bf16_to_double(bits)
    e = s_fwd.astype(np.int64) - 127
    for i in range(2):
        for j in range(4):
            tile = x[32 * i:32 * i + 32, 32 * j:32 * j + 32]
            et = e[32 * i, j]
            amax = np.abs(tile).max()
            qt = orc.e4m3_decode(q[32 * i:32 * i + 32, 32 * j:32 * j + 32])
            assert np.all(np.abs(tile * 2.0 ** -et) <= 448)
            if amax > 0 and et > -127:
                assert amax * 2.0 ** -(et - 1) > 448
                assert 224 <= np.abs(qt).max() <= 448
    # the 32x32 payload is a valid 1x32 quantization of the same data with the
    # coarser (tile) exponent: payload = torch RNE cast of x * 2^-e_tile
    scaled = x * np.power(2.0, -np.repeat(e, 32, axis=1))
    ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(ref.numpy(), q)


def test_quant_32x32_reduces_to_1x32_when_rows_share_amax(orc):
    """If every row of a 32x32 tile has the same group amax, the tile exponent
    equals each row-group exponent, so both quantizers agree exactly."""
    g = torch.Generator().manual_seed(5)
    x = torch.rand(64, 64, generator=g, dtype=torch.float64) * 2 - 1
    for i in range(2):
        for j in range(2):
            x[32 * i:32 * i + 32, 32 * j] = 3.0 * 2.0 ** (4 * i - 3 * j)   # same amax per row group
            x[32 * i:32 * i + 32, 32 * j + 1:32 * j + 32] *= 2.0 ** (4 * i - 3 * j)
    bits = _bf16_bits(x)
    q, s_fwd, _ = orc.quant_32x32(bits)
    q1, s1 = orc.quant_rows(bits)
    assert np.array_equal(q, q1) and np.array_equal(s_fwd, s1)


@pytest.mark.parametrize("rows,groups", [(128, 4), (256, 8), (1, 1), (130, 5), (300, 128)])
def test_scale_tiled_layout(orc, rows, groups):
    g = np.random.default_rng(rows * 1000 + groups)
    s = g.integers(1, 255, size=(rows, groups), dtype=np.uint8)   # non-zero, so padding is visible
    t = orc.scale_tiled(s)
    rp, gp = -(-rows // 128) * 128, -(-groups // 4) * 4
    assert t.size == rp * gp
    # a permutation of the plain scales plus zero padding
    assert np.count_nonzero(t) == rows * groups
    assert np.array_equal(np.sort(t[t != 0]), np.sort(s.ravel()))
    # each 512-byte atom holds exactly the 128-row x 4-group block it names,
    # atoms of one 128-row band are consecutive, and a row's 4 scales are
    # 4 consecutive bytes (one 32-bit word per row per atom)
    per_band = gp // 4
    for r in {0, rows - 1, rows // 2, min(rows - 1, 37)}:
        for c in {0, groups - 1, groups // 2}:
            atom = t[((r // 128) * per_band + c // 4) * 512:][:512]
            word = atom.reshape(32, 4, 4)[r % 32, (r % 128) // 32]
            assert word[c % 4] == s[r, c]
