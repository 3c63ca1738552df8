"""Pins for the oracle's 32x32 block quantizer with the E5M2 destination type.

MindSpeed RFC "Add MXFP8-32x32 quantization support to FSDP", section 3.5.2.3:
``process_quant_result_fn`` serves both the mxfp8 and the mxfp8-32x32 recipes
and takes dst_type float8_e4m3fn or float8_e5m2; section 3.1: one exponent per
32x32 tile of the weight, one payload for forward and backward.  E5M2 is OCP
float8_e5m2 (largest finite 57344); rceil then uses 57344 in place of 448.

Checked against a hand-derived tile (tests/golden), PyTorch's float8_e5m2 cast
of the exactly scaled tile, the invariants rceil implies, transpose
consistency, and the reduction to the pinned 1x32 E5M2 quantizer.
"""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x):
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def _spread(n, k, seed):
    """BF16 [n, k] with a different power-of-two magnitude per 32x32 tile."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, k, generator=g, dtype=torch.float64)
    e = torch.randint(-50, 50, (n // 32, k // 32), generator=g).double()
    x = x * torch.pow(2.0, e).repeat_interleave(32, 0).repeat_interleave(32, 1)
    return x.float().to(torch.bfloat16)


def test_hand_example_32x32_e5m2(orc):
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        t = json.load(f)["tile_32x32_e5m2"]
    w = torch.zeros(32, 32, dtype=torch.bfloat16)
    for rc, v in t["values"].items():
        r, c = map(int, rc.split(","))
        w[r, c] = float(v)
        assert float(w[r, c]) == float(v)
    q, s_fwd, s_bwd = orc.quant_32x32(_bits(w), fmt=1)
    assert np.all(s_fwd == t["tile_scale_code"]) and np.all(s_bwd == t["tile_scale_code"]), t["why"]
    for rc, code in t["payload"].items():
        r, c = map(int, rc.split(","))
        assert q[r, c] == int(code, 16), (rc, t["why"])
    q1, s1 = orc.quant_rows_fmt(_bits(w), 1)
    assert s1[5, 0] == t["row5_1x32_scale_code"] and q1[5, 3] == int(t["row5_1x32_payload_col3"], 16)


def test_32x32_e5m2_matches_torch_cast_and_rceil_invariants(orc):
    w = _spread(96, 160, 11)
    bits = _bits(w)
    q, s_fwd, s_bwd = orc.quant_32x32(bits, fmt=1)
    e = s_fwd.astype(np.int64) - 127                    # [96, 5], repeated down each tile
    x = orc.bf16_to_double(bits)
    scaled = x * np.exp2(-np.repeat(e, 32, axis=1))
    assert np.all(np.abs(scaled) <= 57344.0)
    ref = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    qv = np.abs(orc.e5m2_decode(q)).reshape(3, 32, 5, 32).max(axis=(1, 3))
    assert np.all((qv >= 28672.0) & (qv <= 57344.0))     # the tile's amax element lands in the top binade
    # every row of a tile carries the tile's code; s_bwd holds the same codes transposed
    t = s_fwd.reshape(3, 32, 5)
    assert np.all(t == t[:, :1, :])
    assert np.array_equal(s_bwd.reshape(5, 32, 3)[:, 0, :], t[:, 0, :].T)


def test_32x32_e5m2_transpose_consistency(orc):
    bits = _bits(_spread(64, 128, 12))
    q, s_fwd, s_bwd = orc.quant_32x32(bits, fmt=1)
    qt, sft, sbt = orc.quant_32x32(np.ascontiguousarray(bits.T), fmt=1)
    assert np.array_equal(qt, q.T)
    assert np.array_equal(sft, s_bwd) and np.array_equal(sbt, s_fwd)


def test_32x32_e5m2_reduces_to_1x32_when_rows_share_amax(orc):
    """With every 32-element row group of a tile at the same amax, the tile
    exponent is each group's own, so the payload equals the 1x32 E5M2 one."""
    g = torch.Generator().manual_seed(13)
    x = torch.rand(64, 64, generator=g, dtype=torch.float64) * 0.9
    x[:, ::32] = 3.0                                      # each row group's amax, exactly 3
    x[1::2] *= -1.0
    w = x.float().to(torch.bfloat16)
    q, s_fwd, _ = orc.quant_32x32(_bits(w), fmt=1)
    q1, s1 = orc.quant_rows_fmt(_bits(w), 1)
    assert np.array_equal(q, q1) and np.array_equal(s_fwd, s1)


def test_32x32_e5m2_special_tiles_and_default_format(orc):
    w = _spread(64, 64, 14)
    w[0:32, 32:64] = 0.0
    w[33, 7] = float("inf")
    w[40, 3] = -w[40, 3].abs()
    bits = _bits(w)
    q, s_fwd, s_bwd = orc.quant_32x32(bits, fmt=1)
    assert np.all(s_fwd[0:32, 1] == 0) and np.all(q[0:32, 32:64] == 0)       # zero tile
    assert np.all(s_fwd[32:64, 0] == 0xFF) and np.all(s_bwd[0:32, 1] == 0xFF)
    sign = (bits[32:64, 0:32] >> 15).astype(np.uint8) << 7
    assert np.array_equal(q[32:64, 0:32], sign | 0x7F)                        # NaN/Inf tile
    # fmt 0 is the pinned E4M3 quantizer
    q4, f4, b4 = orc.quant_32x32(bits, fmt=0)
    q0, f0, b0 = orc.quant_32x32(bits)
    assert np.array_equal(q4, q0) and np.array_equal(f4, f0) and np.array_equal(b4, b0)
