"""Pins for the oracle's grouped column quantization (token-axis groups inside
each MoE expert, used by the expert weight gradient).

The pages quantize MoE expert layers (torchtitan-npu tutorial, "MoE 专家层
(Grouped MM)"; MindSpeed RFC section 2.2) but give no rule for token groups
that run past an expert's last token; the reading taken is zero padding, with
groups starting at each expert's first token.  Checked here by reduction to
the already pinned row quantizer applied to each expert's zero-padded block,
against the plain column copy when an expert is a multiple of 32 tokens, and
for the padding and empty-expert structure.
"""
import numpy as np
import pytest
import torch


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


@pytest.mark.parametrize("sizes", [[0, 5, 0, 300, 1, 130], [128], [33, 31, 129, 127, 0], [1, 1, 1]])
def test_grouped_cols_equals_padded_block_quant(orc, sizes):
    off = _offsets(sizes)
    M = int(off[-1])
    C = 96
    g = torch.Generator().manual_seed(len(sizes) * 100 + M)
    x = torch.randn(M, C, generator=g) * torch.pow(2.0, torch.randint(-8, 9, (M, 1), generator=g).float())
    xb = _bits(x)
    P, L = orc.padded_slots(off)
    cap = int(P[-1] + L[-1]) + 128
    q, s = orc.quant_cols_grouped(xb, off, cap)
    for e, m in enumerate(sizes):
        blk = np.zeros((int(L[e]), C), np.uint16)            # the expert's rows, zero-padded
        blk[:m] = xb[off[e]:off[e + 1]]
        if L[e] == 0:
            continue
        _, _, qc, sc = orc.quant_dual(blk, want_row=False, want_col=True)
        assert np.array_equal(q[:, P[e]:P[e] + L[e]], qc)
        assert np.array_equal(s[:, P[e] // 32:(P[e] + L[e]) // 32], sc)
        # groups wholly past the expert's tokens are zero payload with scale code 0
        full_groups = -(-m // 32)
        assert np.all(s[:, P[e] // 32 + full_groups:(P[e] + L[e]) // 32] == 0)
        assert np.all(q[:, P[e] + m:P[e] + L[e]] & 0x7F == 0)
    # nothing past the last slot is written
    end = int(P[-1] + L[-1])
    assert np.all(q[:, end:] == 0) and np.all(s[:, end // 32:] == 0)


def test_grouped_cols_single_aligned_expert_is_plain_column_copy(orc):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(256, 64, generator=g)
    xb = _bits(x)
    q, s = orc.quant_cols_grouped(xb, np.array([0, 256]), 256)
    _, _, qc, sc = orc.quant_dual(xb, want_row=False)
    assert np.array_equal(q, qc) and np.array_equal(s, sc)


def test_grouped_cols_expert_boundary_changes_groups(orc):
    """Tokens of different experts never share a scale: with a boundary at 16,
    the first group of expert 1 starts at token 16, not at token 0."""
    x = torch.ones(48, 32)
    x[0:16] *= 64.0        # expert 0: large values
    xb = _bits(x)
    q, s = orc.quant_cols_grouped(xb, np.array([0, 16, 48]), 256)
    assert np.all(s[:, 0] == 127 + 6 - 8)          # amax 64 -> e = -2
    assert np.all(s[:, 128 // 32] == 127 - 8)      # expert 1 alone: amax 1 -> e = -8


@pytest.mark.parametrize("sizes", [[0, 5, 0, 300, 1, 130], [33, 31, 129, 127, 0]])
def test_grouped_cols_e5m2_equals_padded_block_row_quant(orc, sizes):
    """The E5M2 destination type (MindSpeed RFC section 3.5.2.3) of the same
    layout: each expert's zero-padded block, transposed, quantized by the
    pinned E5M2 row quantizer."""
    off = _offsets(sizes)
    M = int(off[-1])
    C = 64
    g = torch.Generator().manual_seed(M + 5)
    x = torch.randn(M, C, generator=g) * torch.pow(2.0, torch.randint(-20, 21, (M, 1), generator=g).float())
    xb = _bits(x)
    P, L = orc.padded_slots(off)
    cap = int(P[-1] + L[-1]) + 128
    q, s = orc.quant_cols_grouped(xb, off, cap, fmt=1)
    q4, _ = orc.quant_cols_grouped(xb, off, cap, fmt=0)
    assert not np.array_equal(q, q4)                     # the format reaches the payload
    for e, m in enumerate(sizes):
        if L[e] == 0:
            continue
        blk = np.zeros((int(L[e]), C), np.uint16)
        blk[:m] = xb[off[e]:off[e + 1]]
        qe, se = orc.quant_rows_fmt(np.ascontiguousarray(blk.T), 1)
        assert np.array_equal(q[:, P[e]:P[e] + L[e]], qe)
        assert np.array_equal(s[:, P[e] // 32:(P[e] + L[e]) // 32], se)
