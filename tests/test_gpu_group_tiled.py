"""GPU parity of the group-tiled A scales and of the grouped GEMM that reads them.

mxq_scale_regroup_rows must equal, byte for byte, the oracle's group-tiled
layout of the oracle's own row quantization, and leave the bands past the last
group untouched; mxq_grouped_gemm_group_tiled must equal mxq_grouped_gemm on the
same payloads bit for bit (the same products, only the tiling of rows differs)
and the oracle within |gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref).  The MoE
expert layers run the quantized grouped matmul (torchtitan-npu tutorial,
"MoE 专家层 (Grouped MM)"; MindSpeed RFC section 2.2).
"""
import numpy as np
import pytest
import torch

from _util import assert_gemm_close, bits, gpu_or_skip, u8

pytestmark = pytest.mark.gpu

CASES = [
    ([0, 5, 0, 300, 1, 130], 256, 192),          # empty experts, unaligned starts
    ([0, 1, 127, 129, 0, 256, 3], 128, 256),      # sizes around the 128-row tile
    ([0, 0, 0, 500, 0], 384, 128),                # all empty but one
    ([1000], 256, 512),                           # one expert
    ([64] * 16, 128, 96),                         # many small experts, K tail
    ([37, 91, 200, 5, 0, 143, 300, 1], 512, 1024),
    ([1] * 40, 128, 64),                          # one-row experts
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _mods():
    from mxfp8_microscaled_precision_gb300 import mxq, workloads
    from oracle import oracle
    return mxq, workloads, oracle


def _operands(sizes, N, K, seed):
    mxq, workloads, _ = _mods()
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    A = workloads.normal_with_outliers((max(M, 1), K), seed=seed)[:M]
    B = workloads.normal((G * N, K), 0.02, seed=seed + 1)
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    return off, M, A, B, aq, as_, bq, bs


@pytest.mark.parametrize("sizes,N,K", CASES)
def test_regroup_matches_oracle(sizes, N, K):
    mxq, _, oracle = _mods()
    off, M, A, _, _, as_, _, _ = _operands(sizes, N, K, seed=sum(sizes) + K)
    G = len(sizes)
    cap = mxq.group_tiled_bands(M, G)
    out = torch.full((cap * ((K // 32 + 3) // 4) * 512,), 0xA5, dtype=torch.uint8, device="cuda")
    mxq.scale_regroup_rows(as_, M, K, torch.from_numpy(off).cuda(), bands_cap=cap, out=out)
    torch.cuda.synchronize()
    _, osa = oracle.quant_rows(bits(A))
    want = oracle.scale_group_tiled(osa, off)
    got = u8(out)
    assert np.array_equal(got[:want.size], want), "group-tiled scales"
    assert (got[want.size:] == 0xA5).all(), "bands past the last group were written"


@pytest.mark.parametrize("sizes,N,K", CASES)
def test_group_tiled_gemm_equals_grouped_gemm_and_oracle(sizes, N, K):
    mxq, _, oracle = _mods()
    off, M, A, B, aq, as_, bq, bs = _operands(sizes, N, K, seed=sum(sizes) + N + K)
    G = len(sizes)
    offd = torch.from_numpy(off).cuda()
    y_grid = mxq.grouped_gemm(aq, as_, bq, bs, offd, N, K)
    y = mxq.grouped_gemm_group_tiled(aq, mxq.scale_regroup_rows(as_, M, K, offd), bq, bs, offd, N, K)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_grid.view(torch.int16)), "differs from mxq_grouped_gemm"
    oa, osa = oracle.quant_rows(bits(A))
    ob, osb = oracle.quant_rows(bits(B))
    ref = oracle.grouped_gemm(oracle.dequant_rows(oa, osa), oracle.dequant_rows(ob, osb).reshape(G, N, K), off)
    assert_gemm_close(y, ref, f"group-tiled sizes={list(sizes)}")


def test_e5m2_rows_against_e4m3_weights():
    """The dgrad pairing: E5M2 A payload, E4M3 expert weights."""
    mxq, workloads, _ = _mods()
    sizes, N, K = [3, 0, 250, 129, 77], 256, 320
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M, G = int(off[-1]), len(sizes)
    A = workloads.normal((M, K), 1e-3, seed=41)
    B = workloads.normal((G * N, K), 0.02, seed=42)
    aq, as_, _, _ = mxq.quant_1x32_dual_batched(A.cuda(), col=False, fmt="e5m2")
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    offd = torch.from_numpy(off).cuda()
    y_grid = mxq.grouped_gemm(aq[0], as_[0], bq, bs, offd, N, K, a_fmt="e5m2")
    sg = mxq.scale_regroup_rows(as_[0], M, K, offd)
    y = mxq.grouped_gemm_group_tiled(aq[0], sg, bq, bs, offd, N, K, a_fmt="e5m2")
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_grid.view(torch.int16))


def test_rows_written_once():
    """Every expert's rows are written; nothing outside [0, M_total) is."""
    mxq, workloads, _ = _mods()
    sizes = [3, 0, 130, 0, 125]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M, N, K = int(off[-1]), 128, 64
    A = workloads.normal((M, K), 1.0, seed=9)
    B = workloads.normal((len(sizes) * N, K), 0.5, seed=10)
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    offd = torch.from_numpy(off).cuda()
    big = torch.full((M + 2, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = big[1:M + 1]
    mxq.grouped_gemm_group_tiled(aq, mxq.scale_regroup_rows(as_, M, K, offd), bq, bs, offd, N, K, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    assert torch.isnan(big[0]).all() and torch.isnan(big[M + 1]).all()


@pytest.mark.parametrize("offsets", [[0, 200, 50, 300], [0, 300, 0, 300, 0, 300, 0, 300, 300]])
def test_malformed_offsets_stay_in_bounds(offsets):
    """Decreasing offsets (the second case holds more bands than the cap, so
    the last ones are dropped): both calls finish, record no device error and
    write nothing outside the output and the scale buffer."""
    mxq, workloads, _ = _mods()
    M, N, K = 300, 128, 128
    G = len(offsets) - 1
    A = workloads.normal((M, K), 1.0, seed=11)
    B = workloads.normal((G * N, K), 0.5, seed=12)
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    offd = torch.tensor(offsets, dtype=torch.int64, device="cuda")
    cap = mxq.group_tiled_bands(M, G)
    sbuf = torch.full((cap * 512 + 1024,), 0x5A, dtype=torch.uint8, device="cuda")
    sg = mxq.scale_regroup_rows(as_, M, K, offd, bands_cap=cap, out=sbuf[:cap * 512])
    big = torch.full((M + 2, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    mxq.grouped_gemm_group_tiled(aq, sg, bq, bs, offd, N, K, bands_cap=cap, out=big[1:M + 1])
    torch.cuda.synchronize()
    assert mxq.get_device_status() == 0
    assert (sbuf[cap * 512:] == 0x5A).all()
    assert torch.isnan(big[0]).all() and torch.isnan(big[M + 1]).all()


def test_full_moe_forward_equals_grouped_gemm():
    """128 experts, 131072 routed rows (the MoE forward workload): gate_up and
    down through the group-tiled scales equal the 128-row-grid grouped GEMM bit
    for bit over the whole output."""
    mxq, workloads, _ = _mods()
    d = workloads.moe_grouped(weights=False)
    off = d["routing"].offsets
    offd = off.cuda()
    G, M = off.numel() - 1, int(off[-1])
    for a_cpu, K, wseed in ((d["A"], 4096, workloads.seed_for("moe_grouped", "W")),
                            (d["H"], 2048, workloads.seed_for("moe_grouped", "W_down"))):
        N = 4096
        W = workloads.normal((G * N, K), 0.02, seed=wseed, device="cuda")
        aq, as_, _, _ = mxq.quant_1x32_dual(a_cpu.cuda(), col=False)
        bq, bs, _, _ = mxq.quant_1x32_dual(W, col=False)
        del W
        y_grid = mxq.grouped_gemm(aq, as_, bq, bs, offd, N, K)
        y = mxq.grouped_gemm_group_tiled(aq, mxq.scale_regroup_rows(as_, M, K, offd), bq, bs, offd, N, K)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_grid.view(torch.int16)), f"K={K}"
        del y, y_grid
    assert mxq.get_device_status() == 0


def test_max_experts_mostly_empty():
    """G = 1024 (the largest supported), 60 non-empty experts of 1 to 300 rows
    scattered among empty ones, the last expert empty: the band scan runs over
    all 32 groups of 32 and the band lookup over 1024 experts."""
    mxq, workloads, oracle = _mods()
    rng = np.random.default_rng(2024)
    sizes = np.zeros(1024, np.int64)
    sizes[np.sort(rng.choice(1023, 60, replace=False))] = rng.integers(1, 301, 60)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M, N, K = int(off[-1]), 128, 256
    A = workloads.normal_with_outliers((M, K), seed=77)
    B = workloads.normal((1024 * N, K), 0.02, seed=78, device="cuda")
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B, col=False)
    offd = torch.from_numpy(off).cuda()
    sg = mxq.scale_regroup_rows(as_, M, K, offd)
    y = mxq.grouped_gemm_group_tiled(aq, sg, bq, bs, offd, N, K)
    y_grid = mxq.grouped_gemm(aq, as_, bq, bs, offd, N, K)
    torch.cuda.synchronize()
    _, osa = oracle.quant_rows(bits(A))
    want = oracle.scale_group_tiled(osa, off)
    assert np.array_equal(u8(sg)[:want.size], want), "group-tiled scales"
    assert torch.equal(y.view(torch.int16), y_grid.view(torch.int16)), "differs from mxq_grouped_gemm"
    assert mxq.get_device_status() == 0
