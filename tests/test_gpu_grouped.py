"""GPU parity of the grouped (MoE expert) block-scaled GEMM against the
oracle: variable group sizes including empty experts, groups that start and
end inside a 128-row tile, and the full 128-expert workload on sampled rows.

The MoE expert layers run the quantized grouped matmul (torchtitan-npu
tutorial, "MoE 专家层 (Grouped MM)"; MindSpeed RFC section 2.2, gate_up_proj
and down_proj).
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


def _run_case(sizes, N, K, seed):
    mxq, workloads, oracle = _mods()
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    A = workloads.normal_with_outliers((max(M, 1), K), seed=seed)[:M]
    B = workloads.normal((G * N, K), 0.02, seed=seed + 1)
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    y = mxq.grouped_gemm(aq, as_, bq, bs, torch.from_numpy(off).cuda(), N, K)
    torch.cuda.synchronize()
    oa, osa = oracle.quant_rows(bits(A))
    ob, osb = oracle.quant_rows(bits(B))
    ref = oracle.grouped_gemm(oracle.dequant_rows(oa, osa),
                              oracle.dequant_rows(ob, osb).reshape(G, N, K), off)
    assert_gemm_close(y, ref, f"grouped sizes={list(sizes)}")


@pytest.mark.parametrize("sizes,N,K", [
    ([0, 5, 0, 300, 1, 130], 256, 192),          # empty experts, unaligned starts
    ([0, 1, 127, 129, 0, 256, 3], 128, 256),      # sizes around the 128-row tile
    ([0, 0, 0, 500, 0], 384, 128),                # all empty but one
    ([1000], 256, 512),                           # one expert
    ([64] * 16, 128, 96),                         # many small experts, K tail
    ([37, 91, 200, 5, 0, 143, 300, 1], 512, 1024),
])
def test_grouped_matches_oracle(sizes, N, K):
    _run_case(sizes, N, K, seed=sum(sizes) + N + K)


def test_grouped_single_row_groups():
    _run_case([1] * 40, 128, 64, seed=5)


def test_grouped_all_rows_written_once():
    """Rows of every expert are written; nothing outside [0, M_total) is."""
    mxq, workloads, _ = _mods()
    sizes = [3, 0, 130, 0, 125]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M, N, K = int(off[-1]), 128, 64
    A = workloads.normal((M, K), 1.0, seed=9)
    B = workloads.normal((len(sizes) * N, K), 0.5, seed=10)
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    big = torch.full((M + 2, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = big[1:M + 1]
    mxq.grouped_gemm(aq, as_, bq, bs, torch.from_numpy(off).cuda(), N, K, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    assert torch.isnan(big[0]).all() and torch.isnan(big[M + 1]).all()


def test_full_moe_gate_up_and_down_sampled():
    """128 experts, 131072 routed rows, Zipf(1.1) loads with empty experts:
    gate_up (N 4096, K 4096) and down (N 4096, K 2048) on sampled rows of
    selected experts."""
    mxq, workloads, oracle = _mods()
    d = workloads.moe_grouped(weights=False)
    off = d["routing"].offsets.numpy()
    sizes = np.diff(off)
    G = sizes.size
    assert (sizes == 0).sum() >= 4 and off[-1] == 131072
    offd = torch.from_numpy(off).cuda()
    nz = np.flatnonzero(sizes)
    rng = np.random.default_rng(7)
    unaligned = [g for g in nz if off[g] % 128 != 0][:2]
    experts = sorted(set([int(nz[np.argmax(sizes[nz])]), int(nz[np.argmin(sizes[nz])])] +
                         [int(g) for g in unaligned] + [int(g) for g in rng.choice(nz, 3, replace=False)]))
    for name, a_cpu, K, wseed in (("gate_up", d["A"], 4096, workloads.seed_for("moe_grouped", "W")),
                                  ("down", d["H"], 2048, workloads.seed_for("moe_grouped", "W_down"))):
        N = 4096
        W = workloads.normal((G * N, K), 0.02, seed=wseed, device="cuda")   # expert weights on the GPU
        aq, as_, _, _ = mxq.quant_1x32_dual(a_cpu.cuda(), col=False)
        bq, bs, _, _ = mxq.quant_1x32_dual(W, col=False)
        y = mxq.grouped_gemm(aq, as_, bq, bs, offd, N, K)
        torch.cuda.synchronize()
        for g in experts:
            lo, hi = int(off[g]), int(off[g + 1])
            rows = np.unique(np.concatenate([[lo, hi - 1], rng.integers(lo, hi, size=min(24, hi - lo))]))
            oa, osa = oracle.quant_rows(bits(a_cpu[torch.from_numpy(rows)]))
            ob, osb = oracle.quant_rows(bits(W[g * N:(g + 1) * N]))
            ref = oracle.gemm(oracle.dequant_rows(oa, osa), oracle.dequant_rows(ob, osb))
            assert_gemm_close(y[torch.from_numpy(rows).cuda()], ref, f"{name} expert {g}")
        del W, bq, bs, y


# ---- the workspace of mxq_grouped_gemm (A scales tiled per expert) -------------------

def _c_grouped(mxq, aq, as_, bq, bs, offd, G, M, N, K, y, ws):
    import ctypes
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    nbytes = 0 if ws is None else ws.numel()
    return mxq.lib().mxq_grouped_gemm(p(aq), p(as_), p(bq), p(bs), p(offd), G, M, N, K, p(y), p(ws),
                                      ctypes.c_size_t(nbytes), mxq._stream())


@pytest.mark.parametrize("sizes,N,K", [
    ([0, 5, 0, 300, 1, 130], 256, 192),
    ([0, 1, 127, 129, 0, 256, 3], 128, 256),
    ([37, 91, 200, 5, 0, 143, 300, 1], 512, 1024),
    ([1] * 40, 128, 64),
])
def test_c_abi_grouped_workspace(sizes, N, K):
    """mxq_grouped_gemm through the C ABI with and without its workspace: the
    workspace (prefilled with garbage) changes only the tile schedule, so both
    outputs are bit-identical and within the GEMM tolerance of the oracle."""
    mxq, workloads, oracle = _mods()
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    A = workloads.normal_with_outliers((M, K), seed=M + 3)
    B = workloads.normal((G * N, K), 0.02, seed=G + 4)
    aq, as_, _, _ = mxq.quant_1x32_dual(A.cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B.cuda(), col=False)
    offd = torch.from_numpy(off).cuda()
    need = mxq.grouped_gemm_workspace_size(G, M, N, K)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    y0 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y1 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _c_grouped(mxq, aq, as_, bq, bs, offd, G, M, N, K, y0, None) == 0
    assert _c_grouped(mxq, aq, as_, bq, bs, offd, G, M, N, K, y1, ws) == 0
    assert _c_grouped(mxq, aq, as_, bq, bs, offd, G, M, N, K, y1, ws[:need - 16]) == 1   # too small
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    oa, osa = oracle.quant_rows(bits(A))
    ob, osb = oracle.quant_rows(bits(B))
    ref = oracle.grouped_gemm(oracle.dequant_rows(oa, osa), oracle.dequant_rows(ob, osb).reshape(G, N, K), off)
    assert_gemm_close(y1, ref, f"grouped with workspace sizes={sizes}")
    # the workspace now holds A's scales tiled per expert (oracle layout, written bands only)
    want = oracle.scale_group_tiled(osa, off)
    assert np.array_equal(ws.cpu().numpy()[:want.size], want)


def test_full_moe_with_workspace_bit_identical():
    """The 128-expert routing (131072 rows): gate_up with the workspace equals
    the call without it bit for bit."""
    mxq, workloads, _ = _mods()
    d = workloads.moe_grouped(weights=False)
    off = d["routing"].offsets.numpy()
    G, N, K = off.size - 1, 4096, 4096
    offd = torch.from_numpy(off).cuda()
    W = workloads.normal((G * N, K), 0.02, seed=workloads.seed_for("moe_grouped", "W"), device="cuda")
    aq, as_, _, _ = mxq.quant_1x32_dual(d["A"].cuda(), col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(W, col=False)
    del W
    y0 = mxq.grouped_gemm(aq, as_, bq, bs, offd, N, K)
    y1 = mxq.grouped_gemm(aq, as_, bq, bs, offd, N, K, workspace="alloc")
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
