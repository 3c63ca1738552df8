"""GPU parity of the GEMM whose epilogue quantizes its own output
(mxq_gemm_mxfp8out): the BF16 result rounded once, then the 1x32 E4M3
quantization of every 32-column run of each row, written from registers.

Fusing the quantization into the producing kernel keeps the BF16 tensor from
a second HBM pass (DeepSeek-V4 Ascend training write-up, "AutoFuse 收益分析").
Two bars:

* against the oracle (expected values computed on the CPU from the same BF16
  inputs): the BF16 output within the GEMM tolerance; every scale code within
  one of the oracle's (the amax may cross a power of two between the two
  sums); the dequantized payload within the GEMM tolerance plus E4M3's
  rounding bound (half an ulp: 2^-4 |y| for normals, 2^-10 * scale below);
* against the oracle's 1x32 quantizer applied to the kernel's own BF16 output
  (the quantization of a given BF16 tensor has exactly one correct byte
  string): payload and scales byte for byte, at every shape and both full
  sizes;
* against the library's own two-pass path (mxq_gemm_bf16out, then the row
  copy of mxq_quant_1x32_dual, both already pinned to the oracle): bit-exact,
  payload, scales and padding, at small and full sizes.
"""
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


def _untile(s_tiled: np.ndarray, R: int, G: int) -> np.ndarray:
    """Plain [R, G] view of MMA-tiled scale bytes.  The permutation comes from
    the oracle's own layout function applied to labelled matrices (three label
    bytes, label 0 marking padding), so no layout arithmetic is retyped here."""
    _, _, oracle = _mods()
    idx = np.arange(1, R * G + 1, dtype=np.int64).reshape(R, G)
    pos = np.zeros(s_tiled.size, np.int64)
    for sh in (0, 8, 16):
        pos |= oracle.scale_tiled(((idx >> sh) & 0xFF).astype(np.uint8)).astype(np.int64) << sh
    out = np.zeros(R * G, np.uint8)
    live = pos > 0
    out[pos[live] - 1] = s_tiled[live]
    assert np.all(s_tiled[~live] == 0), "tiled padding must be zero"
    return out.reshape(R, G)


def _operands(M, N, K, seed, mn_major=False):
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=seed)
    W = workloads.normal((N, K), 0.02, seed=seed + 1)
    xq, xs, _, _ = mxq.quant_1x32_dual(X.cuda(), col=False)
    oxq, oxs = oracle.quant_rows(bits(X))
    if mn_major:   # dgrad-style: B is the 32x32 payload of W^T [K, N] read MN-major
        Wt = W.t().contiguous()
        wq, _, ws = mxq.quant_32x32(Wt.cuda())
        owq, owsf, _ = oracle.quant_32x32(bits(Wt))
        wd = np.ascontiguousarray(oracle.dequant_rows(owq, owsf).T)
    else:
        wq, ws, _, _ = mxq.quant_1x32_dual(W.cuda(), col=False)
        owq, ows = oracle.quant_rows(bits(W))
        wd = oracle.dequant_rows(owq, ows)
    return (xq, xs, wq, ws), (oracle.dequant_rows(oxq, oxs), wd)


def _two_pass(ops, M, N, K, mn_major):
    mxq, _, _ = _mods()
    y = mxq.gemm(*ops, M, N, K, b_mn_major=mn_major)
    q, s, _, _ = mxq.quant_1x32_dual(y, col=False)
    return y, q, s


def _fused(ops, M, N, K, mn_major, want_bf16=True, fill=0xA5):
    mxq, _, _ = _mods()
    dev = ops[0].device
    y = torch.full((M, N), -7.0, dtype=torch.bfloat16, device=dev) if want_bf16 else None
    q = torch.full((M, N), fill, dtype=torch.uint8, device=dev)
    s = torch.full((mxq.scale_bytes(M, N, "tiled"),), fill, dtype=torch.uint8, device=dev)
    return mxq.gemm_mxfp8out(*ops, M, N, K, b_mn_major=mn_major, out=(y, q, s))


SHAPES = [
    (256, 512, 512, False),    # the small linear layer
    (300, 288, 416, False),    # ragged M, N not a multiple of 128, K tail of 32
    (1, 128, 32, False),       # one row, one 32-group of K
    (129, 96, 256, False),     # N of 3 groups: a partly filled scale atom
    (1000, 160, 160, False),   # second half-tile holds one group
    (300, 256, 384, True),     # MN-major B (the 32x32 dgrad operand)
    (640, 1024, 2048, False),  # several tiles each way
]


@pytest.mark.parametrize("M,N,K,mn", SHAPES)
def test_fused_against_oracle(M, N, K, mn):
    mxq, _, oracle = _mods()
    ops, (xd, wd) = _operands(M, N, K, seed=M + 3 * N + 7 * K, mn_major=mn)
    y, q, s = _fused(ops, M, N, K, mn)
    torch.cuda.synchronize()
    y_ref = oracle.gemm(xd, wd)
    assert_gemm_close(y, y_ref, f"fused bf16 {M}x{N}x{K}")
    q_ref, s_ref = oracle.quant_rows(y_ref)
    s_gpu = _untile(u8(s), M, N // 32)
    assert np.all(np.abs(s_gpu.astype(int) - s_ref.astype(int)) <= 1)
    qg = u8(q)
    assert np.all((qg & 0x7F) != 0x7F), "no NaN codes for finite outputs"
    deq = oracle.dequant_rows(qg, s_gpu)
    r = oracle.bf16_to_double(y_ref)
    rms = float(np.sqrt(np.mean(r * r)))
    step = np.repeat(np.exp2(s_gpu.astype(np.float64) - 127.0 - 10.0), 32, axis=1)
    bound = 1e-2 * np.abs(r) + 1e-3 * rms + 2.0 ** -4 * (1.01 * np.abs(r) + 1e-3 * rms) + step
    err = np.abs(deq - r)
    assert np.all(err <= bound), f"{int((err > bound).sum())} payload values outside the bound"


@pytest.mark.parametrize("M,N,K,mn", SHAPES)
def test_fused_bytes_equal_oracle_quant_of_own_output(M, N, K, mn):
    """The quantized output is integer work on the kernel's BF16 result: the
    oracle's 1x32 row quantizer applied to exactly those BF16 values must give
    the same payload and scale bytes (tiled padding zero)."""
    mxq, _, oracle = _mods()
    ops, _ = _operands(M, N, K, seed=5 * M + N + 3 * K, mn_major=mn)
    y, q, s = _fused(ops, M, N, K, mn)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_rows(bits(y))
    assert np.array_equal(u8(q), q_ref), f"fused payload {M}x{N}x{K}"
    assert np.array_equal(_untile(u8(s), M, N // 32), s_ref), f"fused scales {M}x{N}x{K}"
    assert np.array_equal(u8(s), oracle.scale_tiled(s_ref)), "tiled scale bytes incl. padding"


@pytest.mark.parametrize("M,N,K,mn", SHAPES)
def test_fused_equals_two_pass(M, N, K, mn):
    ops, _ = _operands(M, N, K, seed=11 * M + N + K, mn_major=mn)
    y2, q2, s2 = _two_pass(ops, M, N, K, mn)
    y1, q1, s1 = _fused(ops, M, N, K, mn)
    yq, q0, s0 = _fused(ops, M, N, K, mn, want_bf16=False, fill=0x5A)
    torch.cuda.synchronize()
    assert yq is None
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    for q, s in ((q1, s1), (q0, s0)):
        assert torch.equal(q, q2)
        assert torch.equal(s, s2)


def test_fused_non_finite_groups():
    """Products past the FP32 range give Inf in the accumulator: that group's
    scale is the NaN code 0xFF and its payload 0x7F | sign, as in the quantizer."""
    mxq, _, _ = _mods()
    M, N, K = 128, 256, 64
    g = torch.Generator().manual_seed(5)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = torch.randn(N, K, generator=g).to(torch.bfloat16)
    X[3, :32] = 2.0 ** 100
    W[40, :32] = 2.0 ** 100
    W[41, :32] = -(2.0 ** 100)
    xq, xs, _, _ = mxq.quant_1x32_dual(X.cuda(), col=False)
    wq, ws, _, _ = mxq.quant_1x32_dual(W.cuda(), col=False)
    ops = (xq, xs, wq, ws)
    y2, q2, s2 = _two_pass(ops, M, N, K, False)
    y1, q1, s1 = _fused(ops, M, N, K, False)
    torch.cuda.synchronize()
    assert not torch.isfinite(y2[3, 40:42].float()).any()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    s_plain = _untile(u8(s1), M, N // 32)
    assert s_plain[3, 1] == 0xFF and np.all(np.delete(s_plain[3], 1) != 0xFF)


@pytest.mark.parametrize("M,N,K", [(8192, 4096, 4096), (4096, 7168, 2048)])
def test_fused_full_size_equals_two_pass(M, N, K):
    """At the training-step sizes the fused output equals the two-pass output
    bit for bit (both computed on the device), and a sampled block of rows
    stays within the oracle tolerance."""
    mxq, workloads, oracle = _mods()
    X = workloads.normal_with_outliers((M, K), seed=M + N, device="cuda")
    W = workloads.normal((N, K), 0.02, seed=K, device="cuda")
    xq, xs, _, _ = mxq.quant_1x32_dual(X, col=False)
    wq, ws, _, _ = mxq.quant_1x32_dual(W, col=False)
    ops = (xq, xs, wq, ws)
    y2, q2, s2 = _two_pass(ops, M, N, K, False)
    y1, q1, s1 = _fused(ops, M, N, K, False)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    # every byte against the oracle's quantization of the kernel's own BF16 output
    q_ref, s_ref = oracle.quant_rows(bits(y1))
    assert np.array_equal(u8(q1), q_ref), "fused payload at full size"
    assert np.array_equal(u8(s1), oracle.scale_tiled(s_ref)), "fused tiled scales at full size"
    del q_ref
    oxq, oxs = oracle.quant_rows(bits(X[M - 64:].cpu()))
    owq, ows = oracle.quant_rows(bits(W.cpu()))
    y_ref = oracle.gemm(oracle.dequant_rows(oxq, oxs), oracle.dequant_rows(owq, ows))
    assert_gemm_close(y1[M - 64:], y_ref, "fused full-size rows")
