"""GPU parity of the pre-quantized weight all-gather path (MindSpeed RFC "Add
MXFP8-32x32 quantization support to FSDP", section 3.3.2): every rank
quantizes its row shard of W into its payload, the payloads are gathered
back to back, and mxq_fsdp_unpack rebuilds the full operands.

The expected bytes are the oracle's quantization of the whole of W (row and
column copies for mxfp8, payload and both scales for mxfp8-32x32), laid out
by the oracle's tiled-scale function: gathering shards must change nothing.
The all-gather itself is stood in for by device copies (one GPU).
"""
import numpy as np
import pytest
import torch

from _util import bits, gpu_or_skip, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _mods():
    from mxfp8_microscaled_precision_gb300 import mxq, workloads
    from oracle import oracle
    return mxq, workloads, oracle


def _gather(W_dev, recipe, world, fill=0xEE):
    """Each rank's payload written by its own quantizer call, then the
    payloads concatenated (the all-gather's result on every rank)."""
    mxq, _, _ = _mods()
    n, k = W_dev.shape
    ns = n // world
    _, P = mxq.fsdp_payload_layout(recipe, n, k, world)
    sends = [torch.full((P,), fill, dtype=torch.uint8, device=W_dev.device) for _ in range(world)]
    for r in range(world):
        mxq.fsdp_quant_shard(W_dev[r * ns:(r + 1) * ns], recipe, n, world, sends[r])
    gathered = torch.cat(sends)
    return gathered, P


def _unpack(recipe, gathered, n, k, world, fill=0xA5):
    mxq, _, _ = _mods()
    dev = gathered.device
    dual = recipe == "mxfp8"
    out = (torch.full((n, k), fill, dtype=torch.uint8, device=dev),
           torch.full((mxq.scale_bytes(n, k, "tiled"),), fill, dtype=torch.uint8, device=dev),
           torch.full((k, n), fill, dtype=torch.uint8, device=dev) if dual else None,
           torch.full((mxq.scale_bytes(k, n, "tiled"),), fill, dtype=torch.uint8, device=dev))
    return mxq.fsdp_unpack(recipe, gathered, n, k, world, out=out)


CASES = [(1024, 320, 8), (1024, 320, 1), (768, 512, 2), (2048, 1024, 4), (512, 96, 4)]


@pytest.mark.parametrize("recipe", ["mxfp8", "mxfp8-32x32"])
@pytest.mark.parametrize("n,k,world", CASES)
def test_gathered_shards_equal_whole_weight_quant(recipe, n, k, world):
    mxq, workloads, oracle = _mods()
    W = workloads.normal_with_outliers((n, k), seed=n + k + world)
    gathered, P = _gather(W.cuda(), recipe, world)
    q_fwd, s_fwd, q_bwd, s_bwd = _unpack(recipe, gathered, n, k, world)
    torch.cuda.synchronize()
    if recipe == "mxfp8":
        oq, os_, oqc, osc = oracle.quant_dual(bits(W))
        assert np.array_equal(u8(q_bwd), oqc)
    else:
        oq, os_, osc = oracle.quant_32x32(bits(W))
        assert q_bwd is None
    assert np.array_equal(u8(q_fwd), oq)
    assert np.array_equal(u8(s_fwd), oracle.scale_tiled(os_))
    assert np.array_equal(u8(s_bwd), oracle.scale_tiled(osc))
    assert gathered.numel() == world * P


@pytest.mark.parametrize("recipe", ["mxfp8", "mxfp8-32x32"])
def test_full_size_gather_feeds_the_gemms(recipe):
    """The 7168x7168 weight over 8 ranks: the rebuilt operands equal the
    single-call quantization byte for byte, so forward and dgrad GEMMs on them
    equal the GEMMs on the directly quantized weight; a sampled block of the
    payload is checked against the oracle."""
    mxq, workloads, oracle = _mods()
    n = k = 7168
    world = 8
    W = workloads.normal((n, k), 0.02, seed=17, device="cuda")
    gathered, P = _gather(W, recipe, world)
    q_fwd, s_fwd, q_bwd, s_bwd = _unpack(recipe, gathered, n, k, world)
    if recipe == "mxfp8":
        dq, ds, dqc, dsc = mxq.quant_1x32_dual(W)
        torch.cuda.synchronize()
        assert torch.equal(q_bwd, dqc) and torch.equal(s_bwd, dsc)
    else:
        dq, ds, dsc = mxq.quant_32x32(W)
        torch.cuda.synchronize()
        assert torch.equal(s_bwd, dsc)
    assert torch.equal(q_fwd, dq) and torch.equal(s_fwd, ds)
    # payload bytes: mxfp8-32x32 moves one weight payload fewer (RFC section 3.3.2)
    ns = n // world
    expect = ns * k * (2 if recipe == "mxfp8" else 1) + mxq.scale_bytes(ns, k) + mxq.scale_bytes(k, ns)
    assert P == expect
    rows = slice(896 * 3, 896 * 3 + 64)                    # rank 3's first rows
    wb = bits(W[rows])
    oq, _ = oracle.quant_rows(wb) if recipe == "mxfp8" else oracle.quant_32x32(wb)[:2]
    assert np.array_equal(u8(q_fwd[rows]), oq)
