"""Host-side checks of the C ABI (no GPU needed): the library builds, loads
and exports every function include/mxq.h declares, and argument validation
rejects bad calls with the documented status before any CUDA work.

The RFC's interface rejects unsupported configurations with an explicit
error (MindSpeed RFC "Add MXFP8-32x32 quantization support to FSDP",
sections 3.4 and 3.5.2.1); the ABI does the same with status codes.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxq.h")


@pytest.fixture(scope="module")
def L():
    from mxfp8_microscaled_precision_gb300 import build, mxq
    build.build()
    return mxq.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_hot_path_calls():
    names = _declared_functions()
    for f in ("mxq_quant_1x32_dual", "mxq_quant_32x32", "mxq_gemm_bf16out", "mxq_grouped_gemm"):
        assert f in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_version_and_strings(L):
    assert L.mxq_abi_version() == 2
    for s in range(6):
        assert L.mxq_status_string(s)
    assert L.mxq_scale_bytes(256, 512, 0) == 256 * 16
    assert L.mxq_scale_bytes(1, 32, 1) == 128 * 4
    assert L.mxq_scale_bytes(130, 160, 1) == 256 * 8
    assert L.mxq_scale_bytes(4, 33, 0) == 0


FAKE = ctypes.c_void_p(0x10000)        # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)         # misaligned


def test_quant_argument_errors(L):
    q = L.mxq_quant_1x32_dual
    assert q(FAKE, 64, 48, 48, FAKE, FAKE, None, None, 1, None) == 2      # cols % 32
    assert q(FAKE, 48, 64, 64, None, None, FAKE, FAKE, 1, None) == 2      # rows % 32 (col copy)
    assert q(None, 64, 64, 64, FAKE, FAKE, None, None, 1, None) == 1      # null input
    assert q(FAKE, 64, 64, 64, None, None, None, None, 1, None) == 1      # no output asked
    assert q(FAKE, 64, 64, 64, FAKE, None, None, None, 1, None) == 1      # half a pair
    assert q(FAKE, 64, 64, 60, FAKE, FAKE, None, None, 1, None) == 1      # ld < cols
    assert q(ODD, 64, 64, 64, FAKE, FAKE, None, None, 1, None) == 1       # misaligned
    assert q(FAKE, 64, 64, 64, FAKE, FAKE, None, None, 7, None) == 1      # bad layout
    assert q(FAKE, -1, 64, 64, FAKE, FAKE, None, None, 1, None) == 1
    assert q(FAKE, 0, 64, 64, FAKE, FAKE, None, None, 1, None) == 0       # empty: nothing to do
    b = L.mxq_quant_32x32
    assert b(FAKE, 48, 64, 64, FAKE, FAKE, FAKE, 1, None) == 2            # n % 32
    assert b(FAKE, 64, 40, 40, FAKE, FAKE, FAKE, 1, None) == 2            # k % 32 (block size)
    assert b(None, 64, 64, 64, FAKE, FAKE, FAKE, 1, None) == 1
    bf = L.mxq_quant_32x32_fmt
    assert bf(FAKE, 64, 64, 64, FAKE, FAKE, FAKE, 1, 2, None) == 1        # bad format
    assert bf(FAKE, 64, 40, 40, FAKE, FAKE, FAKE, 1, 1, None) == 2        # k % 32 (E5M2 too)
    assert bf(FAKE, 0, 64, 64, FAKE, FAKE, FAKE, 1, 1, None) == 0         # empty


def test_gemm_argument_errors(L):
    g = L.mxq_gemm_bf16out
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 128, 48, 0, FAKE, 128, 1, None) == 2   # K % 32
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 120, 64, 0, FAKE, 120, 1, None) == 2   # N % 16
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 144, 64, 1, FAKE, 144, 1, None) == 2   # MN-major N % 128
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 128, 64, 2, FAKE, 128, 1, None) == 1   # bad flag
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 128, 64, 0, FAKE, 100, 1, None) == 1   # ldy < N
    assert g(None, FAKE, FAKE, FAKE, 64, 128, 64, 0, FAKE, 128, 1, None) == 1
    assert g(FAKE, FAKE, ODD, FAKE, 64, 128, 64, 0, FAKE, 128, 1, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, 0, 128, 64, 0, FAKE, 128, 1, None) == 0    # empty
    # the tensor cores read MMA-tiled scales only: row-major scales are refused
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 128, 64, 0, FAKE, 128, 0, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, 0, 128, 64, 0, FAKE, 128, 0, None) == 1    # even with nothing to do
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 128, 64, 0, FAKE, 128, 9, None) == 1   # unknown layout
    gg = L.mxq_grouped_gemm
    W = ctypes.c_size_t
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 64, 128, 64, FAKE, None, W(0), None) == 1     # G < 1
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 2000, 64, 128, 64, FAKE, None, W(0), None) == 2  # G too big
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 192, 64, FAKE, None, W(0), None) == 2     # N % 128
    assert gg(FAKE, FAKE, FAKE, FAKE, None, 4, 64, 128, 64, FAKE, None, W(0), None) == 1     # no offsets
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0, 128, 64, FAKE, None, W(0), None) == 0      # no rows
    need = L.mxq_grouped_gemm_workspace_size(4, 300, 128, 64)
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 300, 128, 64, FAKE, FAKE, W(need - 1), None) == 1  # too small
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 300, 128, 64, FAKE, None, W(need), None) == 1      # bytes, no pointer
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 300, 128, 64, FAKE, FAKE, W(0), None) == 1         # pointer, no bytes
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 300, 128, 64, FAKE, ODD, W(need), None) == 1       # misaligned
    assert gg(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0, 128, 64, FAKE, FAKE, W(need), None) == 0        # no rows


def test_grouped_gemm_workspace_size(L):
    """The workspace holds A's scales tiled per expert for any routing:
    (ceil(M_total/128) + G) bands of ceil(K/128) 512-byte atoms."""
    ws = L.mxq_grouped_gemm_workspace_size
    assert ws(128, 131072, 4096, 4096) == (1024 + 128) * 32 * 512
    assert ws(128, 131072, 4096, 2048) == (1024 + 128) * 16 * 512
    assert ws(3, 300, 256, 96) == (3 + 3) * 1 * 512          # K tail: the atom is padded
    assert ws(1, 0, 128, 64) == 1 * 1 * 512                   # no rows still has G bands
    assert ws(4, 300, 256, 48) == 0                           # K % 32
    assert ws(0, 300, 256, 64) == 0 and ws(2000, 300, 256, 64) == 0
    assert ws(4, -1, 256, 64) == 0 and ws(4, 300, 256, 0) == 0
    from mxfp8_microscaled_precision_gb300 import mxq
    assert mxq.grouped_gemm_workspace_size(16, 16384, 4096, 4096) == (128 + 16) * 32 * 512


def test_moe_backward_argument_errors(L):
    b = L.mxq_quant_1x32_dual_batched
    assert b(FAKE, 2, 64, 48, 48, 64 * 48, FAKE, FAKE, None, None, 1, 0, None) == 2     # cols % 32
    assert b(FAKE, 2, 64, 64, 64, 100, FAKE, FAKE, None, None, 1, 0, None) == 1         # stride < rows*ld
    assert b(FAKE, 0, 64, 64, 64, 4096, FAKE, FAKE, None, None, 1, 0, None) == 0        # empty batch
    assert b(FAKE, 2, 64, 64, 64, 4096, FAKE, FAKE, None, None, 1, 7, None) == 1        # bad format
    f = L.mxq_gemm_bf16out_fmt
    assert f(FAKE, FAKE, 2, FAKE, FAKE, 0, 64, 128, 64, 0, FAKE, 128, None) == 1       # bad format
    assert f(FAKE, FAKE, 1, FAKE, FAKE, 0, 64, 128, 48, 0, FAKE, 128, None) == 2       # K % 32
    c = L.mxq_quant_1x32_cols_grouped
    assert c(FAKE, 300, 64, 64, FAKE, 4, 384, FAKE, FAKE, 1, None) == 1   # capacity < rows + 127 G
    assert c(FAKE, 300, 64, 64, FAKE, 4, 1000, FAKE, FAKE, 1, None) == 2  # capacity % 128
    assert c(FAKE, 300, 48, 48, FAKE, 4, 1024, FAKE, FAKE, 1, None) == 2  # cols % 32
    assert c(FAKE, 300, 64, 64, None, 4, 1024, FAKE, FAKE, 1, None) == 1  # no offsets
    w = L.mxq_grouped_gemm_wgrad
    assert w(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 300, 1024, 128, 120, FAKE, 120, None) == 2   # N % 16
    assert w(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 300, 512, 128, 128, FAKE, 128, None) == 1    # capacity small
    assert w(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 300, 1024, 128, 128, FAKE, 128, None) == 1   # G < 1
    cf = L.mxq_quant_1x32_cols_grouped_fmt
    assert cf(FAKE, 300, 64, 64, FAKE, 4, 1024, FAKE, FAKE, 1, 2, None) == 1   # bad format
    assert cf(FAKE, 300, 48, 48, FAKE, 4, 1024, FAKE, FAKE, 1, 1, None) == 2   # cols % 32
    assert cf(FAKE, 0, 64, 64, FAKE, 4, 1024, FAKE, FAKE, 1, 1, None) == 0     # no rows
    gf = L.mxq_grouped_gemm_fmt
    Z = ctypes.c_size_t(0)
    assert gf(FAKE, FAKE, 5, FAKE, FAKE, 0, FAKE, 4, 64, 128, 64, FAKE, 128, None, Z, None) == 1   # bad a format
    assert gf(FAKE, FAKE, 1, FAKE, FAKE, 3, FAKE, 4, 64, 128, 64, FAKE, 128, None, Z, None) == 1   # bad b format
    assert gf(FAKE, FAKE, 1, FAKE, FAKE, 0, FAKE, 4, 64, 192, 64, FAKE, 192, None, Z, None) == 2   # N % 128
    assert gf(FAKE, FAKE, 1, FAKE, FAKE, 0, FAKE, 4, 0, 128, 64, FAKE, 128, None, Z, None) == 0    # no rows
    assert gf(FAKE, FAKE, 1, FAKE, FAKE, 0, FAKE, 4, 64, 128, 64, FAKE, 120, None, Z, None) == 1   # ldy < N
    wf = L.mxq_grouped_gemm_wgrad_fmt
    assert wf(FAKE, FAKE, 9, FAKE, FAKE, 0, FAKE, 4, 300, 1024, 128, 128, FAKE, 128, None) == 1  # bad format
    assert wf(FAKE, FAKE, 1, FAKE, FAKE, 0, FAKE, 4, 300, 1024, 128, 120, FAKE, 120, None) == 2  # N % 16


def test_group_tiled_argument_errors(L):
    r = L.mxq_scale_regroup_rows
    assert r(FAKE, 300, 256, FAKE, 4, 6, FAKE, None) == 1        # bands_cap < ceil(300/128) + 4
    assert r(FAKE, 300, 256, FAKE, 0, 7, FAKE, None) == 1        # G < 1
    assert r(FAKE, 300, 256, FAKE, 2000, 2003, FAKE, None) == 2  # G too big
    assert r(FAKE, 300, 48, FAKE, 4, 7 + 1, FAKE, None) == 2     # cols % 32
    assert r(FAKE, 300, 256, None, 4, 8, FAKE, None) == 1        # no offsets
    assert r(FAKE, 300, 256, FAKE, 4, 8, ODD, None) == 1         # misaligned output
    assert r(FAKE, 0, 256, FAKE, 4, 4, FAKE, None) == 0          # no rows
    t = L.mxq_grouped_gemm_group_tiled
    assert t(FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 4, 300, 128, 64, 6, FAKE, 128, None) == 1   # cap too small
    assert t(FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 4, 300, 192, 64, 7, FAKE, 192, None) == 2   # N % 128
    assert t(FAKE, FAKE, 7, FAKE, FAKE, 0, FAKE, 4, 300, 128, 64, 7, FAKE, 128, None) == 1   # bad format
    assert t(FAKE, FAKE, 0, FAKE, FAKE, 0, None, 4, 300, 128, 64, 7, FAKE, 128, None) == 1   # no offsets
    assert t(FAKE, FAKE, 0, FAKE, FAKE, 0, FAKE, 4, 0, 128, 64, 4, FAKE, 128, None) == 0     # no rows


def test_gemm_multi_argument_errors(L):
    from mxfp8_microscaled_precision_gb300 import mxq
    D = (mxq.GemmDesc * 2)()
    for d in D:
        d.a_q = d.a_s = d.b_q = d.b_s = d.y = 0x10000
        d.M, d.N, d.K, d.ldy, d.a_fmt, d.b_fmt = 64, 128, 64, 128, 0, 0
    f = L.mxq_gemm_bf16out_multi
    assert f(None, 0, 0, None) == 0                # nothing to do
    assert f(None, 1, 0, None) == 1                # no descriptors
    assert f(D, 5, 0, None) == 1                   # more than 4
    assert f(D, 2, 2, None) == 1                   # bad orientation flag
    D[1].K = 48
    assert f(D, 2, 0, None) == 2                   # K % 32 in the second GEMM: nothing runs
    D[1].K, D[1].a_fmt = 64, 3
    assert f(D, 2, 0, None) == 1                   # bad format
    D[1].a_fmt, D[1].N, D[1].ldy = 0, 144, 144
    assert f(D, 2, 1, None) == 2                   # MN-major needs N % 128
    D[1].N, D[1].ldy, D[0].ldy = 128, 128, 100
    assert f(D, 2, 0, None) == 1                   # ldy < N
    D[0].ldy, D[0].M, D[1].M = 128, 0, 0
    assert f(D, 2, 0, None) == 0                   # every GEMM empty


def test_fused_quant_gemm_argument_errors(L):
    g = L.mxq_gemm_mxfp8out
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 48, 64, 0, FAKE, 48, FAKE, FAKE, None) == 2    # N % 32
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 64, 0, 0, FAKE, 64, FAKE, FAKE, None) == 2     # K == 0
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 96, 64, 1, FAKE, 96, FAKE, FAKE, None) == 2    # MN-major N % 128
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 64, 64, 0, FAKE, 64, None, FAKE, None) == 1    # no payload
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 64, 64, 0, FAKE, 64, FAKE, ODD, None) == 1     # misaligned scales
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 64, 64, 0, FAKE, 60, FAKE, FAKE, None) == 1    # ldy < N
    assert g(FAKE, FAKE, FAKE, FAKE, 0, 64, 64, 0, None, 0, None, None, None) == 0      # no rows
    assert g(FAKE, FAKE, FAKE, FAKE, 64, 64, 64, 2, FAKE, 64, FAKE, FAKE, None) == 1    # bad flag


def _layout(L, recipe, n, k, world):
    off = (ctypes.c_int64 * 4)()
    size = ctypes.c_int64()
    st = L.mxq_fsdp_payload_layout(recipe, n, k, world, off, ctypes.byref(size))
    return st, list(off), size.value


@pytest.mark.parametrize("n,k,world", [(7168, 7168, 8), (1024, 320, 8), (4096, 4096, 1), (512, 96, 2)])
def test_fsdp_payload_layout(L, n, k, world):
    """One rank's all-gather payload: its shard's tensors back to back, 4 of
    them for mxfp8 and 3 for mxfp8-32x32 (the counts the RFC states), the
    32x32 payload smaller by exactly one shard payload."""
    import json
    facts = json.load(open(os.path.join(ROOT, "tests", "golden", "page_facts.json")))["allgather_tensor_count"]
    ns = n // world
    sf, sb = L.mxq_scale_bytes(ns, k, 1), L.mxq_scale_bytes(k, ns, 1)
    st, off, size = _layout(L, 0, n, k, world)
    assert st == 0 and off == [0, ns * k, ns * k + sf, 2 * ns * k + sf] and size == 2 * ns * k + sf + sb
    assert sum(o >= 0 for o in off) == facts["value"]["mxfp8"]
    st, off32, size32 = _layout(L, 1, n, k, world)
    assert st == 0 and off32 == [0, ns * k, -1, ns * k + sf] and size32 == ns * k + sf + sb
    assert sum(o >= 0 for o in off32) == facts["value"]["mxfp8-32x32"]
    assert size - size32 == ns * k
    assert all(o % 512 == 0 for o in off + off32 if o >= 0) and size % 512 == 0


def test_fsdp_argument_errors(L):
    assert _layout(L, 0, 1000, 64, 1)[0] == 2           # n % 128
    assert _layout(L, 0, 1024, 64, 16)[0] == 2          # n % (128 world)
    assert _layout(L, 0, 1024, 48, 1)[0] == 2           # k % 32
    assert _layout(L, 0, 1024, 64, 0)[0] == 2           # world < 1
    assert _layout(L, 3, 1024, 64, 1)[0] == 1           # recipe
    u = L.mxq_fsdp_unpack
    assert u(1, 1024, 64, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1    # 32x32 takes no q_bwd
    assert u(0, 1024, 64, 2, FAKE, FAKE, FAKE, None, FAKE, None) == 1    # 1x32 needs q_bwd
    assert u(0, 1024, 64, 2, ODD, FAKE, FAKE, FAKE, FAKE, None) == 1     # misaligned source
    assert u(0, 1024, 64, 3, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 2    # shard not 128-aligned


def test_binding_raises_value_error(L):
    from mxfp8_microscaled_precision_gb300 import mxq
    with pytest.raises(ValueError):
        mxq._check(2, "probe")
    with pytest.raises(ValueError):
        mxq._layout("zigzag")
