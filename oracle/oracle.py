"""ctypes wrapper around the C++ oracle (``mxq_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product package.
It shares nothing with the CUDA path.  Inputs are numpy arrays; BF16 tensors
travel as their raw ``uint16`` bit patterns.

Every function states what it computes; the arithmetic itself is in the C++
file, written from the definitions of the MXFP8 format (the torchtitan-npu
low-precision tutorial, "MXFP8 与 HiF8 架构原理速览") and of the 32x32 block
variant (MindSpeed RFC "Add MXFP8-32x32 quantization support to FSDP",
sections 3.1 and 3.3.3).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxq_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (g++, OpenMP)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_decode.restype = ctypes.c_double
    lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e5m2_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e5m2_decode.restype = ctypes.c_double
    lib.orc_rceil_exponent_fmt.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.orc_rceil_exponent_fmt.restype = ctypes.c_int
    lib.orc_e5m2_encode_array.argtypes = [P, I64, P]
    lib.orc_quant_rows_fmt.argtypes = [P, I64, I64, I64, P, P, ctypes.c_int]
    lib.orc_dequant_rows_fmt.argtypes = [P, P, I64, I64, P, ctypes.c_int]
    lib.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e8m0_decode.restype = ctypes.c_double
    lib.orc_rceil_exponent.argtypes = [ctypes.c_double]
    lib.orc_rceil_exponent.restype = ctypes.c_int
    lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
    lib.orc_bf16_from_double.restype = ctypes.c_uint16
    lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_double.restype = ctypes.c_double
    lib.orc_e4m3_encode_array.argtypes = [P, I64, P]
    lib.orc_bf16_from_double_array.argtypes = [P, I64, P]
    lib.orc_quant_rows.argtypes = [P, I64, I64, I64, P, P]
    lib.orc_quant_dual.argtypes = [P, I64, I64, I64, P, P, P, P]
    lib.orc_quant_32x32.argtypes = [P, I64, I64, I64, P, P, P]
    lib.orc_quant_32x32_fmt.argtypes = [P, I64, I64, I64, P, P, P, ctypes.c_int]
    lib.orc_scale_tiled.argtypes = [P, I64, I64, P]
    lib.orc_quant_cols_grouped.argtypes = [P, I64, I64, I64, P, ctypes.c_int32, I64, P, P]
    lib.orc_quant_cols_grouped_fmt.argtypes = [P, I64, I64, I64, P, ctypes.c_int32, I64, P, P, ctypes.c_int]
    lib.orc_dequant_rows.argtypes = [P, P, I64, I64, P]
    lib.orc_gemm.argtypes = [P, P, I64, I64, I64, P, I64, P]
    lib.orc_grouped_gemm.argtypes = [P, P, P, ctypes.c_int32, I64, I64, P, I64, P]
    for f in ("orc_e4m3_encode_array", "orc_bf16_from_double_array", "orc_quant_rows",
              "orc_quant_cols_grouped", "orc_quant_cols_grouped_fmt", "orc_e5m2_encode_array", "orc_quant_rows_fmt",
              "orc_dequant_rows_fmt",
              "orc_quant_dual", "orc_quant_32x32", "orc_quant_32x32_fmt", "orc_scale_tiled", "orc_dequant_rows",
              "orc_gemm", "orc_grouped_gemm"):
        getattr(lib, f).restype = None
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalars --------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Value of each float8_e4m3fn code (NaN for 0x7F and 0xFF)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c]).reshape(np.shape(codes))


def e4m3_encode(values) -> np.ndarray:
    """Round-to-nearest-even, saturating float8_e4m3fn code of each double."""
    lib = _load()
    v = _c(values, np.float64).ravel()
    out = np.empty(v.shape, np.uint8)
    lib.orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out.reshape(np.shape(values))


def e5m2_decode(codes) -> np.ndarray:
    """Value of each float8_e5m2 code (Inf for 0x7C/0xFC, NaN for the other E=31 codes)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.orc_e5m2_decode(int(v)) for v in c]).reshape(np.shape(codes))


def e5m2_encode(values) -> np.ndarray:
    """Round-to-nearest-even, saturating float8_e5m2 code of each double."""
    lib = _load()
    v = _c(values, np.float64).ravel()
    out = np.empty(v.shape, np.uint8)
    lib.orc_e5m2_encode_array(_ptr(v), v.size, _ptr(out))
    return out.reshape(np.shape(values))


def rceil_exponent_fmt(amax: float, fmt: int) -> int:
    """ceil(log2(amax / max_fmt)), max 448 (fmt 0, E4M3) or 57344 (fmt 1, E5M2)."""
    return _load().orc_rceil_exponent_fmt(float(amax), int(fmt))


def e8m0_decode(code: int) -> float:
    return _load().orc_e8m0_decode(int(code))


def rceil_exponent(amax: float) -> int:
    """ceil(log2(amax/448)) clamped to [-127, 127]; -127 for amax == 0."""
    return _load().orc_rceil_exponent(float(amax))


def bf16_from_double(values) -> np.ndarray:
    """BF16 bit pattern nearest to each double (ties to even), one rounding."""
    lib = _load()
    v = _c(values, np.float64).ravel()
    out = np.empty(v.shape, np.uint16)
    lib.orc_bf16_from_double_array(_ptr(v), v.size, _ptr(out))
    return out.reshape(np.shape(values))


def bf16_to_double(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ---- quantizers -------------------------------------------------------------------

def quant_rows(x_bits: np.ndarray):
    """1x32 quantization along the last axis.  x_bits: uint16 [R, C], C % 32 == 0.
    Returns (q uint8 [R, C], s uint8 [R, C/32]) with plain row-major scales."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    lib.orc_quant_rows(_ptr(x), R, C, C, _ptr(q), _ptr(s))
    return q, s


def quant_rows_fmt(x_bits: np.ndarray, fmt: int):
    """quant_rows with the payload format fmt (0 E4M3, 1 E5M2)."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // 32), np.uint8)
    lib.orc_quant_rows_fmt(_ptr(x), R, C, C, _ptr(q), _ptr(s), int(fmt))
    return q, s


def dequant_rows_fmt(q: np.ndarray, s: np.ndarray, fmt: int) -> np.ndarray:
    lib = _load()
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    R, C = q.shape
    out = np.empty((R, C), np.float64)
    lib.orc_dequant_rows_fmt(_ptr(q), _ptr(s), R, C, _ptr(out), int(fmt))
    return out


def quant_dual(x_bits: np.ndarray, want_row: bool = True, want_col: bool = True):
    """Dual-axis 1x32 quantization.  Returns (q_row [R,C], s_row [R,C/32],
    q_col [C,R], s_col [C,R/32]); a pair not asked for is None."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    assert C % 32 == 0 and (not want_col or R % 32 == 0)
    q_row = np.empty((R, C), np.uint8) if want_row else None
    s_row = np.empty((R, C // 32), np.uint8) if want_row else None
    q_col = np.empty((C, R), np.uint8) if want_col else None
    s_col = np.empty((C, R // 32), np.uint8) if want_col else None
    lib.orc_quant_dual(_ptr(x), R, C, C, _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col))
    return q_row, s_row, q_col, s_col


def quant_32x32(w_bits: np.ndarray, fmt: int = 0):
    """32x32 block quantization with payload format fmt (0 E4M3, 1 E5M2: the
    RFC's dst_type, section 3.5.2.3).  Returns (q [N,K], s_fwd [N,K/32],
    s_bwd [K,N/32])."""
    lib = _load()
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    assert N % 32 == 0 and K % 32 == 0
    q = np.empty((N, K), np.uint8)
    s_fwd = np.empty((N, K // 32), np.uint8)
    s_bwd = np.empty((K, N // 32), np.uint8)
    lib.orc_quant_32x32_fmt(_ptr(w), N, K, K, _ptr(q), _ptr(s_fwd), _ptr(s_bwd), int(fmt))
    return q, s_fwd, s_bwd


def padded_slots(offsets: np.ndarray):
    """(P, L): each expert's 128-aligned token slot start and length."""
    m = np.diff(np.asarray(offsets, dtype=np.int64))
    L = (m + 127) // 128 * 128
    P = np.concatenate([[0], np.cumsum(L)[:-1]]).astype(np.int64)
    return P, L


def quant_cols_grouped(x_bits: np.ndarray, offsets: np.ndarray, capacity: int, fmt: int = 0):
    """Column (token-axis) quantization per expert with zero padding.
    x_bits uint16 [M_total, C] (rows sorted by expert), offsets int64 [G+1];
    fmt 0 = E4M3, 1 = E5M2 payload.
    Returns (q_col [C, capacity], s_col [C, capacity/32]) -- plain scales;
    columns past the last expert's slot are returned as 0 / code 0."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    off = _c(offsets, np.int64)
    G = off.size - 1
    assert capacity % 128 == 0 and off[0] == 0 and off[-1] == R
    P, L = padded_slots(off)
    assert int((P[-1] + L[-1]) if G else 0) <= capacity
    q = np.zeros((C, capacity), np.uint8)
    s = np.zeros((C, capacity // 32), np.uint8)
    lib.orc_quant_cols_grouped_fmt(_ptr(x), R, C, C, _ptr(off), G, capacity, _ptr(q), _ptr(s), int(fmt))
    return q, s


def scale_tiled(s: np.ndarray) -> np.ndarray:
    """Plain [rows, groups] scales -> the MMA-tiled byte layout (flat uint8,
    roundup(rows,128) * roundup(groups,4) bytes, zero padding)."""
    lib = _load()
    s = _c(s, np.uint8)
    rows, groups = s.shape
    n = ((rows + 127) // 128 * 128) * ((groups + 3) // 4 * 4)
    out = np.empty(n, np.uint8)
    lib.orc_scale_tiled(_ptr(s), rows, groups, _ptr(out))
    return out


def scale_group_tiled(s: np.ndarray, offsets) -> np.ndarray:
    """Group-tiled layout of plain [rows, groups] scales: the rows
    [offsets[g], offsets[g+1]) of each group laid out on their own by
    scale_tiled (rows padded to 128 with zeros), the groups' layouts one after
    the other in group order (empty groups contribute nothing).  Returns the
    written bytes: sum over groups of ceil(n_g/128) * ceil(groups/4) * 512.
    Not a layout of the pages: it lets a grouped GEMM's row tiles start at
    every group's first row."""
    s = _c(s, np.uint8)
    parts = [scale_tiled(s[int(lo):int(hi)]) for lo, hi in zip(offsets[:-1], offsets[1:]) if hi > lo]
    return np.concatenate(parts) if parts else np.zeros(0, np.uint8)


def dequant_rows(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """q[r,c] * 2^(s[r,c/32]-127) as float64 [R, C].  With s = s_fwd this is
    also the dequantized 32x32 payload (s_fwd repeats the tile exponent)."""
    lib = _load()
    q = _c(q, np.uint8)
    s = _c(s, np.uint8)
    R, C = q.shape
    assert s.shape == (R, C // 32)
    out = np.empty((R, C), np.float64)
    lib.orc_dequant_rows(_ptr(q), _ptr(s), R, C, _ptr(out))
    return out


# ---- GEMMs ------------------------------------------------------------------------

def gemm(a: np.ndarray, b: np.ndarray, rows=None) -> np.ndarray:
    """y = bf16(a @ b.T) with a [M,K], b [N,K] float64 (dequantized operands),
    each dot product summed in FP64 in increasing k.  rows: optional sample of
    row indices of a; returns uint16 bf16 bits [len(rows) or M, N]."""
    lib = _load()
    a = _c(a, np.float64)
    b = _c(b, np.float64)
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    r = None if rows is None else _c(rows, np.int64)
    nr = M if r is None else r.size
    if r is not None:
        assert r.size == 0 or (r.min() >= 0 and r.max() < M)
    y = np.empty((nr, N), np.uint16)
    lib.orc_gemm(_ptr(a), _ptr(b), M, N, K, _ptr(r), nr, _ptr(y))
    return y


def grouped_gemm(a: np.ndarray, b: np.ndarray, offsets: np.ndarray, rows=None) -> np.ndarray:
    """Per-expert y[r] = bf16(a[r] @ b[g].T) for off[g] <= r < off[g+1].
    a [M_total, K], b [G, N, K] float64; offsets int64 [G+1]."""
    lib = _load()
    a = _c(a, np.float64)
    b = _c(b, np.float64)
    off = _c(offsets, np.int64)
    G, N, K = b.shape
    M = a.shape[0]
    assert off.size == G + 1 and off[0] == 0 and off[-1] == M and np.all(np.diff(off) >= 0)
    r = None if rows is None else _c(rows, np.int64)
    nr = M if r is None else r.size
    if r is not None:
        assert r.size == 0 or (r.min() >= 0 and r.max() < M)
    y = np.empty((nr, N), np.uint16)
    lib.orc_grouped_gemm(_ptr(a), _ptr(b), _ptr(off), G, N, K, _ptr(r), nr, _ptr(y))
    return y
