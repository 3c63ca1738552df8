"""Python binding of libmxq (the C ABI in include/mxq.h).

Argument marshalling only: tensors are allocated by PyTorch on the current
CUDA device, their pointers and sizes go through ctypes to the C ABI, and
every step of the computation runs in the library's CUDA kernels on the
current stream.  There is no fallback: if the library is missing or the
device is not a GB300 the calls raise.

Names follow the pages: ``quant_1x32_dual`` returns the forward and
backward copies (q_row, s_row, q_col, s_col) of the mxfp8 recipe,
``quant_32x32`` the single payload and two scale tensors (q, s_fwd, s_bwd)
of the mxfp8-32x32 recipe (MindSpeed RFC "Add MXFP8-32x32 quantization
support to FSDP", sections 3.3.2-3.3.3), ``gemm`` / ``grouped_gemm`` the
block-scaled FP8 matmuls with BF16 output.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

ROWMAJOR, TILED = 0, 1
E4M3, E5M2 = 0, 1
_FORMATS = {"e4m3": E4M3, "e5m2": E5M2, E4M3: E4M3, E5M2: E5M2}
_LAYOUTS = {"rowmajor": ROWMAJOR, "tiled": TILED, ROWMAJOR: ROWMAJOR, TILED: TILED}
STATUS = {0: "MXQ_OK", 1: "MXQ_ERR_INVALID_ARG", 2: "MXQ_ERR_UNSUPPORTED_SHAPE",
          3: "MXQ_ERR_UNSUPPORTED_DEVICE", 4: "MXQ_ERR_CUDA", 5: "MXQ_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class MXQError(ValueError):
    """A non-OK status from the C ABI."""

    def __init__(self, what: str, status: int, text: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({text})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded C library with argument types declared.  Raises if it has
    not been built (run ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libmxq.so is not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        P, I64, I32, U32, SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                ctypes.c_uint32, ctypes.c_size_t)
        S = ctypes.c_int
        L.mxq_abi_version.argtypes, L.mxq_abi_version.restype = [], ctypes.c_int
        L.mxq_status_string.argtypes, L.mxq_status_string.restype = [S], ctypes.c_char_p
        L.mxq_scale_bytes.argtypes, L.mxq_scale_bytes.restype = [I64, I64, S], SZ
        L.mxq_quant_1x32_dual.argtypes = [P, I64, I64, I64, P, P, P, P, S, P]
        L.mxq_quant_1x32_dual_batched.argtypes = [P, I64, I64, I64, I64, I64, P, P, P, P, S, S, P]
        L.mxq_gemm_bf16out_fmt.argtypes = [P, P, S, P, P, S, I64, I64, I64, S, P, I64, P]
        L.mxq_gemm_bf16out_multi.argtypes = [ctypes.POINTER(GemmDesc), I32, S, P]
        L.mxq_quant_1x32_cols_grouped.argtypes = [P, I64, I64, I64, P, I32, I64, P, P, S, P]
        L.mxq_quant_1x32_cols_grouped_fmt.argtypes = [P, I64, I64, I64, P, I32, I64, P, P, S, S, P]
        L.mxq_grouped_gemm_fmt.argtypes = [P, P, S, P, P, S, P, I32, I64, I64, I64, P, I64, P, SZ, P]
        L.mxq_grouped_gemm_workspace_size.argtypes = [I32, I64, I64, I64]
        L.mxq_grouped_gemm_workspace_size.restype = SZ
        L.mxq_grouped_gemm_group_tiled.argtypes = [P, P, S, P, P, S, P, I32, I64, I64, I64, I64, P, I64, P]
        L.mxq_scale_regroup_rows.argtypes = [P, I64, I64, P, I32, I64, P, P]
        L.mxq_grouped_gemm_wgrad_fmt.argtypes = [P, P, S, P, P, S, P, I32, I64, I64, I64, I64, P, I64, P]
        L.mxq_grouped_gemm_wgrad.argtypes = [P, P, P, P, P, I32, I64, I64, I64, I64, P, I64, P]
        L.mxq_quant_32x32.argtypes = [P, I64, I64, I64, P, P, P, S, P]
        L.mxq_quant_32x32_fmt.argtypes = [P, I64, I64, I64, P, P, P, S, S, P]
        L.mxq_gemm_bf16out.argtypes = [P, P, P, P, I64, I64, I64, S, P, I64, S, P]
        L.mxq_grouped_gemm.argtypes = [P, P, P, P, P, I32, I64, I64, I64, P, P, SZ, P]
        L.mxq_gemm_mxfp8out.argtypes = [P, P, P, P, I64, I64, I64, S, P, I64, P, P, P]
        L.mxq_fsdp_payload_layout.argtypes = [S, I64, I64, I32, ctypes.POINTER(I64), ctypes.POINTER(I64)]
        L.mxq_fsdp_unpack.argtypes = [S, I64, I64, I32, P, P, P, P, P, P]
        L.mxq_get_device_status.argtypes = [P]
        L.mxq_grouped_gemm_noalloc.argtypes = [P, P, P, P, P, I32, I64, I64, I64, P, P]
        L.mxq_grouped_gemm_noalloc.restype = S
        L.mxq_debug_wait_timeout.argtypes = [U32, P]
        for f in ("mxq_quant_1x32_dual", "mxq_quant_32x32", "mxq_gemm_bf16out",
                  "mxq_grouped_gemm", "mxq_get_device_status", "mxq_debug_wait_timeout",
                  "mxq_quant_1x32_dual_batched", "mxq_quant_1x32_cols_grouped",
                  "mxq_grouped_gemm_wgrad", "mxq_gemm_bf16out_fmt", "mxq_gemm_mxfp8out",
                  "mxq_fsdp_payload_layout", "mxq_fsdp_unpack", "mxq_quant_1x32_cols_grouped_fmt",
                  "mxq_grouped_gemm_fmt", "mxq_grouped_gemm_wgrad_fmt", "mxq_gemm_bf16out_multi",
                  "mxq_grouped_gemm_group_tiled", "mxq_scale_regroup_rows", "mxq_quant_32x32_fmt"):
            getattr(L, f).restype = S
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().mxq_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise MXQError(what, status, status_string(status))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _layout(layout) -> int:
    if layout not in _LAYOUTS:
        raise ValueError(f"unknown scale layout {layout!r}")
    return _LAYOUTS[layout]


def scale_bytes(rows: int, cols: int, layout="tiled") -> int:
    return int(lib().mxq_scale_bytes(rows, cols, _layout(layout)))


def _scale_tensor(rows, cols, layout, device):
    n = scale_bytes(rows, cols, layout)
    if _layout(layout) == ROWMAJOR:
        return torch.empty((rows, cols // 32), dtype=torch.uint8, device=device)
    return torch.empty(n, dtype=torch.uint8, device=device)


def quant_1x32_dual(x: torch.Tensor, row: bool = True, col: bool = True, layout="tiled",
                    out=None):
    """1x32 quantization of a 2-D bf16 CUDA tensor along both axes.
    Returns (q_row [R,C], s_row, q_col [C,R], s_col); pairs not asked for are
    None.  `out` may supply the four output tensors (None where not asked for)."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda:
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor")
    if x.stride(1) != 1:
        raise ValueError("x must have unit stride along its last axis")
    R, C = x.shape
    dev = x.device
    if out is not None:
        q_row, s_row, q_col, s_col = out
    else:
        q_row = torch.empty((R, C), dtype=torch.uint8, device=dev) if row else None
        s_row = _scale_tensor(R, C, layout, dev) if row else None
        q_col = torch.empty((C, R), dtype=torch.uint8, device=dev) if col else None
        s_col = _scale_tensor(C, R, layout, dev) if col else None
    _check(lib().mxq_quant_1x32_dual(_ptr(x), R, C, x.stride(0), _ptr(q_row), _ptr(s_row),
                                     _ptr(q_col), _ptr(s_col), _layout(layout), _stream()),
           "mxq_quant_1x32_dual")
    return q_row, s_row, q_col, s_col


def _fmt(fmt) -> int:
    if fmt not in _FORMATS:
        raise ValueError(f"unknown FP8 format {fmt!r} (e4m3 or e5m2)")
    return _FORMATS[fmt]


def quant_1x32_dual_batched(x: torch.Tensor, row: bool = True, col: bool = True, layout="tiled",
                            fmt="e4m3", out=None):
    """1x32 quantization of every matrix of a 3-D bf16 CUDA tensor [B, R, C]
    (e.g. stacked expert weights; B = 1 for a single matrix) with payload
    format fmt ("e4m3" or "e5m2").  Returns (q_row [B,R,C], s_row [B, bytes],
    q_col [B,C,R], s_col [B, bytes]); pairs not asked for are None.  `out`
    may supply the four output tensors (contiguous per matrix; None where not
    asked for)."""
    if x.dim() == 2:
        x = x.unsqueeze(0)
    if x.dtype != torch.bfloat16 or x.dim() != 3 or not x.is_cuda or x.stride(2) != 1:
        raise ValueError("x must be a 3-D bfloat16 CUDA tensor with unit last stride")
    B, R, C = x.shape
    dev = x.device
    u8 = dict(dtype=torch.uint8, device=dev)
    if out is not None:
        q_row, s_row, q_col, s_col = out
    else:
        q_row = torch.empty((B, R, C), **u8) if row else None
        s_row = torch.empty((B, scale_bytes(R, C, layout)), **u8) if row else None
        q_col = torch.empty((B, C, R), **u8) if col else None
        s_col = torch.empty((B, scale_bytes(C, R, layout)), **u8) if col else None
    _check(lib().mxq_quant_1x32_dual_batched(_ptr(x), B, R, C, x.stride(1), x.stride(0), _ptr(q_row),
                                             _ptr(s_row), _ptr(q_col), _ptr(s_col), _layout(layout),
                                             _fmt(fmt), _stream()), "mxq_quant_1x32_dual_batched")
    return q_row, s_row, q_col, s_col


def grouped_capacity(M_total: int, G: int) -> int:
    """Token-slot capacity that fits any offsets: M_total + 127 G, rounded up to 128."""
    return (M_total + 127 * G + 127) // 128 * 128


def quant_cols_grouped(x: torch.Tensor, offsets: torch.Tensor, capacity: int = None, layout="tiled", fmt="e4m3"):
    """Token-axis quantization inside each expert (see mxq_quant_1x32_cols_grouped).
    x: bf16 [M_total, C] sorted by expert; offsets: int64 CUDA [G+1].
    Returns (q_col [C, capacity], s_col); the columns past the last expert's slot,
    which the kernel does not write, are zero."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor with unit last stride")
    if offsets.dtype != torch.int64 or not offsets.is_cuda:
        raise ValueError("offsets must be an int64 CUDA tensor")
    R, C = x.shape
    G = offsets.numel() - 1
    if capacity is None:
        capacity = grouped_capacity(R, G)
    q_col = torch.zeros((C, capacity), dtype=torch.uint8, device=x.device)
    s_col = _scale_tensor(C, capacity, layout, x.device).zero_()
    _check(lib().mxq_quant_1x32_cols_grouped_fmt(_ptr(x), R, C, x.stride(0), _ptr(offsets), G, capacity,
                                                 _ptr(q_col), _ptr(s_col), _layout(layout), _fmt(fmt), _stream()),
           "mxq_quant_1x32_cols_grouped_fmt")
    return q_col, s_col


def grouped_gemm_wgrad(a_q, a_s, b_q, b_s, offsets: torch.Tensor, M_total: int, out=None, a_fmt="e4m3",
                       b_fmt="e4m3"):
    """Per-expert y[g] = A_g B_g^T over each expert's token slot (see
    mxq_grouped_gemm_wgrad).  a_q [M, capacity], b_q [N, capacity] from
    quant_cols_grouped.  Returns y bf16 [G, M, N]."""
    M, capacity = a_q.shape
    N = b_q.shape[0]
    G = offsets.numel() - 1
    if out is None:
        out = torch.empty((G, M, N), dtype=torch.bfloat16, device=a_q.device)
    _check(lib().mxq_grouped_gemm_wgrad_fmt(_ptr(a_q), _ptr(a_s), _fmt(a_fmt), _ptr(b_q), _ptr(b_s), _fmt(b_fmt),
                                            _ptr(offsets), G, M_total, capacity, M, N, _ptr(out), out.stride(-2),
                                            _stream()), "mxq_grouped_gemm_wgrad_fmt")
    return out


def quant_32x32(w: torch.Tensor, layout="tiled", out=None, fmt="e4m3"):
    """32x32 block quantization of a bf16 weight [n, k] with payload format fmt
    ("e4m3" or "e5m2").  Returns (q [n,k], s_fwd ([n,k/32] scales), s_bwd
    ([k,n/32] scales)); `out` may supply the three output tensors."""
    if w.dtype != torch.bfloat16 or w.dim() != 2 or not w.is_cuda or w.stride(1) != 1:
        raise ValueError("w must be a 2-D bfloat16 CUDA tensor with unit last stride")
    n, k = w.shape
    dev = w.device
    if out is not None:
        q, s_fwd, s_bwd = out
    else:
        q = torch.empty((n, k), dtype=torch.uint8, device=dev)
        s_fwd = _scale_tensor(n, k, layout, dev)
        s_bwd = _scale_tensor(k, n, layout, dev)
    _check(lib().mxq_quant_32x32_fmt(_ptr(w), n, k, w.stride(0), _ptr(q), _ptr(s_fwd), _ptr(s_bwd),
                                     _layout(layout), _fmt(fmt), _stream()), "mxq_quant_32x32_fmt")
    return q, s_fwd, s_bwd


def gemm(a_q, a_s, b_q, b_s, M: int, N: int, K: int, b_mn_major: bool = False, out=None):
    """y [M, N] bf16 = deq(A) deq(B)^T with tiled scales (see mxq_gemm_bf16out)."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    _check(lib().mxq_gemm_bf16out(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), M, N, K,
                                  1 if b_mn_major else 0, _ptr(out), out.stride(0), TILED, _stream()),
           "mxq_gemm_bf16out")
    return out


def gemm_fmt(a_q, a_s, a_fmt, b_q, b_s, b_fmt, M: int, N: int, K: int, b_mn_major: bool = False, out=None):
    """gemm with per-operand payload formats ("e4m3" / "e5m2")."""
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    _check(lib().mxq_gemm_bf16out_fmt(_ptr(a_q), _ptr(a_s), _fmt(a_fmt), _ptr(b_q), _ptr(b_s), _fmt(b_fmt),
                                      M, N, K, 1 if b_mn_major else 0, _ptr(out), out.stride(0), _stream()),
           "mxq_gemm_bf16out_fmt")
    return out


class GemmDesc(ctypes.Structure):
    """mxq_gemm_desc of include/mxq.h."""
    _fields_ = [("a_q", ctypes.c_void_p), ("a_s", ctypes.c_void_p), ("b_q", ctypes.c_void_p),
                ("b_s", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("y", ctypes.c_void_p), ("ldy", ctypes.c_int64), ("a_fmt", ctypes.c_int), ("b_fmt", ctypes.c_int)]


def gemm_multi(gemms, b_mn_major: bool = False):
    """Several independent GEMMs in one launch (see mxq_gemm_bf16out_multi).
    gemms: list of dicts with a_q, a_s, b_q, b_s, M, N, K and optionally out,
    a_fmt, b_fmt ("e4m3" default).  Returns the list of outputs y [M, N] bf16."""
    if not 1 <= len(gemms) <= 4:
        raise ValueError("gemm_multi takes 1 to 4 GEMMs")
    descs = (GemmDesc * len(gemms))()
    outs = []
    for d, g in zip(descs, gemms):
        M, N, K = g["M"], g["N"], g["K"]
        out = g.get("out")
        if out is None:
            out = torch.empty((M, N), dtype=torch.bfloat16, device=g["a_q"].device)
        outs.append(out)
        addr = [None if g[k] is None else g[k].data_ptr() for k in ("a_q", "a_s", "b_q", "b_s")]
        d.a_q, d.a_s, d.b_q, d.b_s = addr
        d.M, d.N, d.K = M, N, K
        d.y, d.ldy = out.data_ptr(), out.stride(0)
        d.a_fmt, d.b_fmt = _fmt(g.get("a_fmt", "e4m3")), _fmt(g.get("b_fmt", "e4m3"))
    _check(lib().mxq_gemm_bf16out_multi(descs, len(gemms), 1 if b_mn_major else 0, _stream()),
           "mxq_gemm_bf16out_multi")
    return outs


def gemm_mxfp8out(a_q, a_s, b_q, b_s, M: int, N: int, K: int, b_mn_major: bool = False,
                  want_bf16: bool = True, out=None):
    """gemm whose epilogue also emits the 1x32 E4M3 quantization of its BF16
    output (MMA-tiled scales).  Returns (y or None, y_q [M, N] u8, y_s u8)."""
    dev = a_q.device
    if out is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if want_bf16 else None
        y_q = torch.empty((M, N), dtype=torch.uint8, device=dev)
        y_s = torch.empty(scale_bytes(M, N, TILED), dtype=torch.uint8, device=dev)
    else:
        y, y_q, y_s = out
    _check(lib().mxq_gemm_mxfp8out(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), M, N, K,
                                   1 if b_mn_major else 0, _ptr(y),
                                   y.stride(0) if y is not None else 0, _ptr(y_q), _ptr(y_s), _stream()),
           "mxq_gemm_mxfp8out")
    return y, y_q, y_s


FSDP_1X32_DUAL, FSDP_32X32 = 0, 1
_RECIPES = {"mxfp8": FSDP_1X32_DUAL, "mxfp8-32x32": FSDP_32X32,
            FSDP_1X32_DUAL: FSDP_1X32_DUAL, FSDP_32X32: FSDP_32X32}


def _recipe(r) -> int:
    if r not in _RECIPES:
        raise ValueError(f"unknown recipe {r!r}")
    return _RECIPES[r]


def fsdp_payload_layout(recipe, n: int, k: int, world: int):
    """(offsets [4] (offsets[2] = -1 for 32x32), payload_bytes) of one rank's
    all-gather payload for a weight [n, k] split into `world` row shards."""
    off = (ctypes.c_int64 * 4)()
    size = ctypes.c_int64()
    _check(lib().mxq_fsdp_payload_layout(_recipe(recipe), n, k, world, off, ctypes.byref(size)),
           "mxq_fsdp_payload_layout")
    return tuple(int(v) for v in off), int(size.value)


def fsdp_quant_shard(w_shard: torch.Tensor, recipe, n: int, world: int, payload: torch.Tensor):
    """Quantizes a rank's weight shard [n/world, k] straight into its payload
    (a uint8 CUDA tensor of payload_bytes): the quantizer's outputs are views
    at the layout's offsets, so the payload needs no separate packing."""
    ns, k = w_shard.shape
    off, size = fsdp_payload_layout(recipe, n, k, world)
    if ns * world != n or payload.dtype != torch.uint8 or payload.numel() < size:
        raise ValueError("shard or payload does not match the layout")

    def view(o, nbytes, shape=None):
        t = payload[o:o + nbytes]
        return t.view(shape) if shape else t

    sf, sb = scale_bytes(ns, k, TILED), scale_bytes(k, ns, TILED)
    if _recipe(recipe) == FSDP_1X32_DUAL:
        quant_1x32_dual(w_shard, out=(view(off[0], ns * k, (ns, k)), view(off[1], sf),
                                      view(off[2], ns * k, (k, ns)), view(off[3], sb)))
    else:
        quant_32x32(w_shard, out=(view(off[0], ns * k, (ns, k)), view(off[1], sf), view(off[3], sb)))
    return payload


def fsdp_unpack(recipe, gathered: torch.Tensor, n: int, k: int, world: int, out=None):
    """Full-weight operands from the gathered payloads: (q_fwd [n,k], s_fwd,
    q_bwd [k,n] or None for 32x32, s_bwd), tiled scales."""
    dual = _recipe(recipe) == FSDP_1X32_DUAL
    dev = gathered.device
    if out is None:
        out = (torch.empty((n, k), dtype=torch.uint8, device=dev),
               torch.empty(scale_bytes(n, k, TILED), dtype=torch.uint8, device=dev),
               torch.empty((k, n), dtype=torch.uint8, device=dev) if dual else None,
               torch.empty(scale_bytes(k, n, TILED), dtype=torch.uint8, device=dev))
    q_fwd, s_fwd, q_bwd, s_bwd = out
    _check(lib().mxq_fsdp_unpack(_recipe(recipe), n, k, world, _ptr(gathered), _ptr(q_fwd), _ptr(s_fwd),
                                 _ptr(q_bwd), _ptr(s_bwd), _stream()), "mxq_fsdp_unpack")
    return out


def grouped_gemm_workspace_size(G: int, M_total: int, N: int, K: int) -> int:
    """Bytes of the optional grouped-GEMM workspace (see mxq_grouped_gemm_workspace_size)."""
    return int(lib().mxq_grouped_gemm_workspace_size(G, M_total, N, K))


def grouped_gemm(a_q, a_s, b_q, b_s, offsets: torch.Tensor, N: int, K: int, out=None, a_fmt="e4m3",
                 b_fmt="e4m3", workspace=None):
    """Per-expert y[r] = deq(A)[r] deq(B_g)^T for rows of expert g
    (offsets: int64 CUDA tensor [G+1]).  Returns y [M_total, N] bf16.
    workspace: None (row tiles on the 128-row grid), a uint8 CUDA tensor of at
    least grouped_gemm_workspace_size bytes, or "alloc" to have one allocated
    here; with a workspace the row tiles start at each expert's first row."""
    if offsets.dtype != torch.int64 or not offsets.is_cuda:
        raise ValueError("offsets must be an int64 CUDA tensor")
    G = offsets.numel() - 1
    M_total = a_q.shape[0]
    if out is None:
        out = torch.empty((M_total, N), dtype=torch.bfloat16, device=a_q.device)
    if isinstance(workspace, str):
        if workspace != "alloc":
            raise ValueError(f"workspace must be None, a tensor or 'alloc', not {workspace!r}")
        workspace = torch.empty(max(1, grouped_gemm_workspace_size(G, M_total, N, K)), dtype=torch.uint8,
                                device=a_q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().mxq_grouped_gemm_fmt(_ptr(a_q), _ptr(a_s), _fmt(a_fmt), _ptr(b_q), _ptr(b_s), _fmt(b_fmt),
                                      _ptr(offsets), G, M_total, N, K, _ptr(out), out.stride(0), _ptr(workspace),
                                      ws_bytes, _stream()), "mxq_grouped_gemm_fmt")
    return out


# Size of the library's own workspace array used by grouped_gemm_noalloc.
NOALLOC_MAX_WORKSPACE = 32 << 20


def grouped_gemm_noalloc(a_q, a_s, b_q, b_s, offsets: torch.Tensor, N: int, K: int, out: torch.Tensor):
    """grouped_gemm (E4M3) for callers that cannot allocate: the output must be
    given (dense [M_total, N] bf16) and the workspace is the library's own
    fixed device array (see mxq_grouped_gemm_noalloc: shared by all calls, so
    calls must not overlap on the GPU; problems whose workspace exceeds
    NOALLOC_MAX_WORKSPACE bytes are refused)."""
    if offsets.dtype != torch.int64 or not offsets.is_cuda:
        raise ValueError("offsets must be an int64 CUDA tensor")
    G = offsets.numel() - 1
    M_total = a_q.shape[0]
    if out.dtype != torch.bfloat16 or tuple(out.shape) != (M_total, N) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor [M_total, N]")
    _check(lib().mxq_grouped_gemm_noalloc(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), _ptr(offsets), G, M_total,
                                          N, K, _ptr(out), _stream()), "mxq_grouped_gemm_noalloc")
    return out


def group_tiled_bands(rows: int, G: int) -> int:
    """Bands a group-tiled scale buffer needs for any offsets: ceil(rows/128) + G."""
    return (rows + 127) // 128 + G


def scale_regroup_rows(s_tiled: torch.Tensor, rows: int, cols: int, offsets: torch.Tensor, bands_cap=None,
                       out=None) -> torch.Tensor:
    """Group-tiled copy (see mxq_scale_regroup_rows) of the MMA-tiled scales of a
    row quantization [rows, cols]; returns uint8 [bands_cap * ceil(cols/128) * 512]."""
    if offsets.dtype != torch.int64 or not offsets.is_cuda:
        raise ValueError("offsets must be an int64 CUDA tensor")
    G = offsets.numel() - 1
    if bands_cap is None:
        bands_cap = group_tiled_bands(rows, G)
    if out is None:
        out = torch.empty(bands_cap * ((cols // 32 + 3) // 4) * 512, dtype=torch.uint8, device=s_tiled.device)
    _check(lib().mxq_scale_regroup_rows(_ptr(s_tiled), rows, cols, _ptr(offsets), G, bands_cap, _ptr(out),
                                        _stream()), "mxq_scale_regroup_rows")
    return out


def grouped_gemm_group_tiled(a_q, a_s_grouped, b_q, b_s, offsets: torch.Tensor, N: int, K: int, bands_cap=None,
                             out=None, a_fmt="e4m3", b_fmt="e4m3"):
    """grouped_gemm with A's scales group-tiled by scale_regroup_rows (same offsets
    and bands_cap); bit-identical results, no row tile spanning two experts."""
    if offsets.dtype != torch.int64 or not offsets.is_cuda:
        raise ValueError("offsets must be an int64 CUDA tensor")
    G = offsets.numel() - 1
    M_total = a_q.shape[0]
    if bands_cap is None:
        bands_cap = group_tiled_bands(M_total, G)
    if out is None:
        out = torch.empty((M_total, N), dtype=torch.bfloat16, device=a_q.device)
    _check(lib().mxq_grouped_gemm_group_tiled(_ptr(a_q), _ptr(a_s_grouped), _fmt(a_fmt), _ptr(b_q), _ptr(b_s),
                                              _fmt(b_fmt), _ptr(offsets), G, M_total, N, K, bands_cap, _ptr(out),
                                              out.stride(0), _stream()), "mxq_grouped_gemm_group_tiled")
    return out


def get_device_status() -> int:
    """Synchronizes with the current stream; returns 0 or the recorded status
    (e.g. 5 = timeout), which the call clears."""
    return int(lib().mxq_get_device_status(_stream()))


def debug_wait_timeout(timeout_us: int) -> int:
    """Launches the bounded-wait probe (see mxq_debug_wait_timeout); 0 on launch."""
    _check(lib().mxq_debug_wait_timeout(int(timeout_us), _stream()), "mxq_debug_wait_timeout")
    return 0
