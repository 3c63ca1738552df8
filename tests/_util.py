"""Helpers shared by the GPU parity tests (no method arithmetic here: the
expected values always come from the oracle)."""
import numpy as np
import pytest
import torch


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor (copied to the host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def gpu_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip(f"needs sm_103 (GB300), found sm_{major}{minor}")
    from mxfp8_microscaled_precision_gb300 import build
    build.build()


def assert_gemm_close(got: torch.Tensor, ref_bits: np.ndarray, what: str = "gemm"):
    """|gpu - ref| <= 1e-2 |ref| + 1e-3 rms(ref), element by element, rms over
    the compared outputs (the tolerance the GEMM parity bar states)."""
    from oracle import oracle
    g = got.detach().float().cpu().numpy().astype(np.float64)
    r = oracle.bf16_to_double(ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    err = np.abs(g - r)
    bound = 1e-2 * np.abs(r) + 1e-3 * rms
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; first at "
                             f"{tuple(i)}: gpu {g[tuple(i)]!r} ref {r[tuple(i)]!r} (rms {rms:.3g})")
    return float((err / np.maximum(bound, 1e-300)).max()) if r.size else 0.0


def tiled_to_plain(s_tiled: np.ndarray, rows: int, groups: int) -> np.ndarray:
    """Inverse of the MMA-tiled scale permutation, taken from the oracle's
    forward map applied to index-valued inputs (the low and high index digits
    in two passes), so that only plain [rows, groups] scales are compared."""
    from oracle import oracle
    idx = np.arange(rows * groups, dtype=np.int64)
    lo = oracle.scale_tiled((idx % 251 + 1).astype(np.uint8).reshape(rows, groups))
    hi = oracle.scale_tiled((idx // 251 % 251 + 1).astype(np.uint8).reshape(rows, groups))
    pos = np.flatnonzero(lo)
    plain_index = (lo[pos].astype(np.int64) - 1) + 251 * (hi[pos].astype(np.int64) - 1)
    out = np.zeros(rows * groups, np.uint8)
    out[plain_index] = s_tiled[pos]
    return out.reshape(rows, groups)
