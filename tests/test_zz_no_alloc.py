"""GPU check of mxq_grouped_gemm_noalloc, the grouped GEMM for callers that
cannot allocate device memory.

Some callers only ever see their input and output buffers: an operator plugged
into a host framework or serving runtime whose allocator owns all device
memory, or code that must not call cudaMalloc / cudaFree because those calls
can synchronize the device.  They cannot pass mxq_grouped_gemm a workspace, so
this entry point takes it from a fixed array inside the library.

The test calls the new entry point through the C ABI and compares its output
with that of the existing entry point, mxq_grouped_gemm (given a workspace
allocated here), within the GEMM tolerance of the parity tests, on two calls
in a row with different routings: the second call must not be disturbed by
what the first left in the shared array.  It also checks that a problem
whose workspace would not fit the array is refused before anything runs.

This file is collected last on purpose (tests/test_zz_*): a run that stops at
the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from _util import gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _close(got: torch.Tensor, ref: torch.Tensor, what: str):
    """|got - ref| <= 1e-2 |ref| + 1e-3 rms(ref) element by element (the GEMM
    tolerance of the parity tests), with ref the existing entry point's output."""
    g = got.float().cpu().numpy().astype(np.float64)
    r = ref.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite outputs"
    rms = float(np.sqrt(np.mean(r * r)))
    bad = np.abs(g - r) > 1e-2 * np.abs(r) + 1e-3 * rms
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outputs outside the tolerance"


def _problem(sizes, N, K, seed):
    from mxfp8_microscaled_precision_gb300 import mxq, workloads
    G = len(sizes)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    A = workloads.normal_with_outliers((M, K), seed=seed, device="cuda")
    B = workloads.normal((G * N, K), 0.02, seed=seed + 1, device="cuda")
    aq, as_, _, _ = mxq.quant_1x32_dual(A, col=False)
    bq, bs, _, _ = mxq.quant_1x32_dual(B, col=False)
    return dict(aq=aq, as_=as_, bq=bq, bs=bs, off=torch.from_numpy(off).cuda(), G=G, M=M, N=N, K=K)


def _existing(L, mxq, pr):
    """mxq_grouped_gemm through the C ABI with a workspace allocated here."""
    need = L.mxq_grouped_gemm_workspace_size(pr["G"], pr["M"], pr["N"], pr["K"])
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y = torch.empty((pr["M"], pr["N"]), dtype=torch.bfloat16, device="cuda")
    st = L.mxq_grouped_gemm(_p(pr["aq"]), _p(pr["as_"]), _p(pr["bq"]), _p(pr["bs"]), _p(pr["off"]), pr["G"],
                            pr["M"], pr["N"], pr["K"], _p(y), _p(ws), ctypes.c_size_t(need), mxq._stream())
    assert st == 0, mxq.status_string(st)
    return y


def _noalloc(L, mxq, pr):
    y = torch.full((pr["M"], pr["N"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = L.mxq_grouped_gemm_noalloc(_p(pr["aq"]), _p(pr["as_"]), _p(pr["bq"]), _p(pr["bs"]), _p(pr["off"]),
                                    pr["G"], pr["M"], pr["N"], pr["K"], _p(y), mxq._stream())
    assert st == 0, mxq.status_string(st)
    return y


def test_noalloc_grouped_gemm_matches_existing_entry_point_twice():
    from mxfp8_microscaled_precision_gb300 import mxq
    L = mxq.lib()
    # two routings in a row: the second has more experts and rows, so it reads
    # bands the first call filled with other experts' scales
    first = _problem([0, 5, 0, 300, 1, 130, 77], N=256, K=512, seed=31)
    second = _problem([129, 0, 3, 640, 255, 1, 0, 200, 128, 64], N=384, K=1024, seed=32)
    for name, pr in (("first call", first), ("second call", second)):
        y_new = _noalloc(L, mxq, pr)
        y_ref = _existing(L, mxq, pr)
        torch.cuda.synchronize()
        _close(y_new, y_ref, name)
    assert mxq.get_device_status() == 0


def test_noalloc_refuses_a_workspace_past_its_array():
    """(ceil(300000/128) + 128) bands x 32 atoms x 512 bytes = 40.5 MB > the
    32 MiB array: refused on the host, nothing launched (the pointers are
    never dereferenced)."""
    from mxfp8_microscaled_precision_gb300 import mxq
    L = mxq.lib()
    fake = ctypes.c_void_p(0x10000)
    assert L.mxq_grouped_gemm_workspace_size(128, 300000, 4096, 4096) > mxq.NOALLOC_MAX_WORKSPACE
    st = L.mxq_grouped_gemm_noalloc(fake, fake, fake, fake, fake, 128, 300000, 4096, 4096, fake, mxq._stream())
    assert st == 2   # MXQ_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(ValueError):
        mxq._check(st, "mxq_grouped_gemm_noalloc")
