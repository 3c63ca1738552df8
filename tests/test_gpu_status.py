"""Failure detection on the GPU without a fault: every wait in the kernels
is bounded; a wait that runs out records MXQ_ERR_TIMEOUT in a device status
word and the kernel returns.  The probe kernel waits on a barrier that no
thread ever completes (1 ms limit) -- the same bounded-wait routine the
GEMM pipeline uses -- and the host reads the status afterwards.  The
context stays usable: a normal call right after still succeeds.
"""
import pytest
import torch

from _util import gpu_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gpu_or_skip()


def test_bounded_wait_reports_timeout_and_context_survives():
    from mxfp8_microscaled_precision_gb300 import mxq
    assert mxq.get_device_status() == 0
    assert mxq.debug_wait_timeout(1000) == 0           # launch OK
    assert mxq.get_device_status() == 5                 # MXQ_ERR_TIMEOUT recorded
    assert mxq.get_device_status() == 0                 # and cleared
    x = torch.randn(64, 64).to(torch.bfloat16).cuda()   # context still usable
    q, s, _, _ = mxq.quant_1x32_dual(x, col=False)
    torch.cuda.synchronize()
    assert q.shape == (64, 64)
    assert mxq.get_device_status() == 0


def test_bad_arguments_raise_value_error():
    from mxfp8_microscaled_precision_gb300 import mxq
    x = torch.randn(64, 48).to(torch.bfloat16).cuda()
    with pytest.raises(ValueError):
        mxq.quant_1x32_dual(x)                          # 48 is not a multiple of 32
    with pytest.raises(ValueError):
        mxq.debug_wait_timeout(0)


def test_status_on_a_side_stream():
    """The status call synchronizes with the stream it is given: a timeout
    recorded by a kernel on a side stream is reported by a call on that
    stream, once."""
    from mxfp8_microscaled_precision_gb300 import mxq
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert mxq.get_device_status() == 0
        assert mxq.debug_wait_timeout(1000) == 0
        assert mxq.get_device_status() == 5
        assert mxq.get_device_status() == 0
    assert mxq.get_device_status() == 0
