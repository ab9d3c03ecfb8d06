"""Failure detection without a GPU fault: a bounded device wait that nothing
completes must give up, record QLIN_ERR_TIMEOUT and leave the context usable."""
import time

import pytest
import torch

import precision_quantized_linear_gb300 as q

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    assert q.qlin_get_device_error() == 0
    t0 = time.perf_counter()
    q.qlin_selftest_wait_timeout(20000)          # 20 ms limit
    status = q.qlin_get_device_error()
    dt = time.perf_counter() - t0
    assert status == 7, q.qlin_status_string(status)
    assert dt < 5.0
    assert q.qlin_get_device_error() == 0          # read-and-clear
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0                # the context still works


def test_selftest_rejects_bad_limit():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    with pytest.raises(q.QlinError) as e:
        q.qlin_selftest_wait_timeout(0)
    assert e.value.status == 1
