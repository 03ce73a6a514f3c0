"""Failure detection on the GPU without a fault: a kernel wait that runs out
(a barrier nothing completes) gives up after about two seconds, records
W4A16_ERR_TIMEOUT, and the context stays usable for the next call."""
import time

import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import DeviceCase, assert_within_tol  # noqa: E402
from w4a16_inputs import make_case  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert w4.device_status() == w4.OK
    t0 = time.perf_counter()
    w4.selftest_wait_timeout()
    assert w4.device_status() == w4.ERR_TIMEOUT        # synchronises, reads and clears the word
    elapsed = time.perf_counter() - t0
    assert 0.5 < elapsed < 30.0, elapsed              # it waited, and it gave up on its own
    assert w4.device_status() == w4.OK                 # the word was cleared
    dc = DeviceCase(make_case(4, 264, 256, 32, "f16", False, seed=3))
    y = w4.gemv(dc.x, dc.qw, dc.s, dc.qz, 32)          # the context still runs work
    assert_within_tol(y, dc.reference(), "f16", "after timeout")
    assert w4.device_status() == w4.OK
