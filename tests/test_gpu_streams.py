"""Calls on a stream other than torch's current one.

The binding keeps one workspace per (device, stream, op), allocated and
zero-filled on the stream the call runs on, so the zero fill is ordered before
the kernel that relies on zeroed ticket words. These tests pass `stream=`
explicitly: the GEMV (FMA and MMA conversions, split column blocks), the
few-row and CTA-pair GEMM, and the MXFP4 GEMV, on a side stream that waits
for the inputs, then a larger shape on the same stream that outgrows the
cached workspace. Every result is compared with the FP64 oracle.
"""
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import DeviceCase, assert_within_tol  # noqa: E402
from w4a16_inputs import make_case, make_mx_case  # noqa: E402

pytestmark = pytest.mark.gpu


def on_side_stream(fn):
    """Run fn(stream) on a fresh stream that first waits for the current one;
    synchronise the device before returning its result."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    out = fn(side)
    torch.cuda.synchronize()
    return out


# (op, M, N, K, g, act): small first, then shapes that need more workspace
CASES = [
    ("gemv", 1, 2048, 2048, 128, "f16"),     # FMA conversion, cluster-summed blocks
    ("gemv", 4, 6144, 2048, 128, "bf16"),    # MMA conversion
    ("gemv", 3, 20480, 512, 32, "f16"),      # stream-K with ticket fix-up (more blocks than SMs)
    ("gemm", 24, 4104, 1024, 64, "bf16"),    # few-row kernel: partial slots and tickets
    ("gemm", 200, 2048, 512, 32, "f16"),     # CTA-pair kernel (no workspace)
]


@pytest.mark.parametrize("op,M,N,K,g,act", CASES)
def test_side_stream_parity(op, M, N, K, g, act):
    dc = DeviceCase(make_case(M, N, K, g, act, False, seed=M + N))
    fn = getattr(w4, op)
    y = on_side_stream(lambda s: fn(dc.x, dc.qw, dc.s, dc.qz, g, stream=s))
    assert_within_tol(y, dc.reference(), act, f"{op} on a side stream M={M} N={N}")
    assert w4.device_status() == w4.OK


def test_side_stream_workspace_grows():
    """A small GEMV then a much larger one on the same side stream: the second
    outgrows the cached workspace, which is replaced on that stream."""
    small = DeviceCase(make_case(2, 1024, 1024, 128, "f16", False, seed=3))
    large = DeviceCase(make_case(2, 30720, 512, 32, "f16", False, seed=4))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    y1 = w4.gemv(small.x, small.qw, small.s, small.qz, 128, stream=side)
    y2 = w4.gemv(large.x, large.qw, large.s, large.qz, 32, stream=side)
    y3 = w4.gemv(small.x, small.qw, small.s, small.qz, 128, stream=side)
    torch.cuda.synchronize()
    assert_within_tol(y1, small.reference(), "f16", "small before growth")
    assert_within_tol(y2, large.reference(), "f16", "large")
    assert torch.equal(y1, y3)
    assert w4.device_status() == w4.OK


def test_side_stream_mxfp4_gemv():
    from test_gpu_mxfp4 import MxDevice, assert_close
    d = MxDevice(make_mx_case(5, 4112, 1024, seed=8))
    y = on_side_stream(lambda s: w4.mxfp4_gemv(d.x, d.qw, d.e, stream=s))
    assert_close(y, d.reference(), "mxfp4 gemv on a side stream")
    assert w4.device_status() == w4.OK
