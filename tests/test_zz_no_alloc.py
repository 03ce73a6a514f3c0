"""w4a16_gemv_noalloc: the decode GEMV for callers that cannot allocate device memory.

Some callers have no allocator to draw scratch memory from (a plugin inside a
host program that owns all device memory, a serving process whose memory is
already reserved, a loop where cudaMalloc's synchronisation is not allowed).
For them the library keeps a fixed scratch array on the device and this entry
point takes no workspace. These tests call it through the C ABI and check that
it gives the same outputs as w4a16_gemv, bit for bit (both run the same plan
and sum split column blocks in the same fixed order), on two calls in a row
(the array keeps the previous call's contents, so the second call checks that
nothing leaks from one call into the next), and, on one case, that it matches
the FP64 oracle within the parity tolerance. This file is collected last.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import TOL, DeviceCase, assert_within_tol, torch_to_f64  # noqa: E402
from w4a16_inputs import make_case  # noqa: E402

pytestmark = pytest.mark.gpu


def call_noalloc(dc, y):
    lib = w4.load_library()
    c = dc.case
    return lib.w4a16_gemv_noalloc(dc.x.data_ptr(), dc.qw.data_ptr(), dc.s.data_ptr(),
                                  None if dc.qz is None else dc.qz.data_ptr(), y.data_ptr(),
                                  c.M, c.N, c.K, c.g, w4.F16 if c.act == "f16" else w4.BF16,
                                  torch.cuda.current_stream().cuda_stream)


CASES = [
    (1, 43008, 5376, 32, "f16", False),     # the gate_up-like decode shape
    (4, 2048, 2048, 128, "bf16", False),
    (3, 264, 256, 32, "f16", True),         # ragged column block, symmetric
    (16, 776, 1024, 64, "bf16", False),
    (1, 4104, 2048, 32, "bf16", False),     # N % 32 != 0: zero-points read per lane
    (8, 8192, 4096, 128, "f16", False),     # MMA conversion, 8-row template
    (12, 43008, 640, 32, "bf16", False),    # MMA conversion, 16-row template
]


@pytest.mark.parametrize("M,N,K,g,act,sym", CASES)
def test_noalloc_matches_gemv_on_two_calls(M, N, K, g, act, sym):
    dc = DeviceCase(make_case(M, N, K, g, act, sym, seed=M + N + K))
    y_ref = w4.gemv(dc.x, dc.qw, dc.s, dc.qz, g)
    torch.cuda.synchronize()
    ref = torch_to_f64(y_ref)
    scale = np.abs(ref).max()
    for _ in range(2):
        y = torch.full_like(y_ref, float("nan"))
        assert call_noalloc(dc, y) == w4.OK
        torch.cuda.synchronize()
        got = torch_to_f64(y)
        assert np.all(np.isfinite(got))
        assert np.abs(got - ref).max() <= TOL[act] * scale
        assert torch.equal(y, y_ref), "w4a16_gemv_noalloc differs from w4a16_gemv"
    assert w4.device_status() == w4.OK


def test_noalloc_matches_oracle():
    """One case through the oracle as well: two calls, each within the parity tolerance."""
    dc = DeviceCase(make_case(2, 1032, 2048, 128, "bf16", False, seed=7))
    ref = dc.reference()
    for _ in range(2):
        y = torch.full((2, 1032), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(dc, y) == w4.OK
        torch.cuda.synchronize()
        assert_within_tol(y, ref, "bf16", "noalloc vs oracle")
    assert w4.device_status() == w4.OK


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """N = 2^30 needs 16 MiB of ticket words alone: rejected on the host, nothing launched."""
    dc = DeviceCase(make_case(1, 256, 256, 32, "f16", False, seed=0))
    lib = w4.load_library()
    y = torch.empty(1, 256, dtype=torch.float16, device="cuda")
    st = lib.w4a16_gemv_noalloc(dc.x.data_ptr(), dc.qw.data_ptr(), dc.s.data_ptr(), dc.qz.data_ptr(),
                                y.data_ptr(), 1, 1 << 30, 256, 32, w4.F16,
                                torch.cuda.current_stream().cuda_stream)
    assert st == w4.ERR_WORKSPACE
