"""GPU parity on the full-size decode and prefill workloads, in the launch
configuration the benchmark times: whole outputs against the FP64 oracle for
every decode GEMV, sampled rows (the first, the last and rows spread over
every M tile edge) for the prefill GEMMs (bf16 and fp16, g = 32 and 128, M = 64
to 2048)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import DeviceCase, assert_within_tol, torch_to_f64  # noqa: E402
from w4a16_inputs import WORKLOADS  # noqa: E402

pytestmark = pytest.mark.gpu

GEMV = [n for n, w in WORKLOADS.items() if w.kernel == "gemv"]
GEMM = [n for n, w in WORKLOADS.items() if w.kernel == "gemm"]


@pytest.mark.parametrize("name", GEMV)
def test_decode_workload(name):
    wl = WORKLOADS[name]
    dc = DeviceCase(wl.case(seed=0))
    y = w4.gemv(dc.x, dc.qw, dc.s, dc.qz, wl.g)
    torch.cuda.synchronize()
    assert_within_tol(y, dc.reference(), wl.act, name)
    assert w4.device_status() == w4.OK


@pytest.mark.parametrize("name", GEMM)
def test_prefill_workload_sampled_rows(name):
    wl = WORKLOADS[name]
    dc = DeviceCase(wl.case(seed=0))
    y = w4.gemm(dc.x, dc.qw, dc.s, dc.qz, wl.g)
    torch.cuda.synchronize()
    assert w4.device_status() == w4.OK
    # both 128-row halves of a CTA pair's 256-row tile, the tile edges, the last rows
    rows = sorted(r for r in {0, 1, 127, 128, 129, 255, 256, 257, 1000, 1023, 1024, 1500,
                              wl.M - 129, wl.M - 2, wl.M - 1} if 0 <= r < wl.M)
    ref = dc.reference(rows=rows)
    got = y[rows]
    assert_within_tol(got, ref, wl.act, name)
    # every output row is finite, and the unsampled rows are not left unwritten
    yf = torch_to_f64(y[::97])
    assert np.all(np.isfinite(yf)) and np.abs(yf).max() > 0
