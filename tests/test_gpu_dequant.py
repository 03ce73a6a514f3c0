"""GPU parity of w4a16_dequant (the dense dequantised copy) against the FP64
oracle: W[k, n] = RN((q - z) * s) bit for bit, on small shapes over both dtypes,
every group size, symmetric and asymmetric, signed scales, and on sampled
rows of the full gate_up weights."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import TORCH_DTYPE, DeviceCase, check_guards, guarded_out, torch_to_f64  # noqa: E402
from oracle import w4a16_oracle as O  # noqa: E402
from w4a16_inputs import WORKLOADS, make_case  # noqa: E402

pytestmark = pytest.mark.gpu


def expected(case, k0=0, k1=None):
    qw, qz = O.pack_rows(case.q), (None if case.z is None else O.pack_cols(case.z))
    return O.round_to_act(O.dequantize(qw, case.s, qz, case.g, case.act, k0, k1), case.act)


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("sym", [False, True])
@pytest.mark.parametrize("g", [32, 64, 128, 256])
@pytest.mark.parametrize("scales", ["uniform", "signed"])
def test_dequant_bit_exact(act, sym, g, scales):
    for (N, K) in ((8, g), (264, 2 * g), (776, 3 * g)):
        case = make_case(1, N, K, g, act, sym, seed=N + K + g, scales=scales)
        dc = DeviceCase(case)
        buf, w, pad = guarded_out(K, N, TORCH_DTYPE[act])
        w4.dequant(dc.qw, dc.s, dc.qz, g, out=w)
        torch.cuda.synchronize()
        check_guards(buf, pad)
        assert np.array_equal(torch_to_f64(w), expected(case)), (act, sym, g, N, K)


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.kernel == "dequant"])
def test_dequant_workload_sampled_rows(name):
    wl = WORKLOADS[name]
    case = wl.case(seed=0)
    dc = DeviceCase(case)
    w = w4.dequant(dc.qw, dc.s, dc.qz, wl.g)
    torch.cuda.synchronize()
    for k0 in (0, 8 * 97, wl.K // 2, wl.K - 8):      # blocks of 8 rows across the matrix
        assert np.array_equal(torch_to_f64(w[k0:k0 + 8]), expected(case, k0, k0 + 8)), (name, k0)


def test_dequant_matches_gemm_operand():
    """The GEMM dequantises to the same values: x = one-hot rows reproduce W rows."""
    case = make_case(130, 264, 256, 32, "bf16", False, seed=11)
    dc = DeviceCase(case)
    w = torch_to_f64(w4.dequant(dc.qw, dc.s, dc.qz, 32))
    eye = torch.zeros((130, 256), dtype=torch.bfloat16, device="cuda")
    ks = [(7 * m + 3) % 256 for m in range(130)]
    eye[torch.arange(130), torch.tensor(ks)] = 1
    y = torch_to_f64(w4.gemm(eye, dc.qw, dc.s, dc.qz, 32))
    assert np.array_equal(y, w[ks])
