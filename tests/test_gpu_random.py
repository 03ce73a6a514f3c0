"""Seeded random sweep of shapes for the three compute entry points against the
FP64 oracle: ragged N (multiples of 8), K spanning 1..12 groups (with and
without a half K step), every group size, both dtypes, symmetric and
asymmetric, and M across the GEMV range and every GEMM row bucket."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import TORCH_DTYPE, DeviceCase, assert_within_tol, check_guards, guarded_out, torch_to_f64  # noqa: E402
from oracle import w4a16_oracle as O  # noqa: E402
from w4a16_inputs import make_case  # noqa: E402

pytestmark = pytest.mark.gpu


def _shapes(seed, count, m_lo, m_hi):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        g = int(rng.choice([32, 64, 128, 256]))
        out.append((int(rng.integers(m_lo, m_hi + 1)), 8 * int(rng.integers(1, 160)), g * int(rng.integers(1, 13)), g,
                    str(rng.choice(["f16", "bf16"])), bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("M,N,K,g,act,sym", _shapes(101, 24, 1, 16))
def test_gemv_random(M, N, K, g, act, sym):
    dc = DeviceCase(make_case(M, N, K, g, act, sym, seed=M * 7 + N + K))
    buf, y, pad = guarded_out(M, N, TORCH_DTYPE[act])
    w4.gemv(dc.x, dc.qw, dc.s, dc.qz, g, out=y)
    torch.cuda.synchronize()
    check_guards(buf, pad)
    assert_within_tol(y, dc.reference(), act, f"gemv {M}x{N}x{K} g{g} {act} sym={sym}")


@pytest.mark.parametrize("M,N,K,g,act,sym", _shapes(202, 24, 1, 400))
def test_gemm_random(M, N, K, g, act, sym):
    dc = DeviceCase(make_case(M, N, K, g, act, sym, seed=M * 7 + N + K))
    buf, y, pad = guarded_out(M, N, TORCH_DTYPE[act])
    w4.gemm(dc.x, dc.qw, dc.s, dc.qz, g, out=y)
    torch.cuda.synchronize()
    check_guards(buf, pad)
    assert_within_tol(y, dc.reference(), act, f"gemm {M}x{N}x{K} g{g} {act} sym={sym}")
    assert w4.device_status() == w4.OK


@pytest.mark.parametrize("M,N,K,g,act,sym", _shapes(303, 12, 1, 1))
def test_dequant_random(M, N, K, g, act, sym):
    case = make_case(1, N, K, g, act, sym, seed=N + K)
    dc = DeviceCase(case)
    w = w4.dequant(dc.qw, dc.s, dc.qz, g)
    qw, qz = O.pack_rows(case.q), (None if case.z is None else O.pack_cols(case.z))
    want = O.round_to_act(O.dequantize(qw, case.s, qz, g, act), act)
    assert np.array_equal(torch_to_f64(w), want)
