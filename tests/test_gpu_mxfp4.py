"""GPU parity of the MXFP4 entry points (E2M1 codes, E8M0 block exponents)
against the FP64 oracle: the dense bf16 copy bit for bit (every code, every
exponent byte including 0, 128/129 around the one-multiply limit, 254 and the
NaN byte 255), the GEMV over every row template, the GEMM over both kernels
(operand-swapped up to 128 rows, CTA pairs above) with tile tails, and sampled
rows of the gate_up-shaped workloads."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import TOL, act_to_torch, check_guards, guarded_out, torch_to_f64  # noqa: E402
from oracle import mxfp4_oracle as X  # noqa: E402
from oracle import w4a16_oracle as O  # noqa: E402
from w4a16_inputs import MX_WORKLOADS, make_mx_case  # noqa: E402

pytestmark = pytest.mark.gpu


class MxDevice:
    """An MXFP4 case on the device, its codes packed by the library's packer."""

    def __init__(self, case):
        self.case = case
        self.x = act_to_torch(case.x, "bf16")
        self.qw = w4.pack(torch.from_numpy(np.ascontiguousarray(case.q)).cuda(), dim=0)
        self.e = torch.from_numpy(np.ascontiguousarray(case.e)).cuda()
        self.qw_oracle = O.pack_rows(case.q)

    def reference(self, rows=None):
        if rows is None:
            return X.reference_mx(self.case.x, self.qw_oracle, self.case.e)
        return X.reference_mx_rows(self.case.x, rows, self.qw_oracle, self.case.e)


def assert_same_values(got, want, what=""):
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.array_equal(got, want, equal_nan=True), what
    assert np.array_equal(np.signbit(got), np.signbit(want)), f"{what}: signs of zero"


def assert_close(y, ref, what=""):
    got = torch_to_f64(y)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref).max()
    scale = np.abs(ref).max()
    assert err <= TOL["bf16"] * scale, f"{what}: max err {err:.3e} > {TOL['bf16']} * {scale:.3e}"


# ---------------------------------------------------------------------------
# dense copy
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["typical", "wide"])
def test_mx_dequant_bit_exact(mode):
    for (N, K) in ((16, 32), (272, 64), (1040, 96)):
        case = make_mx_case(0, N, K, seed=N + K, exponents=mode)
        d = MxDevice(case)
        buf, w, pad = guarded_out(K, N, torch.bfloat16)
        w4.mxfp4_dequant(d.qw, d.e, out=w)
        torch.cuda.synchronize()
        check_guards(buf, pad)
        assert_same_values(torch_to_f64(w), X.dequantize_mx(d.qw_oracle, case.e), (mode, N, K))


def test_mx_dequant_every_code_and_exponent():
    """Every (code, exponent byte) pair: column n has byte n, rows cycle through the 16 codes."""
    N, K = 256, 32
    q = np.tile(np.arange(16, dtype=np.uint8)[:, None], (K // 16, N))
    e = np.arange(N, dtype=np.uint8)[None, :].copy()
    qw = w4.pack(torch.from_numpy(q).cuda(), dim=0)
    w = w4.mxfp4_dequant(qw, torch.from_numpy(e).cuda())
    torch.cuda.synchronize()
    assert_same_values(torch_to_f64(w), X.dequantize_mx(O.pack_rows(q), e))


def test_mx_dequant_workload_sampled_rows():
    wl = MX_WORKLOADS["mx_dequant_43008x5376_bf16"]
    case = wl.case(seed=0)
    d = MxDevice(case)
    w = w4.mxfp4_dequant(d.qw, d.e)
    torch.cuda.synchronize()
    for k0 in (0, 8 * 97, wl.K // 2, wl.K - 8):
        assert_same_values(torch_to_f64(w[k0:k0 + 8]), X.dequantize_mx(d.qw_oracle, case.e, k0, k0 + 8), k0)


# ---------------------------------------------------------------------------
# GEMV (decode, 1 <= M <= 16)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 12, 16])
@pytest.mark.parametrize("mode", ["typical", "wide"])
def test_mx_gemv_parity(M, mode):
    for (N, K) in ((16, 32), (1040, 2048), (4112, 1024)):
        case = make_mx_case(M, N, K, seed=M * 7 + N + K, exponents=mode)
        d = MxDevice(case)
        buf, y, pad = guarded_out(M, N, torch.bfloat16)
        w4.mxfp4_gemv(d.x, d.qw, d.e, out=y)
        torch.cuda.synchronize()
        check_guards(buf, pad)
        assert_close(y, d.reference(), (M, N, K, mode))
    assert w4.device_status() == w4.OK


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("spread", ["uniform-2^-120", "uniform-2^-100", "uniform-2^100", "per-chunk", "in-chunk"])
def test_mx_gemv_activation_range(M, spread):
    """The GEMV rescales each 32-value run of x by a power of two before its
    fp16 products: activations far outside the fp16 range, runs of very
    different magnitude, runs spanning 2^40 inside themselves, and all-zero
    runs all match the oracle."""
    from w4a16_inputs import f32_to_act
    N, K = 1040, 1024
    case = make_mx_case(M, N, K, seed=M + len(spread))
    rng = np.random.Generator(np.random.PCG64(17))
    x = O.widen(case.x, "bf16")
    if spread.startswith("uniform"):
        x = x * 2.0 ** int(spread.split("^")[1])
    elif spread == "per-chunk":
        ex = rng.integers(-60, 61, size=(M, K // 32)).repeat(32, axis=1)
        x = x * np.ldexp(1.0, ex)
        x[:, 64:96] = 0.0                                   # an all-zero run
    else:
        x = x * np.ldexp(1.0, rng.integers(-20, 21, size=(M, K)))
    case.x = f32_to_act(x.astype(np.float32), "bf16")
    d = MxDevice(case)
    y = w4.mxfp4_gemv(d.x, d.qw, d.e)
    torch.cuda.synchronize()
    assert_close(y, d.reference(), (M, spread))


@pytest.mark.parametrize("N,K", [(42992, 512), (39936, 256)])
def test_mx_gemv_wide_blocks(N, K):
    """One row with more 256-column blocks than SMs but at most one 288-column
    block per SM: 9 columns a lane, three 96-column copies of the words and of
    the exponent bytes per chunk, every CTA one whole block (42992: ragged last
    block)."""
    case = make_mx_case(1, N, K, seed=N + K)
    d = MxDevice(case)
    buf, y, pad = guarded_out(1, N, torch.bfloat16)
    w4.mxfp4_gemv(d.x, d.qw, d.e, out=y)
    torch.cuda.synchronize()
    check_guards(buf, pad)
    assert_close(y, d.reference(), (1, N, K))
    assert w4.device_status() == w4.OK


@pytest.mark.parametrize("M,N,K", [(16, 10256, 1024), (8, 43008, 896), (12, 43008, 1280), (3, 4112, 2048)])
def test_mx_gemv_tensor_core_rows(M, N, K):
    """2..16 rows: the GEMV's MMA conversion on fp16-rescaled x (10 and 37 Mi
    weights, 3 rows of 8 Mi), and 12 rows of a 52.5 Mi layer, above the
    hand-over to the few-row tensor-core kernel (9..16 rows, 48 Mi weights):
    parity with the oracle, guards intact, two calls bit-identical."""
    case = make_mx_case(M, N, K, seed=M + N)
    d = MxDevice(case)
    buf, y, pad = guarded_out(M, N, torch.bfloat16)
    w4.mxfp4_gemv(d.x, d.qw, d.e, out=y)
    y2 = w4.mxfp4_gemv(d.x, d.qw, d.e)
    torch.cuda.synchronize()
    check_guards(buf, pad)
    assert torch.equal(y, y2)
    assert_close(y, d.reference(), (M, N, K))
    assert w4.device_status() == w4.OK


def test_mx_gemv_deterministic():
    case = make_mx_case(1, 4112, 4096, seed=5)
    d = MxDevice(case)
    y0 = w4.mxfp4_gemv(d.x, d.qw, d.e)
    for _ in range(3):
        assert torch.equal(w4.mxfp4_gemv(d.x, d.qw, d.e), y0)


# ---------------------------------------------------------------------------
# GEMM (prefill)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 17, 64, 65, 128, 129, 256, 300])
@pytest.mark.parametrize("mode", ["typical", "wide"])
def test_mx_gemm_parity(M, mode):
    N, K = 1040, 1024
    case = make_mx_case(M, N, K, seed=M + 3, exponents=mode)
    d = MxDevice(case)
    buf, y, pad = guarded_out(M, N, torch.bfloat16)
    w4.mxfp4_gemm(d.x, d.qw, d.e, out=y)
    torch.cuda.synchronize()
    check_guards(buf, pad)
    assert_close(y, d.reference(), (M, mode))
    assert w4.device_status() == w4.OK


def test_mx_gemm_reproduces_dense_copy():
    """One-hot rows of x: the GEMM's operand equals the dense copy, bit for bit,
    in both kernels, including blocks that need the two-multiply decode."""
    N, K = 272, 256
    case = make_mx_case(0, N, K, seed=9, exponents="wide")
    d = MxDevice(case)
    w = torch_to_f64(w4.mxfp4_dequant(d.qw, d.e))
    for M in (100, 300):
        ks = [(7 * m + 3) % K for m in range(M)]
        eye = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
        eye[torch.arange(M), torch.tensor(ks)] = 1
        y = torch_to_f64(w4.mxfp4_gemm(eye, d.qw, d.e))
        assert np.array_equal(y, w[ks]), M


@pytest.mark.parametrize("name", [n for n, w in MX_WORKLOADS.items() if w.kernel in ("gemv", "gemm")])
def test_mx_workload_sampled_rows(name):
    wl = MX_WORKLOADS[name]
    case = wl.case(seed=0)
    d = MxDevice(case)
    fn = w4.mxfp4_gemv if wl.kernel == "gemv" else w4.mxfp4_gemm
    y = fn(d.x, d.qw, d.e)
    torch.cuda.synchronize()
    rows = sorted({0, wl.M // 2, wl.M - 1, (wl.M * 5) // 7})
    assert_close(y[rows], d.reference(rows), name)
    assert w4.device_status() == w4.OK


@pytest.mark.parametrize("op,M", [("gemv", 1), ("gemv", 5), ("gemm", 40), ("gemm", 300)])
def test_mx_nan_byte_and_zero_x(op, M):
    """Degenerate inputs: an E8M0 byte 255 (NaN) makes every output of its
    column NaN and leaves the others exact; x = 0 gives y = 0 exactly."""
    N, K = 272, 256
    case = make_mx_case(M, N, K, seed=77)
    case.e[3, 17] = 255
    case.e[0, 200] = 255
    d = MxDevice(case)
    fn = w4.mxfp4_gemv if op == "gemv" else w4.mxfp4_gemm
    got = torch_to_f64(fn(d.x, d.qw, d.e))
    torch.cuda.synchronize()
    ref = d.reference()
    nan_cols = [17, 200]
    assert np.all(np.isnan(got[:, nan_cols])) and np.all(np.isnan(ref[:, nan_cols]))
    keep = [n for n in range(N) if n not in nan_cols]
    err = np.abs(got[:, keep] - ref[:, keep]).max()
    assert err <= TOL["bf16"] * np.abs(ref[:, keep]).max(), err
    zero = torch.zeros_like(d.x)
    case.e[3, 17] = case.e[0, 200] = 120
    d = MxDevice(case)
    y0 = fn(zero, d.qw, d.e)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y0.float()) == 0
    assert w4.device_status() == w4.OK
