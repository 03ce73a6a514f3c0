"""Parity at the largest sizes a single layer meets on one GB300, where 32-bit
offsets would overflow:

* packed weights past 4 GiB (K = 135168, N = 65808: 4.45 GB of codes), through
  the GEMV, both GEMM kernels and the dense copy, for the int4 layer and MXFP4;
* a GEMM output past 2^31 elements (M = 16384, N = 131080);
* a dense copy past 2^32 elements (17.8 GB);
* the packer and unpacker past 2^32 codes.

The weights are drawn as packed words on the device (a uniform random word is
eight uniform codes). The oracle checks sampled columns, which depend only on
their own weights, scales and zero-points (8-column blocks, so that the packed
zero-points slice by whole words), including the ragged last block; the round
trip pack -> unpack is compared over the whole tensor."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import weight_only_int4_gb300 as w4  # noqa: E402
from gpu_util import TOL, act_to_torch, torch_to_f64  # noqa: E402
from oracle import mxfp4_oracle as X  # noqa: E402
from oracle import w4a16_oracle as O  # noqa: E402
from w4a16_inputs import device_codes, make_case, make_large_case, make_large_mx_case  # noqa: E402

pytestmark = pytest.mark.gpu

N_BIG, K_BIG, G_BIG = 65808, 135168, 256          # 4.45 GB of packed weights; N = 257 * 256 + 16
BLOCKS = (0, 4111, N_BIG // 8 - 1)                 # 8-column blocks: first, middle, last (ragged tile)
COLS = np.concatenate([np.arange(8 * b, 8 * b + 8) for b in BLOCKS])


def _host_words(t):
    """int32 device words -> numpy int32 (the oracle reads them as unsigned)."""
    return t.cpu().numpy()


def _assert_close(got, ref, what):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref).max()
    scale = np.abs(ref).max()
    assert err <= TOL["bf16"] * scale, f"{what}: max err {err:.3e} > {TOL['bf16']} * {scale:.3e}"


@pytest.fixture(scope="module")
def big():
    case = make_large_case(160, N_BIG, K_BIG, G_BIG, "bf16", seed=31)
    assert case.qw.numel() * 4 > 2 ** 32
    dev = {
        "x": act_to_torch(case.x, "bf16"),
        "s": act_to_torch(case.s, "bf16"),
        "qz": torch.from_numpy(case.zw.view(np.int32)).cuda(),
    }
    cols_t = torch.from_numpy(COLS).cuda()
    oracle = {   # the sampled columns' operands, on the host
        "qw": _host_words(case.qw.index_select(1, cols_t)),
        "s": np.ascontiguousarray(case.s[:, COLS]),
        "zw": np.ascontiguousarray(case.zw[:, list(BLOCKS)]).view(np.int32),
    }
    yield case, dev, oracle
    del dev
    case.qw = None
    torch.cuda.empty_cache()


def _ref_cols(case, oracle, M):
    return O.reference(case.x[:M], oracle["qw"], oracle["s"], oracle["zw"], G_BIG, "bf16")


@pytest.mark.parametrize("M", [1, 16])
def test_gemv_weights_past_4gib(big, M):
    case, dev, oracle = big
    y = w4.gemv(dev["x"][:M].contiguous(), case.qw, dev["s"], dev["qz"], G_BIG)
    torch.cuda.synchronize()
    _assert_close(torch_to_f64(y[:, COLS]), _ref_cols(case, oracle, M), ("gemv", M))
    assert w4.device_status() == w4.OK


@pytest.mark.parametrize("M", [64, 160])   # operand-swapped stream-K kernel; CTA pairs (M tail)
def test_gemm_weights_past_4gib(big, M):
    case, dev, oracle = big
    y = w4.gemm(dev["x"][:M].contiguous(), case.qw, dev["s"], dev["qz"], G_BIG)
    torch.cuda.synchronize()
    _assert_close(torch_to_f64(y[:, COLS]), _ref_cols(case, oracle, M), ("gemm", M))
    assert w4.device_status() == w4.OK


def test_dequant_past_2pow32_elements(big):
    case, dev, oracle = big
    w = w4.dequant(case.qw, dev["s"], dev["qz"], G_BIG)      # [K, N] bf16: 17.8 GB
    assert w.numel() > 2 ** 32
    torch.cuda.synchronize()
    want = O.round_to_act(O.dequantize(oracle["qw"], oracle["s"], oracle["zw"], G_BIG, "bf16"), "bf16")
    assert np.array_equal(torch_to_f64(w[:, COLS]), want)
    # every column of the last group: the highest offsets of the copy
    k0 = K_BIG - G_BIG
    qw_tail = _host_words(case.qw[k0 // 8:])
    want = O.round_to_act(O.dequantize(qw_tail, case.s[-1:], case.zw[-1:].view(np.int32), G_BIG, "bf16"), "bf16")
    assert np.array_equal(torch_to_f64(w[k0:]), want)
    del w
    torch.cuda.empty_cache()


def test_gemm_output_past_2pow31_elements():
    """y [16384, 131080] bf16 (4.3 GB): rows at both ends of the output."""
    M, N, K, g = 16384, 131080, 96, 32
    case = make_case(M, N, K, g, "bf16", False, seed=5)
    x = act_to_torch(case.x, "bf16")
    s = act_to_torch(case.s, "bf16")
    qw = w4.pack(torch.from_numpy(case.q).cuda(), dim=0)
    qz = w4.pack(torch.from_numpy(case.z).cuda(), dim=1)
    y = w4.gemm(x, qw, s, qz, g)
    assert y.numel() > 2 ** 31
    torch.cuda.synchronize()
    rows = [0, M // 2 + 3, M - 1]
    ref = O.reference_rows(case.x, rows, O.pack_rows(case.q), case.s, O.pack_cols(case.z), g, "bf16")
    _assert_close(torch_to_f64(y[rows]), ref, "gemm rows")
    assert w4.device_status() == w4.OK
    del y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dim", [0, 1])
def test_pack_past_2pow32_codes(dim):
    R, C = 135168, 32776
    codes = device_codes((R, C), seed=3 + dim)
    assert codes.numel() > 2 ** 32
    words = w4.pack(codes, dim=dim)
    torch.cuda.synchronize()
    if dim == 0:
        for w in (0, R // 16 + 5, R // 8 - 1):                # word rows at both ends
            want = O.pack_rows(codes[8 * w:8 * w + 8].cpu().numpy())
            assert np.array_equal(_host_words(words[w:w + 1]), want), w
    else:
        for r in (0, R // 2 + 1, R - 1):
            want = O.pack_cols(codes[r:r + 1].cpu().numpy())
            assert np.array_equal(_host_words(words[r:r + 1]), want), r
    back = w4.unpack(words, dim=dim)
    assert torch.equal(back, codes)
    del codes, words, back
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def big_mx():
    case = make_large_mx_case(64, N_BIG, K_BIG, seed=37)
    x = act_to_torch(case.x, "bf16")
    e = torch.from_numpy(case.s).cuda()
    qw_cols = _host_words(case.qw.index_select(1, torch.from_numpy(COLS).cuda()))
    yield case, x, e, qw_cols
    case.qw = None
    del x, e
    torch.cuda.empty_cache()


@pytest.mark.parametrize("op,M", [("gemv", 1), ("gemv", 16), ("gemm", 64)])
def test_mx_weights_past_4gib(big_mx, op, M):
    case, x, e, qw_cols = big_mx
    fn = w4.mxfp4_gemv if op == "gemv" else w4.mxfp4_gemm
    y = fn(x[:M].contiguous(), case.qw, e)
    torch.cuda.synchronize()
    ref = X.reference_mx(case.x[:M], qw_cols, np.ascontiguousarray(case.s[:, COLS]))
    _assert_close(torch_to_f64(y[:, COLS]), ref, (op, M))
    assert w4.device_status() == w4.OK


def test_mx_dequant_past_2pow32_elements(big_mx):
    case, x, e, qw_cols = big_mx
    w = w4.mxfp4_dequant(case.qw, e)
    torch.cuda.synchronize()
    want = X.dequantize_mx(qw_cols, np.ascontiguousarray(case.s[:, COLS]))
    got = torch_to_f64(w[:, COLS])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
    del w
    torch.cuda.empty_cache()
