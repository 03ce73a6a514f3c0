"""CPU tests of the FP64 oracle against its pins (no GPU, no CUDA library)."""
import numpy as np
import pytest

import oracle_pins as P
from oracle import w4a16_oracle as O
from w4a16_inputs import make_case, make_large_case


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_roundtrip_random_words():
    rng = np.random.default_rng(0)
    for (R, C) in ((8, 1), (64, 24), (16, 8)):
        codes = rng.integers(0, 16, size=(R, C), dtype=np.uint8)
        assert np.array_equal(O.unpack_rows(O.pack_rows(codes)), codes)
        codes_c = rng.integers(0, 16, size=(C, R), dtype=np.uint8)
        assert np.array_equal(O.unpack_cols(O.pack_cols(codes_c)), codes_c)
    w = rng.integers(-(1 << 31), 1 << 31, size=(5, 7), dtype=np.int64).astype(np.int32)
    assert np.array_equal(O.pack_rows(O.unpack_rows(w)), w)
    assert np.array_equal(O.pack_cols(O.unpack_cols(w)), w)


def test_single_word_column_block():
    """N = 8: exactly one packed zero-point word per group row."""
    case = make_case(2, 8, 64, 32, "f16", False, seed=4)
    qz = O.pack_cols(case.z)
    assert qz.shape == (2, 1)
    y = O.reference(case.x, O.pack_rows(case.q), case.s, qz, 32, "f16")
    want = P.exact_layer(case)
    assert np.allclose(y, np.array([[float(v) for v in r] for r in want]), rtol=1e-12, atol=1e-12)


def test_widen_exact():
    f16 = np.array([1.0, -2.5, 65504.0, 2.0 ** -24, 0.0], dtype=np.float16)
    assert np.array_equal(O.widen(f16, "f16"), f16.astype(np.float64))
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F], dtype=np.uint16)
    want = [1.0, -2.0, 1.0078125, 2.0 ** -133, float(np.float32(3.3895313892515355e38))]
    assert np.array_equal(O.widen(bits, "bf16"), np.array(want))


def test_round_to_act_f16_matches_numpy():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000),
                        np.array([0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26])])
    got = O.round_to_act(v, "f16")
    with np.errstate(over="ignore"):
        want = v.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, want)


def test_round_to_act_bf16_by_enumeration():
    """Nearest bf16 by exhaustive search over neighbouring bit patterns, ties to even."""
    rng = np.random.default_rng(3)
    v = rng.standard_normal(3000) * 10.0 ** rng.uniform(-40, 30, 3000)
    # exact ties: midpoints between adjacent bf16 values
    lo = np.array([0x3F80, 0x3F81, 0x4000, 0xC123], dtype=np.uint32)
    mids = (O.widen(lo.astype(np.uint16), "bf16") + O.widen((lo + 1).astype(np.uint16), "bf16")) / 2
    v = np.concatenate([v, mids])
    got = O.round_to_act(v, "bf16")
    for val, r in zip(v, got):
        mag = abs(val)
        b = int(np.float32(mag).view(np.uint32)) >> 16          # truncated magnitude pattern
        cands = [c for c in (b - 1, b, b + 1, b + 2) if 0 <= c <= 0x7F7F]
        vals = O.widen(np.array(cands, dtype=np.uint16), "bf16")
        dist = np.abs(vals - mag)
        best = dist.min()
        ties = [c for c, d in zip(cands, dist) if d == best]
        pick = [c for c in ties if c % 2 == 0] if len(ties) > 1 else ties
        want = O.widen(np.array(pick[:1], dtype=np.uint16), "bf16")[0]
        assert r == np.copysign(want, val), (val, r, want)


def test_sampled_rows_and_cols_match_full():
    case = make_case(5, 64, 256, 128, "bf16", False, seed=8)
    qw, qz = P.packed_operands(case)
    full = O.reference(case.x, qw, case.s, qz, 128, "bf16")
    rows = [0, 3, 4]
    cols = [0, 9, 63, 17]
    assert np.allclose(O.reference_rows(case.x, rows, qw, case.s, qz, 128, "bf16"), full[rows],
                       rtol=1e-13, atol=1e-13)
    assert np.allclose(O.reference_cols(case.x, cols, qw, case.s, qz, 128, "bf16"), full[:, cols],
                       rtol=1e-13, atol=1e-13)


def test_column_blocks_sliced_from_the_operands():
    """Output columns depend only on their own operands: the layer on 8-column
    blocks cut out of qweight, scales and the packed zero-point words (whole
    words) equals those columns of the full layer. The large GPU tests check
    sampled columns this way."""
    case = make_large_case(5, 272, 512, 128, "bf16", seed=3, device="cpu")
    blocks = [0, 17, 33]
    cols = np.concatenate([np.arange(8 * b, 8 * b + 8) for b in blocks])
    qw = case.qw.numpy()
    zw = case.zw.view(np.int32)
    full = O.reference(case.x, qw, case.s, zw, 128, "bf16")
    part = O.reference(case.x, np.ascontiguousarray(qw[:, cols]), np.ascontiguousarray(case.s[:, cols]),
                       np.ascontiguousarray(zw[:, blocks]), 128, "bf16")
    assert np.array_equal(part, full[:, cols])


def test_rejects_bad_operands():
    case = make_case(1, 16, 64, 32, "f16", False, seed=0)
    qw, qz = P.packed_operands(case)
    with pytest.raises(ValueError):
        O.reference(case.x, qw, case.s, qz[:, :1], 32, "f16")      # zero-points of the wrong width
    with pytest.raises(ValueError):
        O.reference(case.x[:, :32], qw, case.s, qz, 32, "f16")     # K mismatch
    with pytest.raises(ValueError):
        O.pack_rows(np.full((8, 2), 16, dtype=np.uint8))            # not a 4-bit code


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

def _reversed_nibbles_rows(words):
    u = O._as_u32(words)
    out = np.empty((u.shape[0] * 8, u.shape[1]), dtype=np.uint8)
    for j in range(8):
        out[j::8] = (u >> np.uint32(4 * (7 - j))) & np.uint32(0xF)
    return out


def _transposed_zero_unpack(words):
    u = O._as_u32(words)
    out = np.empty((u.shape[0], u.shape[1] * 8), dtype=np.uint8)
    for j in range(8):       # column-major nibble placement: wrong order within a word
        out[:, j * u.shape[1]:(j + 1) * u.shape[1]] = (u >> np.uint32(4 * j)) & np.uint32(0xF)
    return out


def _dequant_wrong_group(qweight, scales, qzeros, g, act, k0=0, k1=None, cols=None):
    K = qweight.shape[0] * 8
    k1 = K if k1 is None else k1
    q = O.unpack_rows(qweight[k0 // 8:k1 // 8])
    z = O._zero_points(qzeros, K // g, qweight.shape[1])
    s = O.widen(scales, act)
    grp = np.arange(k0, k1) % (K // g)          # k % groups instead of k // g
    if cols is not None:
        q, z, s = q[:, cols], z[:, cols], s[:, cols]
    return (q.astype(np.float64) - z[grp]) * s[grp]


def _dequant_no_zero(qweight, scales, qzeros, g, act, k0=0, k1=None, cols=None):
    K = qweight.shape[0] * 8
    k1 = K if k1 is None else k1
    q = O.unpack_rows(qweight[k0 // 8:k1 // 8])
    s = O.widen(scales, act)
    grp = np.arange(k0, k1) // g
    if cols is not None:
        q, s = q[:, cols], s[:, cols]
    return q.astype(np.float64) * s[grp]


def _dequant_sign_flip(qweight, scales, qzeros, g, act, k0=0, k1=None, cols=None):
    K = qweight.shape[0] * 8
    k1 = K if k1 is None else k1
    q = O.unpack_rows(qweight[k0 // 8:k1 // 8])
    z = O._zero_points(qzeros, K // g, qweight.shape[1])
    s = O.widen(scales, act)
    grp = np.arange(k0, k1) // g
    if cols is not None:
        q, z, s = q[:, cols], z[:, cols], s[:, cols]
    return (z[grp].astype(np.float64) - q) * s[grp]


def _pack_cols_reversed(codes):
    R, C = codes.shape
    acc = np.zeros((R, C // 8), dtype=np.uint32)
    for j in range(8):
        acc |= codes[:, j::8].astype(np.uint32) << np.uint32(4 * (7 - j))
    return acc.view(np.int32)


def _unpack_cols_reversed(words):
    u = O._as_u32(words)
    out = np.empty((u.shape[0], u.shape[1] * 8), dtype=np.uint8)
    for j in range(8):
        out[:, j::8] = (u >> np.uint32(4 * (7 - j))) & np.uint32(0xF)
    return out


def _signed_shift_unpack_rows(words):
    w = np.ascontiguousarray(words).view(np.int32).astype(np.int64)
    out = np.empty((w.shape[0] * 8, w.shape[1]), dtype=np.uint8)
    for j in range(8):
        v = w >> (4 * j)
        out[j::8] = np.clip(v, 0, 15)                 # sign-extends instead of masking
    return out


def _widen_bf16_as_f16(a, act):
    return np.asarray(a).astype(np.float64) if act == "bf16" else np.asarray(a, np.float16).astype(np.float64)


MUTATIONS = {
    "weight nibble order reversed": ("unpack_rows", _reversed_nibbles_rows),
    "zero-point nibbles placed column-major": ("unpack_cols", _transposed_zero_unpack),
    "group index k % groups": ("dequantize", _dequant_wrong_group),
    "zero-point dropped": ("dequantize", _dequant_no_zero),
    "sign of (q - z) flipped": ("dequantize", _dequant_sign_flip),
    "pack and unpack of zero-points both reversed": (("pack_cols", "unpack_cols"),
                                                     (_pack_cols_reversed, _unpack_cols_reversed)),
    "arithmetic shift without mask": ("unpack_rows", _signed_shift_unpack_rows),
    "bf16 bits read as integers": ("widen", _widen_bf16_as_f16),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attrs, fns = MUTATIONS[name]
    if isinstance(attrs, str):
        attrs, fns = (attrs,), (fns,)
    for a, f in zip(attrs, fns):
        monkeypatch.setattr(O, a, f)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches: {name}"
