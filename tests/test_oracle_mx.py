"""CPU tests of the MXFP4 oracle against its pins (no GPU, no CUDA library)."""
from typing import Optional, Sequence

import numpy as np
import pytest

import oracle_pins_mx as P
from oracle import mxfp4_oracle as X
from oracle import w4a16_oracle as O
from w4a16_inputs import make_mx_case


@pytest.mark.parametrize("pin", P.PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_sampled_rows_and_cols_match_full():
    case = make_mx_case(5, 24, 160, 7, "wide")
    qw = O.pack_rows(case.q)
    full = X.reference_mx(case.x, qw, case.e, k_block=64)
    # same sums; the BLAS may order the FP64 additions differently for a subset
    tol = 1e-13 * np.abs(full).max()
    assert np.abs(X.reference_mx_rows(case.x, [4, 1], qw, case.e, k_block=64) - full[[4, 1]]).max() <= tol
    assert np.abs(X.reference_mx(case.x, qw, case.e, k_block=64, cols=[3, 0, 23]) - full[:, [3, 0, 23]]).max() <= tol


def test_rejects_bad_operands():
    case = make_mx_case(1, 8, 64, 0)
    qw = O.pack_rows(case.q)
    with pytest.raises(ValueError):
        X.dequantize_mx(qw, case.e[:1])            # wrong number of blocks
    with pytest.raises(ValueError):
        X.e2m1_decode(np.array([16]))
    with pytest.raises(ValueError):
        X.reference_mx(case.x[:, :32], qw, case.e)


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------
_true_e2m1 = X.e2m1_decode
_true_e8m0 = X.e8m0_decode


def _e2m1_bias0(codes):
    c = np.asarray(codes).astype(np.int64)
    E = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    v = np.where(E == 0, m / 2.0, np.ldexp(1.0 + m / 2.0, E))
    return np.where((c >> 3) & 1, -v, v)


def _e2m1_no_subnormal(codes):
    c = np.asarray(codes).astype(np.int64)
    E = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    v = np.where(E == 0, np.where(m > 0, 0.75, 0.0), np.ldexp(1.0 + m / 2.0, E - 1))
    return np.where((c >> 3) & 1, -v, v)


def _e2m1_unsigned(codes):
    return np.abs(_true_e2m1(codes))


def _e8m0_off_by_one(e):
    return _true_e8m0(e) * 2.0


def _e8m0_255_finite(e):
    b = np.asarray(e).astype(np.int64)
    return np.ldexp(1.0, b - 127)


def _dequant_block16(qweight, escale, k0=0, k1: Optional[int] = None, cols: Optional[Sequence[int]] = None):
    K = qweight.shape[0] * 8
    k1 = K if k1 is None else k1
    q = O.unpack_rows(qweight[k0 // 8:k1 // 8])
    s = X.e8m0_decode(escale)
    blk = np.minimum(np.arange(k0, k1) // 16, s.shape[0] - 1)
    if cols is not None:
        q, s = q[:, cols], s[:, cols]
    return O.round_to_act(X.e2m1_decode(q) * s[blk], "bf16")


MUTATIONS = {
    "E2M1 exponent bias 0": ("e2m1_decode", _e2m1_bias0),
    "E2M1 exponent 0 read as normal": ("e2m1_decode", _e2m1_no_subnormal),
    "E2M1 sign bit ignored": ("e2m1_decode", _e2m1_unsigned),
    "E8M0 bias 126": ("e8m0_decode", _e8m0_off_by_one),
    "E8M0 byte 255 finite": ("e8m0_decode", _e8m0_255_finite),
    "block of 16 rows": ("dequantize_mx", _dequant_block16),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(X, attr, fn)
    failed = []
    for pin in P.PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches: {name}"
