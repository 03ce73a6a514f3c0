"""Pins for the MXFP4 oracle: checks against facts fixed outside the oracle.

Each pin returns None when it holds and raises AssertionError otherwise, so the
pins serve both the oracle tests and the planted-mistake tests.

Sources of truth, none of which is the oracle's own code:
  * the value table of FP4 E2M1 (1 sign, 2 exponent and 1 mantissa bit,
    exponent bias 1, no infinities or NaN), written out as literals: the eight
    magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, and their negatives for codes 8..15;
  * PyTorch's own decoder of the E8M0 type (torch.float8_e8m0fnu), which
    yields 2^(e - 127), 2^-127 for byte 0 and NaN for byte 255;
  * the construction of "Add BF16xFP4 MoE GEMM stage1 kernel" (section
    "Technical Details"): the E8M0 byte shifted left by 23 bits, read as an
    FP32 bit pattern, is the scale 2^(e - 127);
  * exact rational arithmetic (fractions.Fraction) over the generator's
    unpacked codes on tiny shapes -- no packing, no FP64 summation;
  * closed forms: a one-hot x selects one weight row; all-ones x over
    constant codes gives 32 * value * sum_b 2^(e_b - 127) per column.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

from oracle import mxfp4_oracle as X
from oracle import w4a16_oracle as O
from w4a16_inputs import make_mx_case

# FP4 E2M1 value of each code 0..15 (sign bit 3)
E2M1_TABLE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0)


def _table_fraction(code: int) -> Fraction:
    return Fraction(E2M1_TABLE[code])


def _scale_fraction(e: int) -> Fraction:
    return Fraction(2) ** (int(e) - 127)


def pin_e2m1_table():
    got = X.e2m1_decode(np.arange(16))
    want = np.array(E2M1_TABLE)
    assert np.array_equal(got, want), f"E2M1 decode {got} != table {want}"
    assert np.array_equal(np.signbit(got), np.signbit(want)), "E2M1 sign of zero codes"


def pin_e8m0_torch():
    e = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(e.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = X.e8m0_decode(e)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "E8M0 NaN positions"
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "E8M0 values differ from torch.float8_e8m0fnu"


def pin_e8m0_shift23():
    e = np.arange(1, 255, dtype=np.uint32)
    via_bits = (e << np.uint32(23)).view(np.float32).astype(np.float64)
    assert np.array_equal(X.e8m0_decode(e), via_bits), "E8M0 differs from the FP32 exponent-field construction"


def exact_mx_layer(case):
    """Exact rational y from the generator's unpacked codes and exponent bytes."""
    x = O.widen(case.x, "bf16")
    y = []
    for m in range(case.M):
        row = []
        for n in range(case.N):
            acc = Fraction(0)
            for k in range(case.K):
                w = _table_fraction(int(case.q[k, n])) * _scale_fraction(case.e[k // 32, n])
                acc += Fraction(float(x[m, k])) * w
            row.append(acc)
        y.append(row)
    return y


def pin_mx_bruteforce(shapes=((1, 8, 32), (3, 16, 64), (2, 8, 96)), seeds=(0, 1)):
    for (M, N, K) in shapes:
        for seed in seeds:
            for mode in ("typical", "wide"):
                case = make_mx_case(M, N, K, seed, mode)
                got = X.reference_mx(case.x, O.pack_rows(case.q), case.e)
                want = exact_mx_layer(case)
                for m in range(M):
                    for n in range(N):
                        w = float(want[m][n])
                        assert abs(got[m, n] - w) <= 1e-12 * max(1.0, abs(w)), \
                            f"MX brute force {M}x{N}x{K} seed {seed} {mode}: y[{m},{n}] {got[m, n]} != {w}"


def pin_mx_onehot():
    case = make_mx_case(0, 16, 96, 3, "wide")
    qw = O.pack_rows(case.q)
    for k in (0, 7, 31, 32, 63, 95):
        x = np.zeros((1, case.K), dtype=np.uint16)
        x[0, k] = 0x3F80                            # bf16 1.0
        y = X.reference_mx(x, qw, case.e)[0]
        want = [float(_table_fraction(int(case.q[k, n])) * _scale_fraction(case.e[k // 32, n]))
                for n in range(case.N)]
        assert np.array_equal(y, np.array(want)), f"one-hot row {k}"


def pin_mx_block_sums():
    rng = np.random.Generator(np.random.PCG64(11))
    K, N = 128, 8
    for code in (1, 3, 7, 9, 14):
        q = np.full((K, N), code, dtype=np.uint8)
        e = rng.integers(110, 140, size=(K // 32, N), dtype=np.uint8)
        x = np.full((1, K), 0x3F80, dtype=np.uint16)
        y = X.reference_mx(x, O.pack_rows(q), e)[0]
        for n in range(N):
            want = 32 * _table_fraction(code) * sum(_scale_fraction(e[b, n]) for b in range(K // 32))
            assert y[n] == float(want), f"block sum code {code} column {n}: {y[n]} != {float(want)}"


def pin_mx_weight_range():
    # byte 254 with code 7 exceeds bf16 (6 * 2^127 >= 2^128): +inf; byte 0 with
    # code 1 is the bf16 subnormal 2^-128; byte 255 gives NaN
    q = np.array([[7, 1, 15, 2, 0, 8, 3, 9]] * 32, dtype=np.uint8)
    e = np.array([[254, 0, 254, 255, 255, 128, 0, 1]], dtype=np.uint8)
    w = X.dequantize_mx(O.pack_rows(q), e)[0]
    assert w[0] == np.inf and w[2] == -np.inf, "overflow to +-inf"
    assert w[1] == 2.0 ** -128, "subnormal weight"
    assert np.isnan(w[3]) and np.isnan(w[4]), "byte 255 decodes to NaN"
    assert w[5] == 0.0 and np.signbit(w[5]), "code 8 is -0"
    assert w[6] == 1.5 * 2.0 ** -127 and w[7] == -0.5 * 2.0 ** -126, "small exact weights"


PINS = [pin_e2m1_table, pin_e8m0_torch, pin_e8m0_shift23, pin_mx_bruteforce, pin_mx_onehot,
        pin_mx_block_sums, pin_mx_weight_range]
