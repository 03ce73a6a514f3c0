"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each pin returns None when it holds and raises AssertionError otherwise, so the
same pins serve the oracle tests and the planted-mistake tests (which patch a
mistake into the oracle and expect at least one pin to fail).

Sources of truth used here, none of which is the oracle's own code:
  * exact rational arithmetic (fractions.Fraction) with nibbles extracted by
    integer division, on tiny shapes -- the layer's definition
        y[m,n] = sum_k x[m,k] (q[k,n] - z[k//g,n]) s[k//g,n]
    evaluated with no rounding at all;
  * the unpacked codes drawn by the input generator (before any packing);
  * closed forms: q == z gives 0; a one-hot x selects one dequantised weight
    row; y is linear in x; the symmetric layer equals the asymmetric one with
    every zero-point at 8; constant (q - z) and s give c * s * sum_k x.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from oracle import w4a16_oracle as O
from w4a16_inputs import make_case


def _fr(v):
    return Fraction(float(v))


def packed_operands(case):
    qw = O.pack_rows(case.q)
    qz = None if case.z is None else O.pack_cols(case.z)
    return qw, qz


def exact_layer(case):
    """Exact rational y from the generator's unpacked codes (no packing involved)."""
    x = O.widen(case.x, case.act)
    s = O.widen(case.s, case.act)
    M, K, N, g = case.M, case.K, case.N, case.g
    y = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        col = []
        for k in range(K):
            q = int(case.q[k, n])
            z = 8 if case.z is None else int(case.z[k // g, n])
            col.append((q - z) * _fr(s[k // g, n]))
        for m in range(M):
            y[m][n] = sum((_fr(x[m, k]) * col[k] for k in range(K)), Fraction(0))
    return y


def _golden_rows():
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pack_words.txt")
    out = []
    for line in open(path):
        line = line.split("#", 1)[0].split()
        if line:
            out.append((line[0], [int(v) for v in line[1:9]], int(line[9], 16)))
    return out


def pin_pack_golden():
    """Hand-worked words: least significant nibble first, along N for zero-points
    and along K for weights."""
    for kind, codes, word in _golden_rows():
        c = np.array(codes, dtype=np.uint8)
        if kind == "cols":
            got = O.pack_cols(c.reshape(1, 8))[0, 0]
            back = O.unpack_cols(np.array([[word]], dtype=np.uint32).view(np.int32))[0]
        else:
            got = O.pack_rows(c.reshape(8, 1))[0, 0]
            back = O.unpack_rows(np.array([[word]], dtype=np.uint32).view(np.int32))[:, 0]
        assert int(got) % (1 << 32) == word, (kind, codes, hex(int(got) % (1 << 32)))
        assert np.array_equal(back, c), (kind, codes, back)


def pin_unpack_divmod():
    """Unpacking equals nibble extraction by integer division on random words,
    including words with the top bit set (negative as int32)."""
    rng = np.random.default_rng(1)
    words = rng.integers(0, 1 << 32, size=(6, 5), dtype=np.uint64).astype(np.uint32)
    words[0, 0] = 0xFFFFFFFF
    words[0, 1] = 0x80000000
    w32 = words.view(np.int32)
    rows = O.unpack_rows(w32)
    cols = O.unpack_cols(w32)
    for i in range(6):
        for j in range(5):
            for t in range(8):
                nib = (int(words[i, j]) // 16 ** t) % 16
                assert rows[8 * i + t, j] == nib
                assert cols[i, 8 * j + t] == nib


def pin_bruteforce(shapes=((1, 8, 32, 8), (3, 16, 64, 32), (2, 8, 64, 16)),
                   acts=("f16", "bf16"), scales=("uniform", "signed")):
    for (M, N, K, g) in shapes:
        for act in acts:
            for sym in (False, True):
                for sm in scales:
                    case = make_case(M, N, K, g, act, sym, seed=M * 1000 + N + K + g, scales=sm)
                    qw, qz = packed_operands(case)
                    got = O.reference(case.x, qw, case.s, qz, g, act, k_block=16)
                    want = exact_layer(case)
                    for m in range(M):
                        for n in range(N):
                            w = float(want[m][n])
                            assert abs(got[m, n] - w) <= 1e-12 * max(1.0, abs(w)), \
                                (M, N, K, g, act, sym, sm, m, n, got[m, n], w)


def pin_q_equals_z():
    for act in ("f16", "bf16"):
        case = make_case(3, 24, 96, 32, act, False, seed=7)
        case.q = np.repeat(case.z, case.g, axis=0)          # q[k, n] = z[k // g, n]
        qw, qz = packed_operands(case)
        y = O.reference(case.x, qw, case.s, qz, case.g, act)
        assert np.all(y == 0.0), np.abs(y).max()
        # symmetric layer: every code equal to 8
        case.q[:] = 8
        y = O.reference(case.x, O.pack_rows(case.q), case.s, None, case.g, act)
        assert np.all(y == 0.0)


def pin_onehot():
    for act in ("f16", "bf16"):
        for sym in (False, True):
            case = make_case(1, 16, 64, 16, act, sym, seed=11)
            qw, qz = packed_operands(case)
            s = O.widen(case.s, act)
            for k in (0, 1, 7, 8, 15, 16, 33, 63):
                x = np.zeros((1, case.K), dtype=np.float64)
                x[0, k] = 1.0
                xa = x.astype(np.float16) if act == "f16" else \
                    (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
                y = O.reference(xa, qw, case.s, qz, case.g, act)
                z = np.full(case.N, 8) if sym else case.z[k // case.g].astype(np.int64)
                want = (case.q[k].astype(np.int64) - z) * s[k // case.g]
                assert np.array_equal(y[0], want), (act, sym, k)


def pin_linearity():
    """y(a x1 + b x2) = a y(x1) + b y(x2); x1, x2 small integers so every sum is exact."""
    for act in ("f16", "bf16"):
        case = make_case(2, 16, 128, 32, act, False, seed=5)
        qw, qz = packed_operands(case)
        rng = np.random.default_rng(9)
        x1 = rng.integers(-8, 9, size=(2, 128)).astype(np.float64)
        x2 = rng.integers(-8, 9, size=(2, 128)).astype(np.float64)

        def y_of(xf):
            xa = xf.astype(np.float16) if act == "f16" else \
                (xf.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
            return O.reference(xa, qw, case.s, qz, 32, act)

        y1, y2 = y_of(x1), y_of(x2)
        for a, b in ((1, 1), (2, -3), (0, 1), (-1, 0)):
            y = y_of(a * x1 + b * x2)
            assert np.allclose(y, a * y1 + b * y2, rtol=1e-12, atol=1e-12), (act, a, b)


def pin_symmetric_is_z8():
    for act in ("f16", "bf16"):
        case = make_case(3, 32, 128, 32, act, True, seed=3)
        qw = O.pack_rows(case.q)
        y_sym = O.reference(case.x, qw, case.s, None, 32, act)
        z8 = np.full((case.K // 32, case.N), 8, dtype=np.uint8)
        y_asym = O.reference(case.x, qw, case.s, O.pack_cols(z8), 32, act)
        assert np.array_equal(y_sym, y_asym)


def pin_constant_weight():
    for (c_q, c_z) in ((11, 4), (0, 15), (15, 0), (3, 3)):
        case = make_case(2, 8, 64, 32, "bf16", False, seed=c_q)
        case.q[:] = c_q
        case.z[:] = c_z
        sigma_bits = np.uint16(0x3C00)  # bf16 0.0078125
        case.s[:] = sigma_bits
        qw, qz = packed_operands(case)
        y = O.reference(case.x, qw, case.s, qz, 32, "bf16")
        x = O.widen(case.x, "bf16")
        want = (c_q - c_z) * 0.0078125 * x.sum(axis=1, keepdims=True)
        assert np.allclose(y, np.broadcast_to(want, y.shape), rtol=1e-12, atol=1e-13)


def pin_group_boundaries():
    """Scales that change at every group: y on a one-hot x just before and just
    after each group boundary must pick the scale of its own group."""
    case = make_case(1, 8, 128, 32, "f16", False, seed=21)
    case.q[:] = 9
    case.z[:] = 1
    for t in range(case.K // 32):
        case.s[t, :] = np.float16(2.0 ** -t)
    qw, qz = packed_operands(case)
    for k in (31, 32, 63, 64, 95, 96, 127):
        x = np.zeros((1, 128), dtype=np.float16)
        x[0, k] = 1
        y = O.reference(x, qw, case.s, qz, 32, "f16")
        assert np.all(y == 8 * 2.0 ** -(k // 32)), (k, y)


ALL_PINS = [pin_pack_golden, pin_unpack_divmod, pin_bruteforce, pin_q_equals_z, pin_onehot, pin_linearity, pin_symmetric_is_z8,
            pin_constant_weight, pin_group_boundaries]
