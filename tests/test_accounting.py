"""The byte accounting used for the roofline reproduces the figures printed on
"Keep W4A16 zero-points packed at 4 bits instead of expanding to 2 bytes"."""
import pytest

from weight_only_int4_gb300.accounting import (expanded_zero_bytes, layer_bytes, layer_flops, mx_dequant_bytes,
                                                mx_layer_bytes)


def _rows(golden):
    for key, M, N, K, g, v in golden("p1_byte_counts.txt"):
        yield key, int(M), int(N), int(K), int(g), float(v)


def test_printed_byte_counts(golden):
    seen = set()
    for key, M, N, K, g, v in _rows(golden):
        b = layer_bytes(M, N, K, g, symmetric=False, act="f16")
        zexp = expanded_zero_bytes(N, K, g, "f16")
        if key == "weights_MB":
            assert round(b.weights / 1e6, 1) == v
        elif key == "zexp_MB":
            assert round(zexp / 1e6, 1) == v
        elif key == "zpk_MB":
            assert round(b.zeros / 1e6, 1) == v
        elif key == "reduction_pct":
            before = b.weights + b.scales + zexp
            after = b.operands
            assert round(100.0 * (after - before) / before, 1) == v
        elif key == "saving_pct":
            before = b.total - b.zeros + zexp
            assert round(100.0 * (before - b.total) / before, 1) == v
        elif key == "gibs_band":
            gibs = b.operands / (v * 1e-6) / 2 ** 30
            assert 186.0 <= gibs <= 205.0, gibs
        else:
            pytest.fail(f"unknown golden key {key}")
        seen.add(key)
    assert seen == {"weights_MB", "zexp_MB", "zpk_MB", "reduction_pct", "saving_pct", "gibs_band"}


def test_symmetric_has_no_zero_bytes():
    b = layer_bytes(1, 16384, 5376, 32, symmetric=True, act="bf16")
    assert b.zeros == 0
    assert b.total == 16384 * 5376 // 2 + 168 * 16384 * 2 + 5376 * 2 + 16384 * 2


def test_flops():
    assert layer_flops(2048, 43008, 5376) == 947_040_288_768


def test_mxfp4_bytes():
    b = mx_layer_bytes(1, 43008, 5376)
    assert b.weights == 43008 * 5376 // 2 and b.scales == 168 * 43008 and b.zeros == 0
    assert b.total == 43008 * 5376 // 2 + 168 * 43008 + 5376 * 2 + 43008 * 2
    d = mx_dequant_bytes(43008, 5376)
    assert d.x == 0 and d.y == 43008 * 5376 * 2 and d.operands == b.operands
