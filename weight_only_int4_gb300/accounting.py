"""Algorithmic byte and FLOP counts of one W4A16 layer call.

The byte count is what the layer must move at minimum: packed 4-bit weights,
one scale per (group, column), packed 4-bit zero-points, the activations and
the output. This is the convention of "Keep W4A16 zero-points packed at 4 bits
instead of expanding to 2 bytes" (§Problem: weights + scale + zero-point
bytes streamed per call), extended by the x and y bytes. Expanded zero-points
(one activation-dtype value per group and column, the layout that page
replaces) are counted only by `expanded_zero_bytes`, never in the roofline.
"""
from __future__ import annotations

from dataclasses import dataclass

ACT_BYTES = {"f16": 2, "bf16": 2}


@dataclass(frozen=True)
class LayerBytes:
    weights: int
    scales: int
    zeros: int
    x: int
    y: int

    @property
    def operands(self) -> int:
        """weights + scales + packed zero-points (what the decode kernel streams)."""
        return self.weights + self.scales + self.zeros

    @property
    def total(self) -> int:
        return self.operands + self.x + self.y


def layer_bytes(M: int, N: int, K: int, g: int, symmetric: bool = False, act: str = "f16") -> LayerBytes:
    a = ACT_BYTES[act]
    groups = K // g
    return LayerBytes(
        weights=K * N // 2,
        scales=groups * N * a,
        zeros=0 if symmetric else groups * N // 2,
        x=M * K * a,
        y=M * N * a,
    )


def dequant_bytes(N: int, K: int, g: int, symmetric: bool = False, act: str = "f16") -> LayerBytes:
    """The dense dequantised copy: reads the packed operands once, writes K x N
    activation-dtype values (counted as y; no x)."""
    b = layer_bytes(1, N, K, g, symmetric, act)
    return LayerBytes(weights=b.weights, scales=b.scales, zeros=b.zeros, x=0, y=K * N * ACT_BYTES[act])


def expanded_zero_bytes(N: int, K: int, g: int, act: str = "f16") -> int:
    """Bytes of zero-points stored one activation-dtype value per (group, column)."""
    return (K // g) * N * ACT_BYTES[act]


def mx_layer_bytes(M: int, N: int, K: int) -> LayerBytes:
    """MXFP4 weights ("Add BF16xFP4 MoE GEMM stage1 kernel", section
    "Technical Details"): 4-bit codes, one E8M0 byte per 32 K rows of a
    column, no zero-points; bf16 x and y."""
    return LayerBytes(weights=K * N // 2, scales=(K // 32) * N, zeros=0, x=M * K * 2, y=M * N * 2)


def mx_dequant_bytes(N: int, K: int) -> LayerBytes:
    """The dense bf16 copy of MXFP4 weights: reads codes and exponents once, writes K x N bf16."""
    b = mx_layer_bytes(1, N, K)
    return LayerBytes(weights=b.weights, scales=b.scales, zeros=0, x=0, y=K * N * 2)


def layer_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
