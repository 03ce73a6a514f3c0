"""Seeded synthetic inputs for the W4A16 group-quantized linear layer.

This module is shared by the tests, the benchmark and the CPU oracle. It only
draws random numbers and stores them in the operand dtypes; it holds none of
the layer's arithmetic (no packing, no dequantisation, no matmul). Both the
CUDA path and the oracle pack the unpacked 4-bit codes drawn here with their
own, independent packers. At the largest sizes the packed words themselves are
drawn instead (on the device): a uniformly random 32-bit word is eight
independent uniform codes, so neither side packs anything.

Value distributions follow the decode and prefill workloads of "Keep W4A16
zero-points packed at 4 bits instead of expanding to 2 bytes" (§Problem,
§Results, §Known regression): activations x ~ N(0, 1), 4-bit weight codes and
zero-points uniform on 0..15, scales uniform on [0.002, 0.02]. The optional
"signed" scale mode follows the lesson of "qsa_prompt_attn: Q4_0 KV on tensor
cores" (§What, §Measured "A bug the tests caught"): scales of both signs
spread over two decades.

Generation order is fixed (x, q, s, z) on one numpy PCG64 stream per seed, so
a case is reproducible on any host.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

__all__ = [
    "ACT_DTYPES",
    "Case",
    "MxCase",
    "MX_WORKLOADS",
    "make_mx_case",
    "Workload",
    "WORKLOADS",
    "f32_to_act",
    "make_case",
    "make_case_for",
    "LargeCase",
    "make_large_case",
    "make_large_mx_case",
    "device_codes",
]

ACT_DTYPES = ("f16", "bf16")


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return raw uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + (((u >> 16) & 1) + 0x7FFF)
    return (u >> 16).astype(np.uint16)


def f32_to_act(a: np.ndarray, act: str) -> np.ndarray:
    """Store float32 draws in the activation dtype.

    f16 -> numpy float16 array; bf16 -> numpy uint16 array of bfloat16 bit
    patterns (numpy has no bfloat16 type).
    """
    if act == "f16":
        return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16)
    if act == "bf16":
        return _f32_to_bf16_bits(a)
    raise ValueError(f"unknown activation dtype {act!r}")


@dataclass
class Case:
    """One seeded problem, unpacked.

    x  : [M, K] activations in `act` (float16, or uint16 bf16 bit patterns)
    q  : [K, N] uint8 4-bit weight codes, values 0..15
    s  : [K/g, N] scales in `act`
    z  : [K/g, N] uint8 zero-points 0..15, or None for the symmetric layer
    """

    M: int
    N: int
    K: int
    g: int
    act: str
    x: np.ndarray
    q: np.ndarray
    s: np.ndarray
    z: Optional[np.ndarray]

    @property
    def symmetric(self) -> bool:
        return self.z is None


def make_case(M: int, N: int, K: int, g: int, act: str = "f16", symmetric: bool = False,
              seed: int = 0, scales: str = "uniform", x_dist: str = "normal") -> Case:
    """Draw one case. `scales` is "uniform" (U[0.002, 0.02]) or "signed"
    (random sign, magnitude log-uniform over [0.002, 0.2]). `x_dist` is
    "normal" (N(0, 1)), or one of two skewed, mostly positive activation
    shapes such as a SiLU or GELU output has: "offset" (4 + N(0, 1)) and
    "halfnormal" (3 |N(0, 1)|). All three take the same draws from the stream."""
    if act not in ACT_DTYPES:
        raise ValueError(f"unknown activation dtype {act!r}")
    if M < 0 or N < 0 or K < 0 or g <= 0 or K % g:
        raise ValueError(f"bad shape M={M} N={N} K={K} g={g}")
    rng = np.random.Generator(np.random.PCG64(seed))
    x32 = rng.standard_normal((M, K), dtype=np.float32)
    if x_dist == "offset":
        x32 = x32 + np.float32(4.0)
    elif x_dist == "halfnormal":
        x32 = np.abs(x32) * np.float32(3.0)
    elif x_dist != "normal":
        raise ValueError(f"unknown activation distribution {x_dist!r}")
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    if scales == "uniform":
        s32 = (np.float32(0.002) + np.float32(0.018) * rng.random((K // g, N), dtype=np.float32))
    elif scales == "signed":
        mag = np.power(10.0, rng.uniform(np.log10(0.002), np.log10(0.2), size=(K // g, N)))
        sign = np.where(rng.random((K // g, N)) < 0.5, -1.0, 1.0)
        s32 = (mag * sign).astype(np.float32)
    else:
        raise ValueError(f"unknown scale mode {scales!r}")
    z = None if symmetric else rng.integers(0, 16, size=(K // g, N), dtype=np.uint8)
    return Case(M=M, N=N, K=K, g=g, act=act, x=f32_to_act(x32, act), q=q,
                s=f32_to_act(s32, act), z=z)


@dataclass(frozen=True)
class Workload:
    """A named problem shape. `kernel` is the entry point that serves it."""

    name: str
    kernel: str  # "gemv", "gemm" or "dequant"
    M: int
    N: int
    K: int
    g: int
    act: str
    symmetric: bool

    def case(self, seed: int = 0) -> Case:
        return make_case(self.M, self.N, self.K, self.g, self.act, self.symmetric, seed)


def _w(name, kernel, M, N, K, g, act, sym):
    return Workload(name, kernel, M, N, K, g, act, sym)


# The decode and prefill shapes of the W4A16 pages (M x N x K, group g).
WORKLOADS = {w.name: w for w in [
    # small square decode GEMV, g=128, fp16, asymmetric
    _w("gemv_1x2048x2048_g128_f16_asym", "gemv", 1, 2048, 2048, 128, "f16", False),
    # gate_up-like decode GEMV (~116 MB of int4 weights), g=32, fp16, asymmetric
    _w("gemv_1x43008x5376_g32_f16_asym", "gemv", 1, 43008, 5376, 32, "f16", False),
    # batch-4 g=128 asymmetric sweep, fp16 and bf16
    *[_w(f"gemv_4x{N}x{K}_g128_{a}_asym", "gemv", 4, N, K, 128, a, False)
      for a in ("f16", "bf16")
      for (N, K) in ((2048, 2048), (2048, 2560), (6144, 2048), (4096, 2048))],
    # several decode rows on the gate_up shape (the GEMV's tensor-core MMA conversion)
    _w("gemv_4x43008x5376_g32_f16_asym", "gemv", 4, 43008, 5376, 32, "f16", False),
    _w("gemv_16x43008x5376_g32_bf16_asym", "gemv", 16, 43008, 5376, 32, "bf16", False),
    # qkv-like and down-like decode GEMV, g=32, bf16, symmetric and asymmetric
    *[_w(f"gemv_1x{N}x{K}_g32_bf16_{'sym' if s else 'asym'}", "gemv", 1, N, K, 32, "bf16", s)
      for (N, K) in ((16384, 5376), (5376, 21504)) for s in (True, False)],
    # prefill GEMM on the gate_up shape, g=32, bf16 in/out
    _w("gemm_2048x43008x5376_g32_bf16_asym", "gemm", 2048, 43008, 5376, 32, "bf16", False),
    # the same prefill shape in fp16, and with g=128
    _w("gemm_2048x43008x5376_g32_f16_asym", "gemm", 2048, 43008, 5376, 32, "f16", False),
    _w("gemm_2048x43008x5376_g128_bf16_asym", "gemm", 2048, 43008, 5376, 128, "bf16", False),
    # mid-M prefill chunks on the same weights
    _w("gemm_64x43008x5376_g32_bf16_asym", "gemm", 64, 43008, 5376, 32, "bf16", False),
    _w("gemm_256x43008x5376_g32_bf16_asym", "gemm", 256, 43008, 5376, 32, "bf16", False),
    # dense dequantised copy of the gate_up weights (M is unused)
    _w("dequant_43008x5376_g32_f16_asym", "dequant", 1, 43008, 5376, 32, "f16", False),
    _w("dequant_43008x5376_g32_bf16_asym", "dequant", 1, 43008, 5376, 32, "bf16", False),
]}


def make_case_for(name: str, seed: int = 0) -> Case:
    return WORKLOADS[name].case(seed)


# ---------------------------------------------------------------------------
# MXFP4 weights (E2M1 codes with one E8M0 byte per 32 K rows of a column)
# ---------------------------------------------------------------------------
# "Add BF16xFP4 MoE GEMM stage1 kernel" (section "Technical Details") keeps bf16
# activations and stores weights as E2M1 codes with E8M0 block scales. Codes
# are uniform on 0..15 (every value of the format, both signs). Exponent
# bytes: "typical" draws e uniformly on 118..125, i.e. block scales
# 2^-9..2^-2 and weights of magnitude up to 1.5, the range of trained layer
# weights; "wide" draws 96..160, so blocks with e > 128 (scales above 2) occur.


@dataclass
class MxCase:
    """One seeded MXFP4 problem, unpacked.

    x : [M, K] bf16 bit patterns (uint16)
    q : [K, N] uint8 E2M1 codes, values 0..15
    e : [K/32, N] uint8 E8M0 exponent bytes
    """

    M: int
    N: int
    K: int
    x: np.ndarray
    q: np.ndarray
    e: np.ndarray


_MX_EXPONENTS = {"typical": (118, 125), "wide": (96, 160)}


def make_mx_case(M: int, N: int, K: int, seed: int = 0, exponents: str = "typical") -> MxCase:
    if M < 0 or N < 0 or K < 0 or K % 32:
        raise ValueError(f"bad MXFP4 shape M={M} N={N} K={K}")
    lo, hi = _MX_EXPONENTS[exponents]
    rng = np.random.Generator(np.random.PCG64(seed))
    x32 = rng.standard_normal((M, K), dtype=np.float32)
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    e = rng.integers(lo, hi + 1, size=(K // 32, N), dtype=np.uint8)
    return MxCase(M=M, N=N, K=K, x=f32_to_act(x32, "bf16"), q=q, e=e)


@dataclass(frozen=True)
class MxWorkload:
    """A named MXFP4 problem shape; `kernel` is "gemv", "gemm" or "dequant"."""

    name: str
    kernel: str
    M: int
    N: int
    K: int

    def case(self, seed: int = 0) -> MxCase:
        return make_mx_case(self.M, self.N, self.K, seed)


# The gate_up layer shape of the W4A16 workloads, with MXFP4 weights.
MX_WORKLOADS = {w.name: w for w in [
    MxWorkload("mx_gemv_1x43008x5376_bf16", "gemv", 1, 43008, 5376),
    MxWorkload("mx_gemm_2048x43008x5376_bf16", "gemm", 2048, 43008, 5376),
    MxWorkload("mx_gemm_64x43008x5376_bf16", "gemm", 64, 43008, 5376),
    MxWorkload("mx_dequant_43008x5376_bf16", "dequant", 1, 43008, 5376),
]}


# ---------------------------------------------------------------------------
# Cases at the largest sizes: weights drawn as packed words on the device
# ---------------------------------------------------------------------------
def _device_generator(seed: int, device):
    import torch
    return torch.Generator(device=device).manual_seed(seed)


def device_words(shape, seed: int, device="cuda"):
    """Uniformly random 32-bit words (torch.int32) drawn on `device` by torch's
    seeded generator. A uniform word holds eight independent codes uniform on
    0..15 whichever nibble order reads it, so packed operands of any size can be
    drawn without packing anything."""
    import torch
    return torch.randint(-2 ** 31, 2 ** 31, tuple(shape), dtype=torch.int32, device=device,
                         generator=_device_generator(seed, device))


def device_codes(shape, seed: int, device="cuda"):
    """Codes uniform on 0..15 (torch.uint8) drawn on `device`."""
    import torch
    return torch.randint(0, 16, tuple(shape), dtype=torch.uint8, device=device,
                         generator=_device_generator(seed, device))


@dataclass
class LargeCase:
    """A problem too large to draw code by code on the host.

    x  : [M, K] activations in `act` (host)
    s  : [K/g, N] scales in `act` (host); for MXFP4, E8M0 bytes [K/32, N]
    zw : [K/g, N/8] uint32 zero-point words (host; eight codes each), or None
    qw : [K/8, N] int32 weight words on the device (eight codes each)
    """

    M: int
    N: int
    K: int
    g: int
    act: str
    x: np.ndarray
    s: np.ndarray
    zw: Optional[np.ndarray]
    qw: object


def make_large_case(M: int, N: int, K: int, g: int, act: str = "bf16", symmetric: bool = False,
                    seed: int = 0, device="cuda") -> LargeCase:
    """Same distributions as make_case (x ~ N(0, 1), codes and zero-points
    uniform on 0..15, scales uniform on [0.002, 0.02]); x, s and the zero-point
    words from one numpy PCG64 stream, the weight words on the device."""
    if act not in ACT_DTYPES or M < 0 or N < 8 or N % 8 or K < g or K % g or K % 8:
        raise ValueError(f"bad shape M={M} N={N} K={K} g={g} act={act}")
    rng = np.random.Generator(np.random.PCG64(seed))
    x32 = rng.standard_normal((M, K), dtype=np.float32)
    s32 = np.float32(0.002) + np.float32(0.018) * rng.random((K // g, N), dtype=np.float32)
    zw = None if symmetric else rng.integers(0, 2 ** 32, size=(K // g, N // 8), dtype=np.uint32)
    return LargeCase(M=M, N=N, K=K, g=g, act=act, x=f32_to_act(x32, act), s=f32_to_act(s32, act), zw=zw,
                     qw=device_words((K // 8, N), seed + 1, device))


def make_large_mx_case(M: int, N: int, K: int, seed: int = 0, device="cuda") -> LargeCase:
    """MXFP4 counterpart: bf16 x ~ N(0, 1), E2M1 codes uniform, exponent bytes
    uniform on 118..125 ("typical")."""
    if M < 0 or N < 16 or N % 16 or K < 32 or K % 32:
        raise ValueError(f"bad MXFP4 shape M={M} N={N} K={K}")
    lo, hi = _MX_EXPONENTS["typical"]
    rng = np.random.Generator(np.random.PCG64(seed))
    x32 = rng.standard_normal((M, K), dtype=np.float32)
    e = rng.integers(lo, hi + 1, size=(K // 32, N), dtype=np.uint8)
    return LargeCase(M=M, N=N, K=K, g=32, act="bf16", x=f32_to_act(x32, "bf16"), s=e, zw=None,
                     qw=device_words((K // 8, N), seed + 1, device))
