"""CPU FP64 oracle for the W4A16 group-quantized linear layer.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. The product (the CUDA library and its
Python binding) never calls it, and it shares no code with the product: it has
its own packer, its own unpacker, its own rounding and its own matmul driver.

What it computes (plain definition, no blocking beyond a K-loop that bounds
memory):

    y[m, n] = sum_k x[m, k] * (q[k, n] - z[k // g, n]) * s[k // g, n]

with, as operands,
  * qweight int32 [K/8, N]: nibble j (bits 4j..4j+3, least significant first)
    of word [w, n] holds the 4-bit weight code of row k = 8w + j;
  * qzeros int32 [K/g, N/8]: the zero-point of column n sits in word n // 8 at
    bits 4 * (n % 8) -- the packed layout of "Keep W4A16 zero-points packed at
    4 bits instead of expanding to 2 bytes" (§Change), i.e. the inverse of
    unpacking along the packed dimension;
  * symmetric layer: no qzeros, z = 8 everywhere (the "code - 8" recentring of
    "qsa_prompt_attn: Q4_0 KV on tensor cores", §What);
  * scales [K/g, N] and x [M, K] in fp16 or bf16, widened exactly to FP64.

Words are read as uint32 bit patterns with logical shifts, so words whose top
nibble is >= 8 (negative as int32) unpack correctly. (q - z) is an exact small
integer and (q - z) * s is exact in FP64; only the final sum rounds, in FP64.

Parity status of each function (what pins it is listed in the tests):
  pack_rows / pack_cols / unpack_rows / unpack_cols ... pinned
  widen ................................................. pinned
  dequantize ............................................ pinned
  reference / reference_rows / reference_cols ........... pinned
  round_to_act .......................................... pinned
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

NIBBLES_PER_WORD = 8
SYMMETRIC_ZERO = 8


# ---------------------------------------------------------------------------
# packing (the oracle's own packer, used to build oracle-side operands)
# ---------------------------------------------------------------------------

def _as_u32(words: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(words).view(np.uint32) if words.dtype == np.int32 else \
        np.ascontiguousarray(words, dtype=np.uint32)


def pack_rows(codes: np.ndarray) -> np.ndarray:
    """uint8 [R, C] (values 0..15) -> int32 [R/8, C]; nibble j of word [w, c] = codes[8w + j, c]."""
    codes = np.asarray(codes)
    R, C = codes.shape
    if R % NIBBLES_PER_WORD:
        raise ValueError("rows must be a multiple of 8")
    if codes.size and int(codes.max()) > 15:
        raise ValueError("codes must be 4-bit")
    acc = np.zeros((R // NIBBLES_PER_WORD, C), dtype=np.uint32)
    for j in range(NIBBLES_PER_WORD):
        acc |= codes[j::NIBBLES_PER_WORD, :].astype(np.uint32) << np.uint32(4 * j)
    return acc.view(np.int32)


def pack_cols(codes: np.ndarray) -> np.ndarray:
    """uint8 [R, C] -> int32 [R, C/8]; column c goes to word c // 8, bits 4 * (c % 8)."""
    codes = np.asarray(codes)
    R, C = codes.shape
    if C % NIBBLES_PER_WORD:
        raise ValueError("cols must be a multiple of 8")
    if codes.size and int(codes.max()) > 15:
        raise ValueError("codes must be 4-bit")
    acc = np.zeros((R, C // NIBBLES_PER_WORD), dtype=np.uint32)
    for j in range(NIBBLES_PER_WORD):
        acc |= codes[:, j::NIBBLES_PER_WORD].astype(np.uint32) << np.uint32(4 * j)
    return acc.view(np.int32)


def unpack_rows(words: np.ndarray) -> np.ndarray:
    """int32 [R/8, C] -> uint8 [R, C]; inverse of pack_rows."""
    u = _as_u32(words)
    W, C = u.shape
    out = np.empty((W * NIBBLES_PER_WORD, C), dtype=np.uint8)
    for j in range(NIBBLES_PER_WORD):
        out[j::NIBBLES_PER_WORD, :] = (u >> np.uint32(4 * j)) & np.uint32(0xF)
    return out


def unpack_cols(words: np.ndarray) -> np.ndarray:
    """int32 [R, C/8] -> uint8 [R, C]; row n of a packed zero-point row is word[n/8] bits 4*(n%8)."""
    u = _as_u32(words)
    R, W = u.shape
    out = np.empty((R, W * NIBBLES_PER_WORD), dtype=np.uint8)
    for j in range(NIBBLES_PER_WORD):
        out[:, j::NIBBLES_PER_WORD] = (u >> np.uint32(4 * j)) & np.uint32(0xF)
    return out


# ---------------------------------------------------------------------------
# dtypes
# ---------------------------------------------------------------------------

def widen(a: np.ndarray, act: str) -> np.ndarray:
    """Exact widening of fp16 values, or of bf16 bit patterns (uint16), to FP64."""
    if act == "f16":
        return np.asarray(a, dtype=np.float16).astype(np.float64)
    if act == "bf16":
        bits = np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(f"unknown activation dtype {act!r}")


_PRECISION = {"f16": (11, -13), "bf16": (8, -125)}   # significand bits, clamp of frexp exponent


def round_to_act(v: np.ndarray, act: str) -> np.ndarray:
    """Round FP64 values to the nearest fp16 / bf16 value (ties to even); return FP64.

    Uses v = m * 2^e (0.5 <= |m| < 1): the spacing of representable values
    around v is 2^(e - p) for p significand bits, floored at the subnormal
    spacing. Overflow gives +-inf.
    """
    p, emin = _PRECISION[act]
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    quantum = np.ldexp(1.0, np.maximum(e, emin) - p)
    r = np.rint(v / quantum) * quantum
    top = {"f16": 65504.0, "bf16": float(np.float32(3.3895313892515355e38))}[act]
    return np.where(np.abs(r) > top, np.copysign(np.inf, v), r)


# ---------------------------------------------------------------------------
# the layer
# ---------------------------------------------------------------------------

def _zero_points(qzeros: Optional[np.ndarray], groups: int, N: int) -> np.ndarray:
    if qzeros is None:
        return np.full((groups, N), SYMMETRIC_ZERO, dtype=np.uint8)
    z = unpack_cols(qzeros)
    if z.shape != (groups, N):
        raise ValueError(f"qzeros unpacks to {z.shape}, expected {(groups, N)}")
    return z


def dequantize(qweight: np.ndarray, scales: np.ndarray, qzeros: Optional[np.ndarray], g: int,
               act: str, k0: int = 0, k1: Optional[int] = None,
               cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """FP64 weight rows k0..k1 (k0, k1 multiples of 8): W[k, n] = (q[k, n] - z[k//g, n]) * s[k//g, n]."""
    K = qweight.shape[0] * NIBBLES_PER_WORD
    N = qweight.shape[1]
    if k1 is None:
        k1 = K
    if k0 % NIBBLES_PER_WORD or k1 % NIBBLES_PER_WORD:
        raise ValueError("row range must be word aligned")
    groups = K // g
    if K % g or scales.shape != (groups, N):
        raise ValueError("scales shape does not match K/g x N")
    q = unpack_rows(qweight[k0 // NIBBLES_PER_WORD:k1 // NIBBLES_PER_WORD])
    z = _zero_points(qzeros, groups, N)
    s = widen(scales, act)
    grp = np.arange(k0, k1) // g
    if cols is not None:
        cols = np.asarray(cols)
        q, z, s = q[:, cols], z[:, cols], s[:, cols]
    return (q.astype(np.float64) - z[grp].astype(np.float64)) * s[grp]


def reference(x: np.ndarray, qweight: np.ndarray, scales: np.ndarray,
              qzeros: Optional[np.ndarray], g: int, act: str, k_block: int = 1024,
              cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """FP64 y = x @ dequantize(...), summed over K in blocks of `k_block` rows.

    `cols` restricts the computation to a subset of output columns.
    """
    xd = widen(x, act)
    M, K = xd.shape
    if qweight.shape[0] * NIBBLES_PER_WORD != K:
        raise ValueError("x and qweight disagree on K")
    kb = max(NIBBLES_PER_WORD, (k_block // NIBBLES_PER_WORD) * NIBBLES_PER_WORD)
    ncols = qweight.shape[1] if cols is None else len(cols)
    y = np.zeros((M, ncols), dtype=np.float64)
    for k0 in range(0, K, kb):
        k1 = min(K, k0 + kb)
        y += xd[:, k0:k1] @ dequantize(qweight, scales, qzeros, g, act, k0, k1, cols)
    return y


def reference_rows(x: np.ndarray, rows: Sequence[int], qweight: np.ndarray, scales: np.ndarray,
                   qzeros: Optional[np.ndarray], g: int, act: str, k_block: int = 1024) -> np.ndarray:
    """FP64 output rows `rows` of the layer (used on sampled rows of large problems)."""
    return reference(np.asarray(x)[np.asarray(rows)], qweight, scales, qzeros, g, act, k_block)


def reference_cols(x: np.ndarray, cols: Sequence[int], qweight: np.ndarray, scales: np.ndarray,
                   qzeros: Optional[np.ndarray], g: int, act: str, k_block: int = 1024) -> np.ndarray:
    """FP64 output columns `cols` of the layer."""
    return reference(x, qweight, scales, qzeros, g, act, k_block, cols=cols)
