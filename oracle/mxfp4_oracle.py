"""CPU FP64 oracle for the MXFP4 weight encoding (E2M1 codes, E8M0 block scales).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. The product never calls it and shares
no code with it. It reuses the packer and unpacker of the W4A16 oracle (same
word layout, both are oracle code).

What it computes follows "Add BF16xFP4 MoE GEMM stage1 kernel" (section
"Technical Details"): activations stay bf16, each weight is a 4-bit E2M1 code,
eight codes share a 32-bit word along K, each run of 32 K rows of a column
shares one E8M0 byte e whose value is 2^(e - 127), and the weights are decoded
to bf16 in software before the contraction (FP32 accumulation there, FP64 here):

    W[k, n] = RN_bf16( E2M1(q[k, n]) * 2^(e[k // 32, n] - 127) )
    y[m, n] = sum_k x[m, k] * W[k, n]

Operands:
  * qweight int32 [K/8, N]: nibble j (bits 4j..4j+3) of word [w, n] is the
    code of row k = 8w + j, the layout of the W4A16 layer;
  * escale uint8 [K/32, N]: the E8M0 byte of block b and column n;
  * x [M, K] bf16 bit patterns (uint16), widened exactly to FP64.

Readings where the page is silent (each is listed with the design notes):
  * E2M1 value of a code c: bit 3 is the sign, bits 2..1 the exponent field E
    (bias 1), bit 0 the mantissa bit m. E = 0 has no implicit leading one and
    gives m / 2; otherwise the value is 2^(E - 1) * (1 + m / 2).
  * E8M0 byte 255 is not a power of two in that encoding; it decodes to NaN,
    so every weight of its block is NaN. Byte 0 is 2^-127.
  * Every decoded weight E2M1 * 2^(e - 127) has at most two significant bits
    and is exact in bf16 (subnormals included) unless it exceeds the bf16
    range, where round-to-nearest gives +-inf.

Parity status of each function (pins in the tests):
  e2m1_decode ......... pinned
  e8m0_decode ......... pinned
  dequantize_mx ....... pinned
  reference_mx ........ pinned
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from oracle.w4a16_oracle import NIBBLES_PER_WORD, round_to_act, unpack_rows, widen

MX_BLOCK = 32          # K rows sharing one E8M0 byte
E2M1_BIAS = 1
E8M0_BIAS = 127
E8M0_NAN = 255


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """FP64 value of 4-bit E2M1 codes (any integer array with values 0..15)."""
    c = np.asarray(codes).astype(np.int64)
    if c.size and (c.min() < 0 or c.max() > 15):
        raise ValueError("E2M1 codes are 4-bit")
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    E = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    normal = np.ldexp(1.0 + m / 2.0, np.maximum(E, 1) - E2M1_BIAS)
    subnormal = m / 2.0               # 2^(1 - bias) * (m / 2)
    return sign * np.where(E == 0, subnormal, normal)


def e8m0_decode(e: np.ndarray) -> np.ndarray:
    """FP64 value 2^(e - 127) of E8M0 bytes; NaN for 255."""
    b = np.asarray(e).astype(np.int64)
    if b.size and (b.min() < 0 or b.max() > 255):
        raise ValueError("E8M0 scales are bytes")
    return np.where(b == E8M0_NAN, np.nan, np.ldexp(1.0, b - E8M0_BIAS))


def dequantize_mx(qweight: np.ndarray, escale: np.ndarray, k0: int = 0, k1: Optional[int] = None,
                  cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """FP64 values of the bf16 weights of rows k0..k1 (multiples of 8)."""
    K = qweight.shape[0] * NIBBLES_PER_WORD
    N = qweight.shape[1]
    if k1 is None:
        k1 = K
    if k0 % NIBBLES_PER_WORD or k1 % NIBBLES_PER_WORD:
        raise ValueError("row range must be word aligned")
    if K % MX_BLOCK or escale.shape != (K // MX_BLOCK, N):
        raise ValueError("escale shape does not match K/32 x N")
    q = unpack_rows(qweight[k0 // NIBBLES_PER_WORD:k1 // NIBBLES_PER_WORD])
    s = e8m0_decode(escale)
    blk = np.arange(k0, k1) // MX_BLOCK
    if cols is not None:
        cols = np.asarray(cols)
        q, s = q[:, cols], s[:, cols]
    with np.errstate(over="ignore", invalid="ignore"):
        return round_to_act(e2m1_decode(q) * s[blk], "bf16")


def reference_mx(x: np.ndarray, qweight: np.ndarray, escale: np.ndarray, k_block: int = 1024,
                 cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """FP64 y = x @ dequantize_mx(...), summed over K in blocks of `k_block` rows."""
    xd = widen(x, "bf16")
    M, K = xd.shape
    if qweight.shape[0] * NIBBLES_PER_WORD != K:
        raise ValueError("x and qweight disagree on K")
    kb = max(NIBBLES_PER_WORD, (k_block // NIBBLES_PER_WORD) * NIBBLES_PER_WORD)
    ncols = qweight.shape[1] if cols is None else len(cols)
    y = np.zeros((M, ncols), dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        for k0 in range(0, K, kb):
            k1 = min(K, k0 + kb)
            y += xd[:, k0:k1] @ dequantize_mx(qweight, escale, k0, k1, cols)
    return y


def reference_mx_rows(x: np.ndarray, rows: Sequence[int], qweight: np.ndarray, escale: np.ndarray,
                      k_block: int = 1024) -> np.ndarray:
    """FP64 output rows `rows` of the MXFP4 layer."""
    return reference_mx(np.asarray(x)[np.asarray(rows)], qweight, escale, k_block)
