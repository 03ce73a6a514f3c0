"""weight_only_int4_gb300 -- W4A16 group-quantized linear layer for GB300.

A thin ctypes binding over libw4a16.so (C ABI in include/w4a16.h). Every
function below only checks and marshals its arguments (torch tensors ->
device pointers, the current CUDA stream) and calls the entry point of the
same name; all arithmetic runs in the library's CUDA kernels. There is no
CPU fallback: if the library is missing or the device is not a GB300, calls
raise.

    y = x @ W,   W[k, n] = (q[k, n] - z[k // g, n]) * s[k // g, n]

Operands (all CUDA tensors, contiguous):
    x        [M, K]    torch.float16 or torch.bfloat16
    qweight  [K/8, N]  torch.int32, nibble j of word [w, n] = q[8w + j, n]
    scales   [K/g, N]  same dtype as x
    qzeros   [K/g, N/8] torch.int32 (zero-point of column n in word n // 8 at
             bits 4 * (n % 8)), or None for the symmetric layer (z = 8).
             Zero-points in the activation dtype are rejected, never
             reinterpreted (as "Keep W4A16 zero-points packed at 4 bits
             instead of expanding to 2 bytes" requires, section "Testing").
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .accounting import expanded_zero_bytes, layer_bytes, layer_flops  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libw4a16.so")

STATUS_NAMES = [
    "W4A16_OK", "W4A16_ERR_NULL", "W4A16_ERR_SHAPE", "W4A16_ERR_DTYPE", "W4A16_ERR_ALIGN",
    "W4A16_ERR_UNSUPPORTED", "W4A16_ERR_DEVICE", "W4A16_ERR_WORKSPACE", "W4A16_ERR_CUDA",
    "W4A16_ERR_TIMEOUT",
]
OK, ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_DEVICE, ERR_WORKSPACE, \
    ERR_CUDA, ERR_TIMEOUT = range(10)
F16, BF16 = 0, 1
OP_GEMV, OP_GEMM = 0, 1

# Every symbol include/w4a16.h declares, with (restype, argtypes).
_VP, _I64, _SZ, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
_LAYER_ARGS = [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _INT, _VP, _SZ, _VP]
SIGNATURES = {
    "w4a16_pack": (_INT, [_VP, _VP, _I64, _I64, _INT, _VP]),
    "w4a16_unpack": (_INT, [_VP, _VP, _I64, _I64, _INT, _VP]),
    "w4a16_workspace_bytes": (_SZ, [_INT, _I64, _I64, _I64, _I64]),
    "w4a16_gemv": (_INT, _LAYER_ARGS),
    "w4a16_gemm": (_INT, _LAYER_ARGS),
    "w4a16_gemv_noalloc": (_INT, [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _INT, _VP]),
    "w4a16_device_status": (_INT, [_VP]),
    "w4a16_selftest_wait_timeout": (_INT, [_VP]),
    "w4a16_dequant": (_INT, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _INT, _VP]),
    "w4a16_mxfp4_dequant": (_INT, [_VP, _VP, _VP, _I64, _I64, _VP]),
    "w4a16_mxfp4_gemv": (_INT, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP, _SZ, _VP]),
    "w4a16_mxfp4_gemm": (_INT, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP, _SZ, _VP]),
    "w4a16_status_string": (ctypes.c_char_p, [_INT]),
    "w4a16_abi_version": (_INT, []),
}


class W4A16Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else f"status {status}"
        super().__init__(f"{fn} failed: {name}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libw4a16.so (built by weight_only_int4_gb300.build). Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libw4a16.so not found at {path}; build it with "
                           "`python -m weight_only_int4_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().w4a16_status_string(status).decode()


def abi_version() -> int:
    return load_library().w4a16_abi_version()


def _torch():
    import torch
    return torch


def _stream_ptr(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check(fn: str, status: int) -> None:
    if status != OK:
        raise W4A16Error(fn, status)


def _act_code(dtype) -> int:
    torch = _torch()
    if dtype == torch.float16:
        return F16
    if dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"activations must be float16 or bfloat16, got {dtype}")


def _cuda_contig(name: str, t) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def pack(codes, dim: int, out=None, stream=None):
    """Pack uint8 4-bit codes [R, C] eight to an int32 word along `dim` (0: rows, 1: cols)."""
    torch = _torch()
    _cuda_contig("codes", codes)
    if codes.dtype != torch.uint8 or codes.dim() != 2:
        raise TypeError("codes must be a 2-D torch.uint8 tensor")
    R, C = codes.shape
    shape = (R // 8, C) if dim == 0 else (R, C // 8)
    if out is None:
        out = torch.empty(shape, dtype=torch.int32, device=codes.device)
    _cuda_contig("out", out)
    _check("w4a16_pack", load_library().w4a16_pack(codes.data_ptr(), out.data_ptr(), R, C, dim,
                                                   _stream_ptr(stream)))
    return out


def unpack(words, dim: int, out=None, stream=None):
    """Inverse of pack: int32 words -> uint8 codes [R, C]."""
    torch = _torch()
    _cuda_contig("words", words)
    if words.dtype != torch.int32 or words.dim() != 2:
        raise TypeError("words must be a 2-D torch.int32 tensor")
    W0, W1 = words.shape
    R, C = (W0 * 8, W1) if dim == 0 else (W0, W1 * 8)
    if out is None:
        out = torch.empty((R, C), dtype=torch.uint8, device=words.device)
    _cuda_contig("out", out)
    _check("w4a16_unpack", load_library().w4a16_unpack(words.data_ptr(), out.data_ptr(), R, C, dim,
                                                       _stream_ptr(stream)))
    return out


def workspace_bytes(op: int, M: int, N: int, K: int, g: int) -> int:
    """Device workspace the op needs on the current device (0 if none)."""
    return int(load_library().w4a16_workspace_bytes(op, M, N, K, g))


def new_workspace(nbytes: int, device=None):
    """A zero-filled uint8 device workspace. Calls leave it zeroed where it must
    start at zero, so one workspace serves any number of calls, as long as no
    two calls that use it run at the same time."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8,
                       device=torch.device("cuda") if device is None else device)


_workspaces = {}
_retired = []


def _cached_workspace(nbytes: int, device, stream, op: int):
    """One growing workspace per (device, stream, op): calls on one stream never
    overlap, and the GEMV and the GEMM lay out their workspaces differently.

    The workspace is allocated and zero-filled on the stream the call runs on,
    so the zero fill is ordered before the kernel and the caching allocator
    ties the memory to that stream. A workspace outgrown by a larger shape is
    kept alive (not freed) until release_workspaces(): a CUDA graph captured
    through an earlier call may still replay into it."""
    torch = _torch()
    dev = device.index if device.index is not None else torch.cuda.current_device()
    s = torch.cuda.current_stream(dev) if stream is None else stream
    key = (dev, int(s.cuda_stream), op)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(s):
            fresh = new_workspace(nbytes, device)
        if ws is not None:
            _retired.append(ws)
        _workspaces[key] = ws = fresh
    return ws


def release_workspaces() -> None:
    """Free the workspaces the binding allocated for calls made without one (one
    per device, stream and op, plus any outgrown by larger shapes). Call it only
    when no such call is in flight, and only after dropping every CUDA graph
    captured through such calls: a captured graph replays into the workspace
    address it saw at capture time. The next call allocates a fresh, zeroed
    workspace."""
    _workspaces.clear()
    _retired.clear()


def _layer(fn_name: str, x, qweight, scales, qzeros, group_size: int, out=None, workspace=None,
           stream=None):
    torch = _torch()
    for name, t in (("x", x), ("qweight", qweight), ("scales", scales)):
        _cuda_contig(name, t)
    if x.dim() != 2 or qweight.dim() != 2 or scales.dim() != 2:
        raise ValueError("x, qweight and scales must be 2-D")
    dt = _act_code(x.dtype)
    if scales.dtype != x.dtype:
        raise TypeError(f"scales dtype {scales.dtype} differs from x dtype {x.dtype}")
    if qweight.dtype != torch.int32:
        raise TypeError(f"qweight must be torch.int32, got {qweight.dtype}")
    M, K = x.shape
    N = qweight.shape[1]
    if qweight.shape[0] * 8 != K:
        raise ValueError(f"qweight rows {qweight.shape[0]} do not match K/8 = {K / 8}")
    if K % group_size or scales.shape != (K // group_size, N):
        raise ValueError(f"scales shape {tuple(scales.shape)} does not match (K/g, N)")
    zp = 0
    if qzeros is not None:
        _cuda_contig("qzeros", qzeros)
        if qzeros.dtype != torch.int32:
            raise TypeError(f"qzeros must be packed torch.int32 [K/g, N/8]; got {qzeros.dtype} "
                            "(zero-points in the activation dtype are rejected)")
        if qzeros.shape != (K // group_size, N // 8):
            raise ValueError(f"qzeros shape {tuple(qzeros.shape)} does not match (K/g, N/8)")
        zp = qzeros.data_ptr()
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    _cuda_contig("out", out)
    lib = load_library()
    sp = _stream_ptr(stream)
    if workspace is None:
        op = OP_GEMV if fn_name == "w4a16_gemv" else OP_GEMM
        need = lib.w4a16_workspace_bytes(op, M, N, K, group_size)
        workspace = _cached_workspace(need, x.device, stream, op) if need else None
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (workspace.data_ptr(),
                                                          workspace.numel() * workspace.element_size())
    _check(fn_name, getattr(lib, fn_name)(x.data_ptr(), qweight.data_ptr(), scales.data_ptr(), zp,
                                          out.data_ptr(), M, N, K, group_size, dt, ws_ptr, ws_bytes, sp))
    return out


def gemv(x, qweight, scales, qzeros: Optional[object], group_size: int, out=None, workspace=None,
         stream=None):
    """Decode path (1 <= M <= 16). Returns y [M, N] in x's dtype."""
    return _layer("w4a16_gemv", x, qweight, scales, qzeros, group_size, out, workspace, stream)


def gemm(x, qweight, scales, qzeros: Optional[object], group_size: int, out=None, workspace=None,
         stream=None):
    """Prefill path (any M >= 1, tcgen05 tensor cores). Returns y [M, N] in x's dtype."""
    return _layer("w4a16_gemm", x, qweight, scales, qzeros, group_size, out, workspace, stream)


def dequant(qweight, scales, qzeros: Optional[object], group_size: int, out=None, stream=None):
    """Dense dequantised copy W[k, n] = RN((q - z) * s) in the scales' dtype, [K, N]."""
    torch = _torch()
    for name, t in (("qweight", qweight), ("scales", scales)):
        _cuda_contig(name, t)
    if qweight.dim() != 2 or scales.dim() != 2:
        raise ValueError("qweight and scales must be 2-D")
    if qweight.dtype != torch.int32:
        raise TypeError(f"qweight must be torch.int32, got {qweight.dtype}")
    dt = _act_code(scales.dtype)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    if K % group_size or scales.shape != (K // group_size, N):
        raise ValueError(f"scales shape {tuple(scales.shape)} does not match (K/g, N)")
    zp = 0
    if qzeros is not None:
        _cuda_contig("qzeros", qzeros)
        if qzeros.dtype != torch.int32:
            raise TypeError(f"qzeros must be packed torch.int32 [K/g, N/8]; got {qzeros.dtype} "
                            "(zero-points in the activation dtype are rejected)")
        if qzeros.shape != (K // group_size, N // 8):
            raise ValueError(f"qzeros shape {tuple(qzeros.shape)} does not match (K/g, N/8)")
        zp = qzeros.data_ptr()
    if out is None:
        out = torch.empty((K, N), dtype=scales.dtype, device=scales.device)
    _cuda_contig("out", out)
    if out.shape != (K, N) or out.dtype != scales.dtype:
        raise ValueError(f"out must be {scales.dtype} [K, N] = [{K}, {N}]")
    _check("w4a16_dequant", load_library().w4a16_dequant(qweight.data_ptr(), scales.data_ptr(), zp, out.data_ptr(),
                                                         N, K, group_size, dt, _stream_ptr(stream)))
    return out


def _mx_weights(qweight, escale):
    torch = _torch()
    for name, t in (("qweight", qweight), ("escale", escale)):
        _cuda_contig(name, t)
    if qweight.dim() != 2 or escale.dim() != 2:
        raise ValueError("qweight and escale must be 2-D")
    if qweight.dtype != torch.int32:
        raise TypeError(f"qweight must be torch.int32, got {qweight.dtype}")
    if escale.dtype != torch.uint8:
        raise TypeError(f"escale must be torch.uint8 E8M0 bytes, got {escale.dtype}")
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    if escale.shape != (K // 32, N) or K % 32:
        raise ValueError(f"escale shape {tuple(escale.shape)} does not match (K/32, N)")
    return K, N


def _mx_layer(fn_name: str, x, qweight, escale, out, workspace, stream):
    torch = _torch()
    K, N = _mx_weights(qweight, escale)
    _cuda_contig("x", x)
    if x.dim() != 2 or x.dtype != torch.bfloat16:
        raise TypeError("x must be a 2-D torch.bfloat16 tensor")
    M = x.shape[0]
    if x.shape[1] != K:
        raise ValueError(f"x has {x.shape[1]} columns, qweight holds K = {K} rows")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda_contig("out", out)
    if out.shape != (M, N) or out.dtype != torch.bfloat16:
        raise ValueError(f"out must be bf16 [M, N] = [{M}, {N}]")
    lib = load_library()
    sp = _stream_ptr(stream)
    if workspace is None:
        op = OP_GEMM if fn_name == "w4a16_mxfp4_gemm" else OP_GEMV
        need = lib.w4a16_workspace_bytes(op, M, N, K, 32)
        workspace = _cached_workspace(need, x.device, stream, op) if need else None
    ws_ptr, ws_bytes = (0, 0) if workspace is None else (workspace.data_ptr(),
                                                          workspace.numel() * workspace.element_size())
    if fn_name == "w4a16_mxfp4_gemm":
        _check(fn_name, lib.w4a16_mxfp4_gemm(x.data_ptr(), qweight.data_ptr(), escale.data_ptr(), out.data_ptr(),
                                              M, N, K, ws_ptr, ws_bytes, sp))
        return out
    _check(fn_name, lib.w4a16_mxfp4_gemv(x.data_ptr(), qweight.data_ptr(), escale.data_ptr(), out.data_ptr(),
                                          M, N, K, ws_ptr, ws_bytes, sp))
    return out


def mxfp4_gemv(x, qweight, escale, out=None, workspace=None, stream=None):
    """Decode path for MXFP4 weights (E2M1 codes in `qweight`, E8M0 bytes
    `escale` [K/32, N]); x bf16 [M, K] with 1 <= M <= 16. Returns bf16 y [M, N]."""
    return _mx_layer("w4a16_mxfp4_gemv", x, qweight, escale, out, workspace, stream)


def mxfp4_gemm(x, qweight, escale, out=None, workspace=None, stream=None):
    """Prefill path for MXFP4 weights (any M >= 1, tcgen05). Returns bf16 y [M, N]."""
    return _mx_layer("w4a16_mxfp4_gemm", x, qweight, escale, out, workspace, stream)


def mxfp4_dequant(qweight, escale, out=None, stream=None):
    """Dense bf16 copy W[k, n] = E2M1(q[k, n]) * 2^(e[k/32, n] - 127), [K, N]."""
    torch = _torch()
    K, N = _mx_weights(qweight, escale)
    if out is None:
        out = torch.empty((K, N), dtype=torch.bfloat16, device=qweight.device)
    _cuda_contig("out", out)
    if out.shape != (K, N) or out.dtype != torch.bfloat16:
        raise ValueError(f"out must be bf16 [K, N] = [{K}, {N}]")
    _check("w4a16_mxfp4_dequant", load_library().w4a16_mxfp4_dequant(qweight.data_ptr(), escale.data_ptr(),
                                                                       out.data_ptr(), N, K, _stream_ptr(stream)))
    return out


def device_status(stream=None) -> int:
    """Synchronise the stream, return and clear the device-side error status."""
    return int(load_library().w4a16_device_status(_stream_ptr(stream)))


def selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self-test (one warp waits on a barrier nothing
    completes; it gives up after about two seconds and records
    W4A16_ERR_TIMEOUT, which `device_status` then returns)."""
    _check("w4a16_selftest_wait_timeout", load_library().w4a16_selftest_wait_timeout(_stream_ptr(stream)))
