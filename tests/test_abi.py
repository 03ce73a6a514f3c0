"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects bad arguments on the host before anything reaches a device."""
import os
import re

import pytest

import weight_only_int4_gb300 as w4
from weight_only_int4_gb300 import build as w4build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(w4.LIB_PATH):
        w4build.build()
    return w4.load_library()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_table():
    assert declared_symbols() == sorted(w4.SIGNATURES)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert w4.abi_version() == 1
    for code, name in enumerate(w4.STATUS_NAMES):
        assert w4.status_string(code) == name
    assert w4.status_string(1234) == "W4A16_ERR_UNKNOWN"


# Pointers that are never dereferenced: every case below fails a host check first.
P = 0x10000
MIS = 0x10008


def _gemv(lib, **kw):
    a = dict(x=P, qw=P, s=P, z=P, y=P, M=1, N=64, K=128, g=32, dt=w4.F16)
    a.update(kw)
    return lib.w4a16_gemv(a["x"], a["qw"], a["s"], a["z"], a["y"], a["M"], a["N"], a["K"], a["g"],
                          a["dt"], a.get("ws", P), a.get("ws_bytes", 1 << 30), None)


def _gemm(lib, **kw):
    a = dict(x=P, qw=P, s=P, z=P, y=P, M=300, N=64, K=128, g=32, dt=w4.BF16)
    a.update(kw)
    return lib.w4a16_gemm(a["x"], a["qw"], a["s"], a["z"], a["y"], a["M"], a["N"], a["K"], a["g"],
                          a["dt"], a.get("ws", P), a.get("ws_bytes", 1 << 30), None)


@pytest.mark.parametrize("call", [_gemv, _gemm])
def test_layer_rejections(lib, call):
    assert call(lib, x=None) == w4.ERR_NULL
    assert call(lib, qw=None) == w4.ERR_NULL
    assert call(lib, s=None) == w4.ERR_NULL
    assert call(lib, y=None) == w4.ERR_NULL
    assert call(lib, dt=7) == w4.ERR_DTYPE
    assert call(lib, N=60) == w4.ERR_SHAPE            # N % 8
    assert call(lib, K=100) == w4.ERR_SHAPE           # K % g
    assert call(lib, M=0) == w4.ERR_SHAPE
    assert call(lib, N=-8) == w4.ERR_SHAPE
    assert call(lib, K=1 << 33, g=32) == w4.ERR_SHAPE
    assert call(lib, g=48, K=96) == w4.ERR_UNSUPPORTED
    assert call(lib, g=16, K=128) == w4.ERR_UNSUPPORTED
    assert call(lib, x=MIS) == w4.ERR_ALIGN
    assert call(lib, z=MIS) == w4.ERR_ALIGN
    assert call(lib, y=MIS) == w4.ERR_ALIGN


def test_gemv_row_limit(lib):
    assert _gemv(lib, M=17) == w4.ERR_SHAPE


def test_gemv_needs_an_aligned_workspace(lib):
    assert _gemv(lib, ws=None) == w4.ERR_WORKSPACE
    assert _gemv(lib, ws=MIS) == w4.ERR_WORKSPACE


def test_dequant_rejections(lib):
    d = lambda **kw: lib.w4a16_dequant(kw.get("qw", P), kw.get("s", P), kw.get("z", P), kw.get("w", P),
                                       kw.get("N", 64), kw.get("K", 128), kw.get("g", 32), kw.get("dt", w4.F16), None)
    assert d(qw=None) == w4.ERR_NULL
    assert d(w=None) == w4.ERR_NULL
    assert d(dt=5) == w4.ERR_DTYPE
    assert d(N=60) == w4.ERR_SHAPE
    assert d(K=100) == w4.ERR_SHAPE
    assert d(g=48, K=96) == w4.ERR_UNSUPPORTED
    assert d(w=MIS) == w4.ERR_ALIGN
    assert d(z=MIS) == w4.ERR_ALIGN


def test_pack_rejections(lib):
    assert lib.w4a16_pack(None, P, 8, 8, 0, None) == w4.ERR_NULL
    assert lib.w4a16_pack(P, P, 12, 8, 0, None) == w4.ERR_SHAPE      # rows % 8 for dim 0
    assert lib.w4a16_pack(P, P, 8, 12, 1, None) == w4.ERR_SHAPE      # cols % 8 for dim 1
    assert lib.w4a16_pack(P, P, 8, 8, 2, None) == w4.ERR_SHAPE
    assert lib.w4a16_pack(P, MIS, 8, 8, 0, None) == w4.ERR_ALIGN
    assert lib.w4a16_unpack(P, None, 8, 8, 0, None) == w4.ERR_NULL
    assert lib.w4a16_unpack(P, P, 0, 8, 0, None) == w4.ERR_SHAPE


def _has_cuda_device():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(_has_cuda_device(), reason="needs a host without a CUDA device")
def _mx(lib, fn, **kw):
    a = dict(x=P, qw=P, e=P, y=P, M=1, N=64, K=128)
    a.update(kw)
    if fn == "dequant":
        return lib.w4a16_mxfp4_dequant(a["qw"], a["e"], a["y"], a["N"], a["K"], None)
    if fn == "gemv":
        return lib.w4a16_mxfp4_gemv(a["x"], a["qw"], a["e"], a["y"], a["M"], a["N"], a["K"], a.get("ws", P),
                                    a.get("ws_bytes", 1 << 30), None)
    return lib.w4a16_mxfp4_gemm(a["x"], a["qw"], a["e"], a["y"], a["M"], a["N"], a["K"], a.get("ws", P),
                                a.get("ws_bytes", 1 << 30), None)


@pytest.mark.parametrize("fn", ["dequant", "gemv", "gemm"])
def test_mxfp4_rejections(lib, fn):
    assert _mx(lib, fn, qw=0) == w4.ERR_NULL
    assert _mx(lib, fn, e=0) == w4.ERR_NULL
    assert _mx(lib, fn, y=0) == w4.ERR_NULL
    assert _mx(lib, fn, N=8) == w4.ERR_SHAPE           # exponent rows must start 16-byte aligned
    assert _mx(lib, fn, K=48) == w4.ERR_SHAPE          # K % 32
    assert _mx(lib, fn, K=0) == w4.ERR_SHAPE
    assert _mx(lib, fn, e=MIS) == w4.ERR_ALIGN
    assert _mx(lib, fn, qw=MIS) == w4.ERR_ALIGN
    assert _mx(lib, fn, y=MIS) == w4.ERR_ALIGN
    if fn != "dequant":
        assert _mx(lib, fn, x=0) == w4.ERR_NULL
        assert _mx(lib, fn, M=0) == w4.ERR_SHAPE
        assert _mx(lib, fn, x=MIS) == w4.ERR_ALIGN
    if fn == "gemv":
        assert _mx(lib, fn, M=17) == w4.ERR_SHAPE
    if fn != "dequant":
        assert _mx(lib, fn, ws=0) == w4.ERR_WORKSPACE      # M <= 128: the GEMM needs its workspace too
        assert _mx(lib, fn, ws=MIS) == w4.ERR_WORKSPACE


def test_gemm_few_rows_needs_a_workspace(lib):
    # M <= 128 runs the stream-K kernel, whose partial sums live in the workspace
    assert _gemm(lib, M=64, ws=0) == w4.ERR_WORKSPACE
    assert _gemm(lib, M=64, ws=MIS) == w4.ERR_WORKSPACE
    assert _gemm(lib, M=300, ws=0) == w4.ERR_DEVICE         # the CTA-pair kernel needs none
    assert lib.w4a16_workspace_bytes(w4.OP_GEMM, 300, 64, 128, 32) == 0


def test_valid_arguments_stop_at_the_device_gate(lib):
    assert _gemv(lib) == w4.ERR_DEVICE
    assert _gemm(lib) == w4.ERR_DEVICE
    assert lib.w4a16_pack(P, P, 8, 8, 0, None) == w4.ERR_DEVICE
    assert lib.w4a16_device_status(None) == w4.ERR_DEVICE
    assert lib.w4a16_selftest_wait_timeout(None) == w4.ERR_DEVICE
    assert lib.w4a16_dequant(P, P, P, P, 64, 128, 32, w4.F16, None) == w4.ERR_DEVICE
    for fn in ("dequant", "gemv", "gemm"):
        assert _mx(lib, fn) == w4.ERR_DEVICE
    assert _mx(lib, "gemm", M=4096) == w4.ERR_DEVICE
    assert lib.w4a16_workspace_bytes(w4.OP_GEMV, 1, 64, 128, 32) == 0


def test_binding_rejects_activation_dtype_zero_points():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 64, dtype=torch.float16)
    qw = torch.zeros(8, 64, dtype=torch.int32)
    s = torch.zeros(2, 64, dtype=torch.float16)
    z_expanded = torch.zeros(2, 64, dtype=torch.float16)
    # CPU tensors are rejected before any dtype reasoning reaches the library
    with pytest.raises(ValueError):
        w4.gemv(x, qw, s, z_expanded, 32)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libw4a16.so the binding raises; there is no fallback path."""
    monkeypatch.setattr(w4, "_lib", None)
    with pytest.raises(RuntimeError, match="libw4a16.so not found"):
        w4.load_library(str(tmp_path / "libw4a16.so"))


def test_release_workspaces_drops_the_cache(monkeypatch):
    monkeypatch.setattr(w4, "_workspaces", {(0, 0, w4.OP_GEMV): object()})
    w4.release_workspaces()
    assert w4._workspaces == {}
