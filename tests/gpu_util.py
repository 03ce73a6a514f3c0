"""Helpers for the GPU parity tests: move a seeded case to the device, pack it
with the library's own packer, run an entry point, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import weight_only_int4_gb300 as w4
from oracle import w4a16_oracle as O

# max |y - y_ref| <= TOL * max |y_ref|, y_ref in FP64 (fp16 output / bf16 output)
TOL = {"f16": 4e-3, "bf16": 1.6e-2}
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}


def act_to_torch(a: np.ndarray, act: str, device="cuda") -> torch.Tensor:
    if act == "f16":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def torch_to_f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        bits = t.detach().cpu().view(torch.int16).numpy().view(np.uint16)
        return O.widen(bits, "bf16")
    return t.detach().cpu().to(torch.float64).numpy()


class DeviceCase:
    """A case on the device: x, scales, packed qweight / qzeros made by w4a16_pack."""

    def __init__(self, case):
        self.case = case
        self.act = case.act
        self.g = case.g
        self.x = act_to_torch(case.x, case.act)
        self.s = act_to_torch(case.s, case.act)
        self.q_u8 = torch.from_numpy(np.ascontiguousarray(case.q)).cuda()
        self.qw = w4.pack(self.q_u8, dim=0)
        self.qz = None if case.z is None else w4.pack(torch.from_numpy(np.ascontiguousarray(case.z)).cuda(), dim=1)

    def oracle_operands(self):
        c = self.case
        return O.pack_rows(c.q), (None if c.z is None else O.pack_cols(c.z))

    def reference(self, rows=None):
        qw, qz = self.oracle_operands()
        if rows is None:
            return O.reference(self.case.x, qw, self.case.s, qz, self.g, self.act)
        return O.reference_rows(self.case.x, rows, qw, self.case.s, qz, self.g, self.act)


def guarded_out(M: int, N: int, dtype, pad: int = 1024, sentinel: float = -1536.0):
    """Output [M, N] inside a sentinel-filled buffer (16-byte aligned view)."""
    buf = torch.full((M * N + 2 * pad,), sentinel, dtype=dtype, device="cuda")
    return buf, buf[pad:pad + M * N].view(M, N), pad


def check_guards(buf: torch.Tensor, pad: int, sentinel: float = -1536.0):
    head = buf[:pad].float().cpu()
    tail = buf[-pad:].float().cpu()
    assert torch.all(head == sentinel), "write before the output buffer"
    assert torch.all(tail == sentinel), "write after the output buffer"


def assert_within_tol(y: torch.Tensor, ref: np.ndarray, act: str, what: str = ""):
    got = torch_to_f64(y)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref).max() if ref.size else 0.0
    scale = np.abs(ref).max() if ref.size else 0.0
    assert err <= TOL[act] * scale, f"{what}: max err {err:.3e} > {TOL[act]} * {scale:.3e}"
    return err, scale
