"""Shared helpers of the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI, bring results back as dtype bit patterns."""

from __future__ import annotations

import numpy as np
import torch

from w4a16_int4_weight_gb300 import build as wbuild
from w4a16_int4_weight_gb300 import inputs as synth

TORCH = {"fp16": torch.float16, "bf16": torch.bfloat16}
TOL = {"bf16": 1e-2, "fp16": 2e-3}   # max|C - C_ref| / (max|C_ref| + 1e-6)

_B = None


def B():
    global _B
    if _B is None:
        wbuild.build()
        from w4a16_int4_weight_gb300 import binding
        _B = binding
    return _B


def to_dev_bits(bits: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(TORCH[dtype])


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceWeight:
    """A quantised weight uploaded and packed on the device by w4a16_pack."""

    def __init__(self, p: synth.Problem, q, scales, zeros, stream=None):
        b = B()
        self.p = p
        self.q = torch.from_numpy(np.ascontiguousarray(q)).cuda()
        self.scales_in = to_dev_bits(scales, p.dtype)
        self.zeros_in = torch.from_numpy(np.ascontiguousarray(zeros)).cuda() if zeros is not None else None
        tot, so, zo, ldq = b.packed_layout(p.N, p.K, p.group_size, p.qtype, p.dtype)
        self.total, self.so, self.zo, self.ldq = tot, so, zo, ldq
        self.buf = torch.empty(tot, dtype=torch.uint8, device="cuda")
        b.pack(self.q, self.scales_in, self.zeros_in, self.buf, p.N, p.K, p.group_size, p.qtype,
               p.dtype, stream)
        base = self.buf.data_ptr()
        self.Wq = base
        self.scales = base + so
        self.zeros = base + zo if p.qtype == "uint4" else None

    def words(self) -> np.ndarray:
        return self.buf[: self.p.N * self.ldq * 4].view(torch.int32).cpu().numpy().view(
            np.uint32).reshape(self.p.N, self.ldq)

    def dequant(self) -> torch.Tensor:
        p = self.p
        W = torch.empty(p.N, p.K, dtype=TORCH[p.dtype], device="cuda")
        B().dequant(self.Wq, self.scales, self.zeros, W, p.N, p.K, p.group_size, p.qtype, p.dtype)
        return W


def run_gemm(w: DeviceWeight, A_bits: np.ndarray, path="auto", Wdense=None, M=None):
    p = w.p
    M = A_bits.shape[0] if M is None else M
    A = to_dev_bits(A_bits, p.dtype)
    C = torch.full((M, p.N), float("nan"), dtype=TORCH[p.dtype], device="cuda")   # NaN canary
    B().gemm_ex(A, w.Wq, w.scales, w.zeros, Wdense, C, M, p.N, p.K, p.group_size, p.qtype,
                p.dtype, path)
    torch.cuda.synchronize()
    return to_host_bits(C)


def assert_device_status_ok():
    code, site = B().device_status()
    assert code == 0, f"device status {code} at wait site {site}: {B().last_error()}"
