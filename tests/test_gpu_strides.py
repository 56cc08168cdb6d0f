"""Padded row pitches of A and C (w4a16_linear's lda and ldc) on every path.

A is a view into a wider buffer whose padding holds NaN (any read of it would
poison the result); C is written into a wider buffer whose padding holds a guard
value that must survive.  Results are compared with the oracle.
"""

import numpy as np
import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

from gpu_helpers import TOL, TORCH, B, DeviceWeight, assert_device_status_ok, to_dev_bits, to_host_bits

pytestmark = pytest.mark.gpu

SHAPES = [
    (3, 200, 1024, 64, "uint4", "bf16", 1032, 208),
    (16, 384, 768, 32, "uint4", "fp16", 1024, 400),
    (40, 136, 4112, -1, "uint4b8", "bf16", 4160, 137),
    (300, 384, 512, 128, "uint4b8", "bf16", 520, 512),
]


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_padded_a_and_c(sh):
    M, N, K, G, qt, dt, lda, ldc = sh
    p = synth.Problem(M, N, K, G, qt, dt)
    x = synth.make_inputs(p)
    C_ref = orc.linear(x.A, x.q, x.scales, x.zeros, G, dt)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    Wd = w.dequant()
    A_wide = torch.full((M, lda), float("nan"), dtype=TORCH[dt], device="cuda")
    A_wide[:, :K] = to_dev_bits(x.A, dt)
    paths = (["decode"] if M <= 64 else []) + ["fused_tmem", "fused_smem", "dense", "auto"]
    for path in paths:
        C_wide = torch.full((M, ldc), 7.0, dtype=TORCH[dt], device="cuda")
        B().linear(A_wide, w.Wq, w.scales, w.zeros, None, Wd if path in ("dense", "auto") else None,
                   C_wide, M, N, K, G, qt, dt, path, lda=lda, ldc=ldc)
        torch.cuda.synchronize()
        C = to_host_bits(C_wide[:, :N])
        err = orc.rel_error(orc.values(C, dt), C_ref)
        assert err <= TOL[dt], (path, err)
        if ldc > N:
            assert torch.all(C_wide[:, N:] == 7.0), path
    assert_device_status_ok()


@pytest.mark.parametrize("path", ["fused_tmem", "fused_smem", "dense"])
def test_c_base_off_sixteen_byte_alignment(path):
    # C starts one element into its buffer: the tcgen05 kernels must take their
    # direct-store epilogue (no TMA store) and still write exactly [M, N].
    M, N, K, G, qt, dt = 130, 264, 1024, 128, "uint4b8", "bf16"
    p = synth.Problem(M, N, K, G, qt, dt)
    x = synth.make_inputs(p)
    C_ref = orc.linear(x.A, x.q, x.scales, x.zeros, G, dt)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    ldc = N + 8
    buf = torch.full((M + 1, ldc), 7.0, dtype=TORCH[dt], device="cuda")
    flat = buf.view(-1)
    C = flat[1:1 + M * ldc].view(M, ldc)          # base address 2 bytes past a 16-byte boundary
    assert C.data_ptr() % 16 == 2
    A = to_dev_bits(x.A, dt)
    B().linear(A, w.Wq, w.scales, w.zeros, None, w.dequant() if path == "dense" else None,
               C, M, N, K, G, qt, dt, path, ldc=ldc)
    torch.cuda.synchronize()
    got = to_host_bits(C[:, :N])
    assert orc.rel_error(orc.values(got, dt), C_ref) <= TOL[dt]
    assert torch.all(C[:, N:] == 7.0) and float(flat[0]) == 7.0
    assert torch.all(flat[1 + M * ldc:] == 7.0)
    assert_device_status_ok()
