"""The linear layer's bias (w4a16_linear) on every GEMM path, against the oracle.

The bias is added to the fp32 accumulator before the output's one rounding:
parity within the GEMM tolerance on ragged and split-K shapes, and two exact
cases - zero weights give the bias itself, and one-hot activations give
rne(w + b) bit for bit (the fp32 sum of a weight and a bias of these
magnitudes is exact), where w is the dequantised weight for the tcgen05 kernels
and the unrounded (q - z) * s for the small-M kernel, which scales group sums.
"""

import numpy as np
import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

from gpu_helpers import TOL, TORCH, B, DeviceWeight, assert_device_status_ok, to_dev_bits, to_host_bits

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 512, 512, 128, "uint4b8", "fp16"),
    (8, 384, 768, 32, "uint4", "fp16"),
    (13, 136, 2048, 128, "uint4b8", "bf16"),   # ragged N, K split over a cluster
    (40, 136, 4112, -1, "uint4b8", "bf16"),    # K % 32 == 16
    (77, 200, 1088, 64, "uint4", "fp16"),
    (300, 384, 512, 128, "uint4b8", "bf16"),
]


def _bias(N, dtype, seed):
    rng = np.random.default_rng(seed)
    b = rng.uniform(0.25, 2.0, N) * np.where(rng.random(N) < 0.5, -1.0, 1.0)   # never 0
    return orc.round_to(b, dtype)


def _paths(M):
    return (["decode"] if M <= 64 else []) + ["fused_tmem", "fused_smem", "dense", "auto"]


def run_linear(w, A_bits, bias_bits, path, Wdense=None):
    p = w.p
    M = A_bits.shape[0]
    A = to_dev_bits(A_bits, p.dtype)
    bias = to_dev_bits(bias_bits, p.dtype) if bias_bits is not None else None
    C = torch.full((M, p.N), float("nan"), dtype=TORCH[p.dtype], device="cuda")
    B().linear(A, w.Wq, w.scales, w.zeros, bias, Wdense, C, M, p.N, p.K, p.group_size, p.qtype,
               p.dtype, path)
    torch.cuda.synchronize()
    return to_host_bits(C)


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_linear_with_bias_matches_oracle_on_every_path(sh):
    p = synth.Problem(*sh)
    x = synth.make_inputs(p)
    bias = _bias(p.N, p.dtype, 3)
    C_ref = orc.linear(x.A, x.q, x.scales, x.zeros, p.group_size, p.dtype, bias=bias)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    Wd = w.dequant()
    for path in _paths(p.M):
        C = run_linear(w, x.A, bias, path, Wdense=Wd if path in ("dense", "auto") else None)
        Cv = orc.values(C, p.dtype)
        assert np.all(np.isfinite(Cv)), path
        err = orc.rel_error(Cv, C_ref)
        assert err <= TOL[p.dtype], (path, err)
    assert_device_status_ok()


@pytest.mark.parametrize("path", ["decode", "fused_tmem", "fused_smem", "dense"])
def test_zero_weights_give_the_bias_exactly(path):
    p = synth.Problem(24, 200, 1024, 64, "uint4", "bf16")
    x = synth.make_inputs(p)
    ng = p.ngroups
    q = np.empty((p.N, p.K), dtype=np.uint8)
    for n in range(p.N):
        for g in range(ng):
            q[n, 64 * g:64 * (g + 1)] = orc.zero_point(x.zeros, ng, n, g)
    bias = _bias(p.N, p.dtype, 9)
    w = DeviceWeight(p, q, x.scales, x.zeros)
    C = run_linear(w, x.A, bias, path, Wdense=w.dequant() if path == "dense" else None)
    assert np.array_equal(C, np.broadcast_to(bias, C.shape))


@pytest.mark.parametrize("path", ["decode", "fused_tmem", "fused_smem", "dense"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_one_hot_plus_bias_is_rounded_once(path, dtype):
    M, N, K, G = 24, 256, 1024, 64
    p = synth.Problem(M, N, K, G, "uint4", dtype)
    q, s, z = synth.make_weights(p)
    if path == "decode":
        # The small-M kernel applies the scale to each group's fp32 sum instead
        # of rounding each dequantised weight; with power-of-two scales (sign and
        # exponent bits of the seeded ones) the dequantised weight (q - z) * s is
        # exact, so both orders give the oracle's value.
        s = s & np.uint16(0xFF80 if dtype == "bf16" else 0xFC00)
    km = (np.arange(M) * 37 + 5) % K
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), km] = 0x3F80 if dtype == "bf16" else 0x3C00
    bias = _bias(N, dtype, 4)
    w = DeviceWeight(p, q, s, z)
    # a one-hot row gives the dequantised weight plus the bias, rounded once
    wk = orc.values(orc.dequant(q, s, z, G, dtype), dtype)[:, km].T
    want = orc.round_to(wk + orc.values(bias, dtype)[None, :], dtype)
    C = run_linear(w, A, bias, path, Wdense=w.dequant() if path == "dense" else None)
    assert np.array_equal(C, want)


def test_null_bias_equals_gemm_ex():
    p = synth.Problem(5, 256, 1024, 128, "uint4b8", "bf16")
    x = synth.make_inputs(p)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    C0 = run_linear(w, x.A, None, "auto")
    A = to_dev_bits(x.A, p.dtype)
    C1 = torch.empty(p.M, p.N, dtype=TORCH[p.dtype], device="cuda")
    B().gemm_ex(A, w.Wq, w.scales, w.zeros, None, C1, p.M, p.N, p.K, p.group_size, p.qtype, p.dtype)
    torch.cuda.synchronize()
    assert np.array_equal(C0, to_host_bits(C1))
