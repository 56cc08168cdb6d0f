"""Seeded synthetic inputs for the W4A16 linear layer.

This module only draws random numbers and puts them in the input containers the
layer consumes.  It holds none of the layer's arithmetic (no unpacking, no
dequantisation, no GEMM): both the CUDA path and the CPU oracle receive the
very same arrays from here, so neither side can influence the other's inputs.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: draw ``i`` of a stream is
``mix64(key + (i + 1) * GOLDEN_GAMMA)``, so any slice can be produced on its own.
Each tensor has its own stream (``key`` derived from the seed and a fixed stream
id), so changing one tensor's size never shifts another tensor's values.

Distributions (the workloads of the int4-weight linear layer pages):
  * q       uniform integers 0..15, one per byte, natural ``[N, K]`` order
  * scales  uniform in ``[lo, hi]`` drawn in float64, rounded (RNE) to the dtype
  * zeros   uniform nibbles 0..15, delivered already in the checkpoint container
            ``int32 [N/8, K/G]`` (8 zero points per word along N); since every
            nibble of a uniform 32-bit draw is itself uniform, a word is just one
            32-bit draw, so no packing arithmetic happens here
  * A       standard normal by Box-Muller in float64, rounded (RNE) to the dtype
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q = 1
STREAM_SCALES = 2
STREAM_ZEROS = 3
STREAM_A = 4

_CHUNK = 1 << 22  # draws per vectorised chunk (bounds temporary memory)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * GOLDEN_GAMMA
                         + np.uint64(stream)], dtype=np.uint64)
    return _mix64(base)[0]


def draws(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """64-bit draws ``start .. start+count-1`` of stream ``stream``."""
    key = stream_key(seed, stream)
    out = np.empty(count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for c0 in range(0, count, _CHUNK):
            n = min(_CHUNK, count - c0)
            idx = np.arange(start + c0 + 1, start + c0 + 1 + n, dtype=np.uint64)
            out[c0:c0 + n] = _mix64(key + idx * GOLDEN_GAMMA)
    return out


def uniform01(seed: int, stream: int, count: int) -> np.ndarray:
    """Doubles in [0, 1) from the top 53 bits of each draw."""
    d = draws(seed, stream, 0, count)
    return (d >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def nibbles(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` uniform integers 0..15 as uint8 (16 per 64-bit draw)."""
    nd = (count + 15) // 16
    d = draws(seed, stream, 0, nd)
    out = np.empty((nd, 16), dtype=np.uint8)
    for j in range(16):
        out[:, j] = ((d >> np.uint64(4 * j)) & np.uint64(15)).astype(np.uint8)
    return out.reshape(-1)[:count]


def words32(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` uniform 32-bit words as int32 (two per 64-bit draw)."""
    nd = (count + 1) // 2
    d = draws(seed, stream, 0, nd)
    lo = (d & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    hi = (d >> np.uint64(32)).astype(np.uint32)
    out = np.stack([lo, hi], axis=1).reshape(-1)[:count]
    return out.view(np.int32)


def normals(seed: int, stream: int, count: int) -> np.ndarray:
    """Standard normal doubles by Box-Muller (pairs from consecutive draws)."""
    npairs = (count + 1) // 2
    u = uniform01(seed, stream, 2 * npairs).reshape(npairs, 2)
    u1 = 1.0 - u[:, 0]  # (0, 1]: keeps log finite
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u[:, 1]
    z = np.stack([r * np.cos(t), r * np.sin(t)], axis=1).reshape(-1)
    return z[:count]


TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def to_dtype_bits(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 draws to float32, then (torch's RNE cast) to ``dtype``.

    Returns the uint16 bit patterns.  Both the CUDA path and the oracle consume
    exactly these bits, so how the draw was rounded does not affect parity.
    """
    x32 = np.ascontiguousarray(x64, dtype=np.float64).astype(np.float32)
    t = torch.from_numpy(x32).to(TORCH_DTYPES[dtype])
    return t.view(torch.int16).numpy().view(np.uint16).copy()


@dataclasses.dataclass(frozen=True)
class Problem:
    """One W4A16 linear-layer problem: ``C[M,N] = A[M,K] . dequant(W)^T``."""

    M: int
    N: int
    K: int
    group_size: int          # -1 (one group spanning K), 32, 64, 128 or 256
    qtype: str               # "uint4b8" (zero 8 implicit) or "uint4" (explicit zeros)
    dtype: str               # "fp16" or "bf16": activation = scale = output dtype
    scale_lo: float = 0.002
    scale_hi: float = 0.02
    seed: int = 0

    @property
    def g_eff(self) -> int:
        return self.K if self.group_size == -1 else self.group_size

    @property
    def ngroups(self) -> int:
        return self.K // self.g_eff


@dataclasses.dataclass
class Inputs:
    q: np.ndarray            # uint8 [N, K], values 0..15
    scales: np.ndarray       # uint16 bits [N, K/G_eff] of dtype
    zeros: np.ndarray | None  # int32 [N/8, K/G_eff] (8 nibbles per word along N) or None
    A: np.ndarray            # uint16 bits [M, K] of dtype


def make_scales(p: Problem) -> np.ndarray:
    ng = p.ngroups
    s64 = p.scale_lo + (p.scale_hi - p.scale_lo) * uniform01(p.seed, STREAM_SCALES, p.N * ng)
    return to_dtype_bits(s64, p.dtype).reshape(p.N, ng)


def make_zeros(p: Problem):
    if p.qtype != "uint4":
        return None
    if p.N % 8:
        raise ValueError("explicit zero points need N % 8 == 0")
    return words32(p.seed, STREAM_ZEROS, (p.N // 8) * p.ngroups).reshape(p.N // 8, p.ngroups)


def make_weights(p: Problem):
    q = nibbles(p.seed, STREAM_Q, p.N * p.K).reshape(p.N, p.K)
    return q, make_scales(p), make_zeros(p)


def make_activations(p: Problem) -> np.ndarray:
    a64 = normals(p.seed, STREAM_A, p.M * p.K)
    return to_dtype_bits(a64, p.dtype).reshape(p.M, p.K)


def make_inputs(p: Problem) -> Inputs:
    q, s, z = make_weights(p)
    return Inputs(q=q, scales=s, zeros=z, A=make_activations(p))


# Workloads of the int4-weight linear layer, named by what they are.
WORKLOADS = {
    # small single-token case (fp16, scales U[0.005, 0.02])
    "gemv_m1_k512_n512_g128_u4b8_fp16": [
        Problem(1, 512, 512, 128, "uint4b8", "fp16", 0.005, 0.02)],
    # decode GEMV on a 7B attention projection shape
    "decode_k4096_n4096_g128_u4b8_bf16": [
        Problem(m, 4096, 4096, 128, "uint4b8", "bf16") for m in (1, 4, 8)],
    # asymmetric (explicit zero points) g32, two MLP layers at M=16
    "zp_m16_g32_bf16_mlp_pair": [
        Problem(16, 11008, 4096, 32, "uint4", "bf16"),
        Problem(16, 4096, 11008, 32, "uint4", "bf16")],
    # prefill on an 8B MLP up-projection shape
    "prefill_m2048_k4096_n14336_g128_u4b8_bf16": [
        Problem(2048, 14336, 4096, 128, "uint4b8", "bf16")],
}


def crossover_sweep():
    """The 144-point sweep over M on a 70B MLP shape (K=8192, N=28672)."""
    pts = []
    for m in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 4096):
        for g in (-1, 64, 256):
            for qt in ("uint4b8", "uint4"):
                for dt in ("fp16", "bf16"):
                    pts.append(Problem(m, 28672, 8192, g, qt, dt))
    return pts
