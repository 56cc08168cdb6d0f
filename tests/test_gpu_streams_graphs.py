"""The C ABI driven the ways a caller drives a GPU: captured into a CUDA graph and
replayed, launched on a non-default stream (passed explicitly, or as torch's
current stream), and called from several host threads at once.

Every path is deterministic: split-K partials are summed in a fixed order and
no kernel uses atomics, so each of these runs must give the eager call's bits.
The eager results are checked against the oracle first.
"""

import dataclasses
import threading

import numpy as np
import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

from gpu_helpers import TOL, TORCH, B, DeviceWeight, assert_device_status_ok, to_dev_bits, to_host_bits

pytestmark = pytest.mark.gpu

# (M, N, K, G, qtype, dtype, path): the small-M kernel with an 8-way cluster
# split, the tensor-memory kernel with and without a split, the shared-memory
# fused kernel and the dense-copy kernel.
CASES = [
    (4, 4096, 4096, 128, "uint4b8", "bf16", "decode"),
    (16, 1024, 4096, 32, "uint4", "bf16", "auto"),
    (48, 2048, 2048, 64, "uint4b8", "fp16", "fused_tmem"),
    (200, 1024, 1024, 128, "uint4b8", "bf16", "fused_smem"),
    (300, 512, 1024, -1, "uint4", "fp16", "dense"),
]


class Layer:
    """One case's packed weight, its dense copy (dense path only) and a call."""

    def __init__(self, case, seed=0):
        M, N, K, G, qt, dt, path = case
        self.p = synth.Problem(M, N, K, G, qt, dt, seed=seed)
        self.path = path
        self.x = synth.make_inputs(self.p)
        self.w = DeviceWeight(self.p, self.x.q, self.x.scales, self.x.zeros)
        self.Wd = self.w.dequant() if path == "dense" else None

    def call(self, A, C, stream=None):
        p, w = self.p, self.w
        B().gemm_ex(A, w.Wq, w.scales, w.zeros, self.Wd, C, p.M, p.N, p.K, p.group_size, p.qtype,
                    p.dtype, self.path, stream=stream)

    def new_c(self):
        return torch.full((self.p.M, self.p.N), float("nan"), dtype=TORCH[self.p.dtype], device="cuda")

    def activations(self, seed):
        return to_dev_bits(synth.make_activations(dataclasses.replace(self.p, seed=seed)), self.p.dtype)

    def eager_bits(self, A):
        C = self.new_c()
        self.call(A, C)
        torch.cuda.synchronize()
        return to_host_bits(C)


def ids(c):
    return "x".join(map(str, c))


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_graph_replay_gives_the_eager_bits(case):
    L = Layer(case)
    p = L.p
    A = to_dev_bits(L.x.A, p.dtype)
    ref = L.eager_bits(A)
    err = orc.rel_error(orc.values(ref, p.dtype), orc.linear(L.x.A, L.x.q, L.x.scales, L.x.zeros,
                                                             p.group_size, p.dtype))
    assert err <= TOL[p.dtype], err
    assert np.array_equal(L.eager_bits(A), ref), "two eager calls differ"

    C = L.new_c()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.call(A, C)          # the binding launches on the capturing stream
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(C), ref)

    # the graph reads the live input buffer: new activations, same graph
    A.copy_(L.activations(seed=1))
    ref2 = L.eager_bits(A)
    assert not np.array_equal(ref2, ref)
    C.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(C), ref2)
    assert_device_status_ok()


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4]], ids=ids)
def test_non_default_stream(case):
    L = Layer(case)
    A = to_dev_bits(L.x.A, L.p.dtype)
    ref = L.eager_bits(A)
    C_current, C_explicit = L.new_c(), L.new_c()   # filled on the default stream ...
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())      # ... before s may write them
    with torch.cuda.stream(s):
        L.call(A, C_current)              # stream=None: torch's current stream, here s
    L.call(A, C_explicit, stream=s)       # the stream passed by the caller
    s.synchronize()
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(C_current), ref)
    assert np.array_equal(to_host_bits(C_explicit), ref)
    assert_device_status_ok()


def test_concurrent_host_threads():
    # One thread per case, each on its own stream and buffers, calling repeatedly
    # while the others do (the library's tensor-map and launch caches are shared),
    # plus a thread whose calls fail validation: its error message must stay its own.
    layers = [Layer(c) for c in CASES]
    As = [to_dev_bits(L.x.A, L.p.dtype) for L in layers]
    refs = [L.eager_bits(A) for L, A in zip(layers, As)]
    outs = [[L.new_c() for _ in range(2)] for L in layers]
    streams = [torch.cuda.Stream() for _ in layers]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    errors = []
    start = threading.Barrier(len(layers) + 1)
    reps = 24

    def work(i):
        try:
            start.wait()
            for r in range(reps):
                layers[i].call(As[i], outs[i][r % 2], stream=streams[i])
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append((i, repr(e)))

    def invalid():
        try:
            start.wait()
            L = layers[0]
            p = L.p
            C = L.new_c()
            for _ in range(reps):
                try:
                    B().gemm_ex(As[0], L.w.Wq, L.w.scales, L.w.zeros, None, C, p.M, p.N, p.K, 7,
                                p.qtype, p.dtype, "auto", stream=streams[0])
                    errors.append(("invalid", "group size 7 was accepted"))
                except B().W4A16Error as e:
                    if "group size" not in str(e):
                        errors.append(("invalid", f"another thread's message: {e}"))
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(("invalid", repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(layers))]
    threads.append(threading.Thread(target=invalid))
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a calling thread did not finish"
    torch.cuda.synchronize()
    assert not errors, errors
    for i, ref in enumerate(refs):
        for C in outs[i]:
            assert np.array_equal(to_host_bits(C), ref), CASES[i]
    assert_device_status_ok()
