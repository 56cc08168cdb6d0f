"""Parity in the launch configuration the benchmark times: 4096 x 4096 layers
(G = 128, uint4b8, bf16) called back to back with the static-weights promise
(W4A16_OPT_STATIC_WEIGHTS: each kernel fetches its weights before the previous
kernel in the stream has finished, under programmatic dependent launch) and
replayed from one CUDA graph.

The layers are chained, as in a model: layer l + 1 reads layer l's output as its
activations, and every output is reset to NaN before each replay, so an
activation read that ran ahead of the previous kernel's completion would see NaN.
Each layer is checked against the oracle on the GPU's own input bits (every
token row, or 16 sampled rows at 2048 tokens).  20480 x 20480 layers at 32 and
64 tokens run the same way on the tensor-memory kernel's mixed whole/split
cluster grids (2 sampled rows per layer).
"""

import numpy as np
import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

from gpu_helpers import TOL, B, DeviceWeight, assert_device_status_ok, to_dev_bits, to_host_bits

pytestmark = pytest.mark.gpu

N = K = 4096
G, QT, DT = 128, "uint4b8", "bf16"
LAYERS = 6


@pytest.mark.parametrize("M", [1, 4, 8, 64, 2048])
def test_chained_layers_static_weights_graph_replay(M):
    probs = [synth.Problem(M, N, K, G, QT, DT, seed=s) for s in range(LAYERS)]
    xs = [synth.make_weights(p) for p in probs]
    ws = [DeviceWeight(p, q, s, z) for p, (q, s, z) in zip(probs, xs)]
    a0_bits = synth.make_activations(synth.Problem(M, N, K, G, QT, DT, seed=7))
    A0 = to_dev_bits(a0_bits, DT)
    Cs = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(LAYERS)]

    def step():
        a = A0
        for w, C in zip(ws, Cs):
            B().gemm_ex(a, w.Wq, w.scales, None, None, C, M, N, K, G, QT, DT, "auto",
                        static_weights=True)
            a = C

    step()                       # eager warm-up of the instantiations, as the benchmark does
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        for C in Cs:
            C.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert_device_status_ok()

    rows = np.arange(M) if M <= 64 else np.random.default_rng(11).choice(M, 16, replace=False)
    a_bits = a0_bits[rows]
    for l, ((q, s, _), C) in enumerate(zip(xs, Cs)):
        got = to_host_bits(C)[rows]
        ref = orc.linear(np.ascontiguousarray(a_bits), q, s, None, G, DT)
        err = orc.rel_error(orc.values(got, DT), ref)
        assert err <= TOL[DT], (l, err)
        a_bits = got             # the next layer's activations: this layer's output bits


@pytest.mark.parametrize("M", [32, 64])
def test_chained_layers_mixed_clusters_graph_replay(M):
    # 20480 x 20480 layers: 160 row tiles, between one and two per SM, so the
    # tensor-memory kernel runs clusters that take two whole tiles next to
    # clusters that split one tile's K (at 64 tokens through the activation ring),
    # chained and replayed from a graph like the 4096 x 4096 layers above
    n = k = 20480
    layers = 3
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = B().launch_plan(M, n, k, G, QT, DT, "auto", False, sms)
    assert plan["path"] == "fused_tmem"
    if sms < n // 128 < 2 * sms:
        assert (plan["k_split"], plan["grid"]) == (2, 2 * sms)
    probs = [synth.Problem(M, n, k, G, QT, DT, seed=s) for s in range(layers)]
    xs = [synth.make_weights(p) for p in probs]
    ws = [DeviceWeight(p, q, s, z) for p, (q, s, z) in zip(probs, xs)]
    a0_bits = synth.make_activations(synth.Problem(M, n, k, G, QT, DT, seed=7))
    A0 = to_dev_bits(a0_bits, DT)
    Cs = [torch.empty(M, n, dtype=torch.bfloat16, device="cuda") for _ in range(layers)]

    def step():
        a = A0
        for w, C in zip(ws, Cs):
            B().gemm_ex(a, w.Wq, w.scales, None, None, C, M, n, k, G, QT, DT, "auto", static_weights=True)
            a = C

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        for C in Cs:
            C.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert_device_status_ok()

    rows = np.array([0, M - 1])
    a_bits = a0_bits[rows]
    for l, ((q, s, _), C) in enumerate(zip(xs, Cs)):
        got = to_host_bits(C)[rows]
        ref = orc.linear(np.ascontiguousarray(a_bits), q, s, None, G, DT)
        err = orc.rel_error(orc.values(got, DT), ref)
        assert err <= TOL[DT], (l, err)
        a_bits = got
    del ws
    torch.cuda.empty_cache()
