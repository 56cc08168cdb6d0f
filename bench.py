#!/usr/bin/env python
"""Benchmark of the W4A16 int4-weight linear layer on GB300.

Default workload: the 70B-MLP layer (K = 8192, N = 28672), group size 64,
uint4b8, bf16 activations, seeded synthetic weights and activations.  One step
runs the layer at every decode batch size M in {1, 2, 4, 8, 16} on each of two
distinct weight copies (2 x 125 MB > the 129 MB L2), so every launch streams
its weights from HBM.  `per_m` times the same layer at every M of the
crossover sweep (1 .. 4096) through the router: HBM-bound decode at small M,
tensor-bound prefill at large M.

Prints one JSON line (rank 0).  `value` is whole-job weight throughput
(packed q + scale bytes per second) of the decode points with inputs resident
in HBM, from CUDA events around K replays of a CUDA graph of one step; `e2e` is
the same metric through the C ABI called eagerly with the activations copied
from pinned host memory and the outputs copied back inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (the plain float64 definition, from
oracle/) on a bounded sample of the same workload.  With several GPUs
(torchrun) every rank runs its own replica of the workload (no data exchange;
weak scaling) and rank 0 reports the aggregate.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMM TFLOP/s and weight GB/s vs M; % of HBM / bf16 tensor roofline"
WORKLOAD = "mlp70b_k8192_n28672_g64_uint4b8_bf16_decode_m1_2_4_8_16"
MS = (1, 2, 4, 8, 16)                      # the decode points of one step
PER_M = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 4096)   # the "vs M" curve
N_, K_, G_ = 28672, 8192, 64
QTYPE, DTYPE = "uint4b8", "bf16"
LAYERS = 2                                 # distinct weight copies: 2 x 125 MB > L2
PER_M_PASSES = 4                           # passes over the copies in one "vs M" graph
L2_BYTES = 129 * 1024 * 1024


def weight_bytes(N, K, G, zp):
    ng = K // (K if G == -1 else G)
    return N * K // 2 + N * ng * 2 + ((N // 8) * ng * 4 if zp else 0)


def alg_bytes(M, N, K, G, zp):
    return weight_bytes(N, K, G, zp) + M * K * 2 + M * N * 2


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the prefill/zero-point side measurements")
    ap.add_argument("--profile-case", choices=["decode", "decode16", "decode_large", "decode_small", "zp", "mid", "mid32",
                                               "prefill", "prefill_smem", "dense", "dequant"],
                    help="only run `--reps` eager launches of one kernel (for ncu), then exit")
    ap.add_argument("--reps", type=int, default=8)
    ap.add_argument("--sweep", action="store_true",
                    help="time the 70B-MLP crossover sweep (12 M x 3 group sizes x 2 quant types x 2 dtypes) "
                         "through the router and print it as a table, then exit")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas only)
# ---------------------------------------------------------------------------
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:   # host-only rank plumbing (tests): the same barrier and reduction over gloo
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for ln in self.out.strip().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = set()
        for _, _, flags in rows:
            for nm, f in zip(names, flags):
                if f.lower() == "active":
                    seen.add(nm)
        # samples taken while the GPU was busy (clock above idle) describe the load
        busy = [r for r in rows if r[0] > 0.5 * r[1]] or rows
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(seen), "samples": len(rows)}


# ---------------------------------------------------------------------------
# ncu-derived DRAM traffic of the dominant kernel, if taken on the current source
# ---------------------------------------------------------------------------
def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "w4a16_int4_weight_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_name, sources, scale):
    """Bytes per launch from a profiles/ summary, or None if the kernel changed."""
    path = os.path.join(ROOT, "profiles", summary_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    mh = re.search(r"source hash:\s*([0-9a-f]{16})", text)
    mt = re.search(r"dram bytes per launch \(read \+ write\):\s*([0-9]+)", text)
    if not mh or not mt or mh.group(1) != kernel_source_hash(sources):
        return None
    return int(mt.group(1)) * scale


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline / reference arm)
# ---------------------------------------------------------------------------
def cpu_model():
    """The host CPU's model name (lscpu), for the baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


_ORACLE_INPUTS = {}
ORACLE_COLS = 2048   # output columns the oracle inputs are generated for


def oracle_inputs(layer):
    """Seeded inputs of the first ORACLE_COLS output columns of one layer of the
    workload (the generators are counter-based, so these are exactly the first
    rows of the full weight), generated once, outside any timed region."""
    if layer not in _ORACLE_INPUTS:
        import oracle as orc
        from w4a16_int4_weight_gb300 import inputs as synth
        p = synth.Problem(max(MS), ORACLE_COLS, K_, G_, QTYPE, DTYPE, seed=layer)
        q, s, _ = synth.make_weights(p)
        _ORACLE_INPUTS[layer] = (orc.pack_q(q), s, synth.make_activations(p))
    return _ORACLE_INPUTS[layer]


def oracle_sample(n_cols, layer=0):
    """Time the oracle on the first n_cols output columns of one layer, for each
    decode M of the step.  Returns (seconds, weight bytes processed)."""
    import oracle as orc
    words, s, A = oracle_inputs(layer)
    rows = np.arange(max(MS))
    total_t, total_b = 0.0, 0
    for M in MS:
        t0 = time.perf_counter()
        orc.linear_rows_packed(A, words[:n_cols], K_, s[:n_cols], None, rows[:M], G_, DTYPE)
        total_t += time.perf_counter() - t0
        total_b += weight_bytes(n_cols, K_, G_, False)
    return total_t, total_b


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle as orc
    orc.build()
    # size each step so that warmup + steps stay within about two minutes
    t, b = oracle_sample(64)
    per_step_budget = 100.0 / max(1, args.steps + args.warmup)
    n_cols = int(max(8, min(ORACLE_COLS, 64 * per_step_budget / max(t, 1e-6))) // 8 * 8)
    for _ in range(args.warmup):
        oracle_sample(n_cols)
    tt, bb = 0.0, 0
    for _ in range(args.steps):
        t, b = oracle_sample(n_cols)
        tt += t
        bb += b
    value = bb / tt / 1e9
    sample = (f"oracle (unpack -> dequant -> float64 GEMM) on output columns 0..{n_cols - 1} of one "
              f"layer for M = {', '.join(map(str, MS))} per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": WORKLOAD, "M": list(MS), "K": K_, "N": N_, "group_size": G_,
                   "qtype": QTYPE, "act_dtype": DTYPE},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def make_layers(torch, B, synth, n_layers, M_max, N, K, G, qtype, dtype, seed0=0):
    tdt = {"fp16": torch.float16, "bf16": torch.bfloat16}[dtype]
    layers = []
    tot, so, zo, _ = B.packed_layout(N, K, G, qtype, dtype)
    for l in range(n_layers):
        p = synth.Problem(M_max, N, K, G, qtype, dtype, seed=seed0 + l)
        q, s, z = synth.make_weights(p)
        qd = torch.from_numpy(q).cuda()
        sd = torch.from_numpy(s.view(np.int16)).cuda().view(tdt)
        zd = torch.from_numpy(z).cuda() if z is not None else None
        buf = torch.empty(tot, dtype=torch.uint8, device="cuda")
        B.pack(qd, sd, zd, buf, N, K, G, qtype, dtype)
        base = buf.data_ptr()
        layers.append((buf, base, base + so, base + zo if z is not None else None))
    torch.cuda.synchronize()
    return layers


def time_graph(torch, fn, reps, warmup):
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def extras(torch, B, synth, peaks):
    """Side measurements on the other workloads (not the headline): the decode
    GEMV on the 7B attention shape, the headline layer with fp16 activations,
    the prefill tcgen05 kernels (fused and dense), the dequant kernel and the
    zero-point decode pair."""
    hbm, tc_burst, _, kind = peaks
    out = {}
    tdt = torch.bfloat16
    # decode GEMV, K = N = 4096, G = 128, uint4b8, M = 1, 4, 8: 32 weight copies
    # (277 MB > L2), each M a CUDA graph of the 32 layers
    N, K, G, L = 4096, 4096, 128, 32
    lay = make_layers(torch, B, synth, L, 8, N, K, G, "uint4b8", "bf16", seed0=300)
    A = torch.randn(8, K, device="cuda").to(tdt)
    Cs = torch.empty(L, 8, N, dtype=tdt, device="cuda")
    for M in (1, 4, 8):
        def run_g(M=M):
            for l, (_, wq, sp, _) in enumerate(lay):
                B.gemm_ex(A, wq, sp, None, None, Cs[l], M, N, K, G, "uint4b8", "bf16", "auto",
                          static_weights=True)
        t = time_graph(torch, run_g, 300, 10) / L
        byts = alg_bytes(M, N, K, G, False)
        out[f"decode_m{M}_k4096_n4096_g128"] = {"us": t * 1e6, "gbs": byts / t / 1e9,
                                               "frac_of_hbm": byts / t / 1e9 / hbm}
    del lay, Cs
    torch.cuda.empty_cache()
    # the 70B MLP layer with fp16 activations (K = 8192, N = 28672, G = 64,
    # uint4b8), M = 1, 8, 16: two weight copies (250 MB > L2), each M a CUDA
    # graph of PER_M_PASSES passes over both, as the "vs M" curve
    N, K, G, L = 28672, 8192, 64, 2
    hdt = torch.float16
    lay = make_layers(torch, B, synth, L, 16, N, K, G, "uint4b8", "fp16", seed0=400)
    A = torch.randn(16, K, device="cuda").to(hdt)
    Cs = torch.empty(L, 16, N, dtype=hdt, device="cuda")
    for M in (1, 8, 16):
        def run_h(M=M):
            for _ in range(PER_M_PASSES):
                for l, (_, wq, sp, _) in enumerate(lay):
                    B.gemm_ex(A, wq, sp, None, None, Cs[l], M, N, K, G, "uint4b8", "fp16", "auto",
                              static_weights=True)
        t = time_graph(torch, run_h, 75, 5) / (L * PER_M_PASSES)
        byts = alg_bytes(M, N, K, G, False)
        out[f"decode_fp16_m{M}_k8192_n28672_g64"] = {"us": t * 1e6, "gbs": byts / t / 1e9,
                                                    "frac_of_hbm": byts / t / 1e9 / hbm}
    del lay, Cs
    torch.cuda.empty_cache()
    # prefill M=2048, K=4096, N=14336, G=128, uint4b8: 4 weight copies rotate
    M, N, K, G = 2048, 14336, 4096, 128
    lay = make_layers(torch, B, synth, 4, M, N, K, G, "uint4b8", "bf16", seed0=100)
    A = torch.randn(M, K, device="cuda").to(tdt)
    Cs = [torch.empty(M, N, dtype=tdt, device="cuda") for _ in lay]
    dense = []
    for (_, wq, sp, _) in lay:
        W = torch.empty(N, K, dtype=tdt, device="cuda")
        B.dequant(wq, sp, None, W, N, K, G, "uint4b8", "bf16")
        dense.append(W)
    flops = 2.0 * M * N * K

    def run(path):
        for i, (_, wq, sp, _) in enumerate(lay):
            B.gemm_ex(A, wq, sp, None, dense[i] if path == "dense" else None, Cs[i], M, N, K, G,
                      "uint4b8", "bf16", path)
    for path in ("fused_tmem", "fused_smem", "dense"):
        t = time_graph(torch, lambda: run(path), 10, 3) / len(lay)
        out[f"prefill_{path}_m2048_k4096_n14336"] = {
            "tflops": flops / t / 1e12, "us": t * 1e6,
            "frac_of_bf16_peak": flops / t / 1e12 / tc_burst, "peak_kind": kind}
    # dequant kernel on the same layer: HBM-bound (write 2 B, read 0.5 B per weight)
    (_, wq, sp, _) = lay[0]

    def deq():
        for i, (_, wq_, sp_, _) in enumerate(lay):
            B.dequant(wq_, sp_, None, dense[i], N, K, G, "uint4b8", "bf16")
    t = time_graph(torch, deq, 10, 3) / len(lay)
    byts = weight_bytes(N, K, G, False) + N * K * 2
    out["dequant_k4096_n14336"] = {"gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm}
    del lay, dense, Cs
    torch.cuda.empty_cache()
    # zero-point decode pair: M=16, G=32, uint4, K/N = 4096/11008 and 11008/4096
    for (K, N) in ((4096, 11008), (11008, 4096)):
        M, G = 16, 32
        lay = make_layers(torch, B, synth, 8, M, N, K, G, "uint4", "bf16", seed0=200)
        A = torch.randn(M, K, device="cuda").to(tdt)
        C = torch.empty(M, N, dtype=tdt, device="cuda")

        def run_zp():
            for (_, wq, sp, zp) in lay:
                B.gemm_ex(A, wq, sp, zp, None, C, M, N, K, G, "uint4", "bf16", "auto",
                          static_weights=True)
        t = time_graph(torch, run_zp, 200, 10) / len(lay)
        byts = alg_bytes(M, N, K, G, True)
        out[f"decode_zp_m16_g32_k{K}_n{N}"] = {"gbs": byts / t / 1e9, "frac_of_hbm": byts / t / 1e9 / hbm,
                                               "us": t * 1e6}
        del lay
        torch.cuda.empty_cache()
    return out


def profile_case(args):
    """Eager launches of one kernel on its workload, nothing timed (an ncu target)."""
    import torch
    torch.cuda.set_device(0)
    from w4a16_int4_weight_gb300 import build as wbuild
    wbuild.build()
    from w4a16_int4_weight_gb300 import binding as B
    from w4a16_int4_weight_gb300 import inputs as synth
    tdt = torch.bfloat16
    c = args.profile_case
    if c in ("decode", "decode16", "decode_large", "decode_small", "zp", "mid", "mid32"):
        M, N, K, G, qt = {"decode": (8, N_, K_, G_, QTYPE),
                          "decode16": (16, N_, K_, G_, QTYPE),
                          "decode_large": (1, 28672, 8192, 64, QTYPE),
                          "decode_small": (8, 4096, 4096, 128, QTYPE),
                          "zp": (16, 11008, 4096, 32, "uint4"),
                          "mid": (64, 28672, 8192, 64, QTYPE),
                          "mid32": (32, 28672, 8192, 64, QTYPE)}[c]
        lay = make_layers(torch, B, synth, 4, M, N, K, G, qt, "bf16")
        A = torch.randn(M, K, device="cuda").to(tdt)
        C = torch.empty(M, N, dtype=tdt, device="cuda")
        for r in range(args.reps):
            _, wq, sp, zp = lay[r % len(lay)]
            B.gemm(A, wq, sp, zp, C, M, N, K, G, qt, "bf16")
    else:
        M, N, K, G = 2048, 14336, 4096, 128
        lay = make_layers(torch, B, synth, 1, M, N, K, G, "uint4b8", "bf16", seed0=100)
        _, wq, sp, _ = lay[0]
        A = torch.randn(M, K, device="cuda").to(tdt)
        C = torch.empty(M, N, dtype=tdt, device="cuda")
        W = torch.empty(N, K, dtype=tdt, device="cuda")
        B.dequant(wq, sp, None, W, N, K, G, "uint4b8", "bf16")
        for _ in range(args.reps):
            if c == "dequant":
                B.dequant(wq, sp, None, W, N, K, G, "uint4b8", "bf16")
            else:
                B.gemm_ex(A, wq, sp, None, W if c == "dense" else None, C, M, N, K, G, "uint4b8",
                          "bf16", {"dense": "dense", "prefill": "fused_tmem", "prefill_smem": "fused_smem"}[c])
    torch.cuda.synchronize()
    code, site = B.device_status()
    print(f"profile case {c}: {args.reps} launches, device status {code}")
    return 0 if code == 0 else 1


SWEEP_M = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 4096)
SWEEP_N, SWEEP_K = 28672, 8192


def sweep(args):
    """Crossover sweep on the 70B MLP shape (K = 8192, N = 28672): every M, group
    size, quant type and dtype of the workload, each point the routed layer
    (w4a16_gemm_ex, path AUTO, static weights) on two weight copies (> L2 in
    all), CUDA-graph replay (up to 128 tokens a graph of PER_M_PASSES passes over
    the copies), CUDA events.  Prints a markdown table."""
    import torch
    torch.cuda.set_device(0)
    from w4a16_int4_weight_gb300 import build as wbuild
    wbuild.build()
    from w4a16_int4_weight_gb300 import binding as B
    from w4a16_int4_weight_gb300 import inputs as synth
    hbm_peak, tc_peak, _, peak_kind = measured_peaks()
    N, K, copies = SWEEP_N, SWEEP_K, 2
    names = {v: k for k, v in B.PATHS.items()}
    q_dev = [torch.from_numpy(synth.make_weights(synth.Problem(1, N, K, 64, "uint4b8", "bf16", seed=c))[0]).cuda()
             for c in range(copies)]
    print(f"Crossover sweep, K = {K}, N = {N}; peaks ({peak_kind}): HBM {hbm_peak:.0f} GB/s, "
          f"bf16 {tc_peak:.0f} TFLOP/s; t* = max(algorithmic bytes / HBM, 2MNK / bf16 peak)\n")
    print("| G | qtype | dtype | M | path | us | TFLOP/s | weight GB/s | % HBM | % bf16 | t*/t |")
    print("|---|---|---|---|---|---|---|---|---|---|---|")
    for dt in ("bf16", "fp16"):
        tdt = {"fp16": torch.float16, "bf16": torch.bfloat16}[dt]
        A = torch.from_numpy(synth.make_activations(
            synth.Problem(max(SWEEP_M), N, K, 64, "uint4b8", dt, seed=7)).view(np.int16)).cuda().view(tdt)
        C = torch.empty(max(SWEEP_M), N, dtype=tdt, device="cuda")
        for G in (-1, 64, 256):
            for qt in ("uint4b8", "uint4"):
                tot, so, zo, _ = B.packed_layout(N, K, G, qt, dt)
                bufs = []
                for c in range(copies):
                    p = synth.Problem(1, N, K, G, qt, dt, seed=c)
                    s = torch.from_numpy(synth.make_scales(p).view(np.int16)).cuda().view(tdt)
                    z = synth.make_zeros(p)
                    zd = torch.from_numpy(z).cuda() if z is not None else None
                    buf = torch.empty(tot, dtype=torch.uint8, device="cuda")
                    B.pack(q_dev[c], s, zd, buf, N, K, G, qt, dt)
                    base = buf.data_ptr()
                    bufs.append((buf, base, base + so, base + zo if zd is not None else None))
                torch.cuda.synchronize()
                zp = qt == "uint4"
                for M in SWEEP_M:
                    passes = PER_M_PASSES if M <= 128 else 1   # as the benchmark's "vs M" curve

                    def run(M=M, passes=passes):
                        for _ in range(passes):
                            for (_, wq, sp, zpp) in bufs:
                                B.gemm_ex(A, wq, sp, zpp, None, C, M, N, K, G, qt, dt, "auto",
                                          static_weights=True)
                    reps = 8 if M <= 128 else 10 if M <= 512 else 3
                    t = time_graph(torch, run, reps, 2) / (copies * passes)
                    fl = 2.0 * M * N * K
                    ab = alg_bytes(M, N, K, G, zp)
                    t_star = max(ab / (hbm_peak * 1e9), fl / (tc_peak * 1e12))
                    print(f"| {G} | {qt} | {dt} | {M} | {names.get(B.route(M, N, K, G, qt, dt), '?')} | "
                          f"{t * 1e6:.1f} | {fl / t / 1e12:.0f} | {weight_bytes(N, K, G, zp) / t / 1e9:.0f} | "
                          f"{100 * ab / t / 1e9 / hbm_peak:.0f} | {100 * fl / t / 1e12 / tc_peak:.0f} | "
                          f"{t_star / t:.2f} |", flush=True)
                del bufs
                torch.cuda.empty_cache()
    code, _ = B.device_status()
    print(f"\ndevice status {code}")
    return 0 if code == 0 else 1


def main():
    args = parse()
    if args.profile_case:
        return profile_case(args)
    if args.sweep:
        return sweep(args)
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        return run_reference(args, world, rank)

    import torch
    world, rank, local = dist_setup()
    from w4a16_int4_weight_gb300 import build as wbuild
    if rank == 0 or not os.path.exists(wbuild.LIB):
        wbuild.build()
    barrier(world)
    from w4a16_int4_weight_gb300 import binding as B
    from w4a16_int4_weight_gb300 import inputs as synth

    peaks = measured_peaks()
    hbm_peak, tc_peak, _, peak_kind = peaks
    tdt = torch.bfloat16
    mmax = max(PER_M)
    layers = make_layers(torch, B, synth, LAYERS, 1, N_, K_, G_, QTYPE, DTYPE)
    A_host = torch.from_numpy(synth.make_activations(
        synth.Problem(mmax, N_, K_, G_, QTYPE, DTYPE, seed=7)).view(np.int16)).view(tdt)
    A_dev = A_host.cuda()
    C_dev = {M: torch.empty(LAYERS, M, N_, dtype=tdt, device="cuda") for M in MS}
    C_big = torch.empty(LAYERS, mmax, N_, dtype=tdt, device="cuda")

    # the packed weights are written once before timing and then only read, so
    # the layer is called with the static-weights promise (W4A16_OPT_STATIC_WEIGHTS);
    # each layer's output view is made once, as a serving loop holds its buffers
    C_view = {M: [C_dev[M][l] for l in range(LAYERS)] for M in MS}

    def gemm(M, l, wq, sp, C=None):
        B.gemm_ex(A_dev, wq, sp, None, None, C_view[M][l] if C is None else C, M, N_, K_, G_, QTYPE,
                  DTYPE, "auto", static_weights=True)

    def step():
        for M in MS:
            for l, (_, wq, sp, _) in enumerate(layers):
                gemm(M, l, wq, sp)

    launches_per_step = len(MS) * LAYERS
    wbytes_step = launches_per_step * weight_bytes(N_, K_, G_, False)
    abytes_step = LAYERS * sum(alg_bytes(M, N_, K_, G_, False) for M in MS)
    flops_step = LAYERS * sum(2.0 * M * N_ * K_ for M in MS)

    # ---- device-resident timing: CUDA graph of one step, K replays ----
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    step()   # eager warm-up of every kernel instantiation before capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    gpu_uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    gpu_id = gpu_uuid if gpu_uuid.startswith("GPU-") else f"GPU-{gpu_uuid}"
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    t_dev = e0.elapsed_time(e1) / 1e3
    t_max = max_over_ranks(t_dev, world)
    ms_per_step = 1e3 * t_max / args.steps
    value = world * args.steps * wbytes_step / t_max / 1e9

    # ---- the "vs M" curve: every M of the sweep through the router ----
    names = {v: k for k, v in B.PATHS.items()}
    per_m = {}
    for M in PER_M:
        # up to 128 tokens a graph replays PER_M_PASSES passes over both copies:
        # a launch then follows another one as in the step (the first launch of
        # a replay cannot overlap its predecessor); larger M one pass
        passes = PER_M_PASSES if M <= 128 else 1

        def one_m(M=M, passes=passes):
            for _ in range(passes):
                for l, (_, wq, sp, _) in enumerate(layers):
                    gemm(M, l, wq, sp, C_big[l] if M not in C_view else None)
        reps = 50 if M <= 64 else 30 if M <= 512 else 5
        t = time_graph(torch, one_m, reps, 3) / (LAYERS * passes)
        ab = alg_bytes(M, N_, K_, G_, False)
        fl = 2.0 * M * N_ * K_
        t_star = max(ab / (hbm_peak * 1e9), fl / (tc_peak * 1e12))
        per_m[str(M)] = {"path": names.get(B.route(M, N_, K_, G_, QTYPE, DTYPE), "?"),
                         "us_per_launch": t * 1e6,
                         "weight_gbs": weight_bytes(N_, K_, G_, False) / t / 1e9,
                         "alg_gbs": ab / t / 1e9, "tflops": fl / t / 1e12,
                         "frac_of_hbm": ab / t / 1e9 / hbm_peak,
                         "frac_of_bf16": fl / t / 1e12 / tc_peak, "t_star_over_t": t_star / t}

    # spread of single steps: 200 graph replays, each between its own events
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(200)]
    for a, b in evs:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    step_ms = sorted(a.elapsed_time(b) for a, b in evs)
    step_spread = {"steps": len(step_ms), "p10_ms": step_ms[len(step_ms) // 10],
                   "p50_ms": step_ms[len(step_ms) // 2], "p90_ms": step_ms[(9 * len(step_ms)) // 10]}

    # ---- end to end through the C ABI: host activations in, host outputs out ----
    # Each step copies every M's activations in from pinned host memory and every
    # output back.  Two sets of device activations and outputs alternate between
    # steps; input and output copies run on two more streams, ordered against the
    # layer calls by events: a step's input copies wait until the calls of the
    # step before last (the set's last readers) have finished, its calls wait for
    # its inputs and for that step's output copies, and its output copies wait
    # for its calls.  A step's copies then overlap the neighbouring steps' calls,
    # as a serving loop overlaps them, and the calls of one step follow each
    # other with no wait between them; every copy of the timed steps starts
    # after the start event and ends before the stop event.
    A_pin = {M: A_host[:M].clone().pin_memory() for M in MS}
    C_pin = {M: torch.empty(LAYERS, M, N_, dtype=tdt).pin_memory() for M in MS}
    h2d = sum(A_pin[M].numel() * 2 for M in MS)
    d2h = sum(C_pin[M].numel() * 2 for M in MS)
    e2e_steps = max(1, min(args.steps, 300))
    A_in = [{M: torch.empty(M, K_, dtype=tdt, device="cuda") for M in MS} for _ in range(2)]
    C_set = [C_dev, {M: torch.empty(LAYERS, M, N_, dtype=tdt, device="cuda") for M in MS}]
    C_set_view = [{M: [C_set[b][M][l] for l in range(LAYERS)] for M in MS} for b in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # a set's inputs copied
    ev_done = [torch.cuda.Event() for _ in range(2)]    # a set's layer calls finished
    ev_out = [torch.cuda.Event() for _ in range(2)]     # a set's outputs copied back
    ev_start = torch.cuda.Event()
    cur = [0]

    def e2e_step():
        b = cur[0]
        cur[0] ^= 1
        s_in.wait_event(ev_done[b])
        with torch.cuda.stream(s_in):
            for M in MS:
                A_in[b][M].copy_(A_pin[M], non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])
        for M in MS:
            for l, (_, wq, sp, _) in enumerate(layers):
                B.gemm_ex(A_in[b][M], wq, sp, None, None, C_set_view[b][M][l], M, N_, K_, G_, QTYPE, DTYPE,
                          "auto", static_weights=True)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            for M in MS:
                C_pin[M].copy_(C_set[b][M], non_blocking=True)
        ev_out[b].record(s_out)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    ev_start.record(stream)
    s_in.wait_event(ev_start)
    s_out.wait_event(ev_start)
    for _ in range(e2e_steps):
        e2e_step()
    stream.wait_stream(s_out)   # the last outputs are back before the clock stops
    stream.wait_stream(s_in)
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = world * e2e_steps * wbytes_step / t_e2e / 1e9

    extra = {}
    if rank == 0 and not args.no_extras:
        del C_big
        torch.cuda.empty_cache()
        extra = extras(torch, B, synth, peaks)

    # roofline of the dominant kernel (the small-M kernel: every launch in the step)
    t_launch = t_dev / (args.steps * launches_per_step)
    achieved = (abytes_step / launches_per_step) / t_launch / 1e9
    traffic = profiled_traffic("decode_kernel_m1_k8192_n28672.md",
                               ["decode_kernel.cuh", "decode.cu", "common.cuh"], 1)

    cpu = None
    if rank == 0:
        import oracle as orc
        orc.build()
        # bounded sample: the oracle on the first output columns of the layer for
        # every decode M of the step, until about 10 s of CPU time
        tt, bb, ns = 0.0, 0, 0
        while tt < 10.0 and ns < 200:
            t, b = oracle_sample(512, layer=ns % 2)
            tt += t
            bb += b
            ns += 1
        cpu = {"value": bb / tt / 1e9, "unit": "GB/s", "cores": orc.num_threads(), "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{ns} passes over output columns 0..511 of the layer (2 weight copies), "
                         f"M = {', '.join(map(str, MS))} each (unpack -> dequant -> float64 GEMM), "
                         f"{tt:.1f} s of CPU time"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded SplitMix64 weights and activations)",
            "config": {"workload": WORKLOAD, "M": list(MS), "K": K_, "N": N_, "group_size": G_,
                       "qtype": QTYPE, "act_dtype": DTYPE, "weight_copies": LAYERS,
                       "l2": f"inputs larger than L2: {LAYERS} distinct weight copies, "
                             f"{LAYERS * weight_bytes(N_, K_, G_, False) / 1e6:.0f} MB per pass",
                       "timing": "CUDA graph of one step replayed K times, CUDA events",
                       "call": "w4a16_gemm_ex(path=auto | W4A16_OPT_STATIC_WEIGHTS)",
                       "per_m": f"the same layer at every M of the crossover sweep: a CUDA graph of "
                                f"{PER_M_PASSES} passes over both copies up to 128 tokens, one pass above",
                       "parallelism": f"replicas x{world}"},
            "tflops": world * args.steps * flops_step / t_max / 1e12,
            "alg_gbs": world * args.steps * abytes_step / t_max / 1e9,
            "per_m": per_m,
            "step_spread": step_spread,
            "gpu_launches": args.steps * launches_per_step,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic,
                         "peak_kind": peak_kind, "kernel": "decode_kernel"},
            "roofline_prefill": {"bound": "tensor", "achieved": per_m["4096"]["tflops"], "peak": tc_peak,
                                 "unit": "TFLOP/s", "frac": per_m["4096"]["frac_of_bf16"],
                                 "peak_kind": peak_kind, "kernel": per_m["4096"]["path"], "M": 4096},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "clocks": clk.summary(),
            "extras": extra,
        }
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
