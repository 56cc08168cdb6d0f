"""The benchmark's roofline accounting (host arithmetic, no GPU): algorithmic
bytes and FLOPs per layer call against figures worked out by hand from the
layouts - q N*K/2, scales N*ng*2, zero points (N/8)*ng*4, A M*K*2, C M*N*2 bytes;
2*M*N*K FLOPs - for each workload, and the rule that an ncu traffic figure is
used only while its kernel's sources are unchanged."""

import os

import pytest

import bench

# (M, N, K, G, zero points) -> bytes, worked by hand term by term
CASES = [
    ((1, 512, 512, 128, False), 131072 + 4096 + 1024 + 1024),                          # 137,216
    ((1, 4096, 4096, 128, False), 8388608 + 262144 + 8192 + 8192),                     # 8,667,136
    ((4, 4096, 4096, 128, False), 8388608 + 262144 + 32768 + 32768),                   # 8,716,288
    ((8, 4096, 4096, 128, False), 8388608 + 262144 + 65536 + 65536),                   # 8,781,824
    ((16, 11008, 4096, 32, True), 22544384 + 2818048 + 704512 + 131072 + 352256),      # 26,550,272
    ((2048, 14336, 4096, 128, False), 29360128 + 917504 + 16777216 + 58720256),        # 105,775,104
    ((1, 28672, 8192, 64, True), 117440512 + 7340032 + 1835008 + 16384 + 57344),       # 126,689,280
    ((1, 28672, 8192, -1, False), 117440512 + 57344 + 16384 + 57344),                  # one group per row
]


@pytest.mark.parametrize("case,want", CASES, ids=lambda c: str(c))
def test_algorithmic_bytes(case, want):
    assert bench.alg_bytes(*case) == want


def test_totals_of_the_named_workloads():
    assert bench.alg_bytes(1, 4096, 4096, 128, False) == 8_667_136
    assert bench.alg_bytes(16, 11008, 4096, 32, True) == 26_550_272
    assert bench.alg_bytes(2048, 14336, 4096, 128, False) == 105_775_104
    assert bench.alg_bytes(1, 28672, 8192, 64, True) == 126_689_280
    assert 2 * 2048 * 14336 * 4096 == 240_518_168_576          # prefill FLOPs
    assert 2 * 28672 * 8192 == 469_762_048                     # 70B MLP FLOPs per token


def test_weight_bytes_are_the_streamed_part():
    for (M, N, K, G, zp), want in CASES:
        assert bench.weight_bytes(N, K, G, zp) == want - M * K * 2 - M * N * 2


def test_traffic_is_used_only_for_unchanged_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "w4a16_int4_weight_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash(["k.cu"])
    (tmp_path / "profiles" / "k.md").write_text(
        f"source hash: {h}   (sha256)\n\ndram bytes per launch (read + write): 8761344\n")
    assert bench.profiled_traffic("k.md", ["k.cu"], 1) == 8761344
    assert bench.profiled_traffic("k.md", ["k.cu"], 4) == 4 * 8761344
    (csrc / "k.cu").write_text("kernel v2")          # the kernel changed since the capture
    assert bench.profiled_traffic("k.md", ["k.cu"], 1) is None
    assert bench.profiled_traffic("missing.md", ["k.cu"], 1) is None
    assert os.path.exists(tmp_path / "profiles" / "k.md")
