"""GPU path against the CPU oracle, element by element, through the C ABI.

Pack and dequant must be bit-exact; GEMM output must satisfy
max|C - C_ref| / (max|C_ref| + 1e-6) <= 1e-2 (bf16) or 2e-3 (fp16).
Shapes span several tiles of every kernel and ragged tails in M, N and K.
"""

import numpy as np
import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

from gpu_helpers import TOL, B, DeviceWeight, assert_device_status_ok, run_gemm, to_dev_bits, to_host_bits, TORCH

pytestmark = pytest.mark.gpu

# (M, N, K, G, qtype, dtype)
SHAPES = [
    (1, 512, 512, 128, "uint4b8", "fp16"),
    (3, 200, 1024, 64, "uint4", "bf16"),
    (8, 384, 768, 32, "uint4", "fp16"),
    (13, 136, 2048, 128, "uint4b8", "bf16"),
    (32, 256, 1280, 256, "uint4", "bf16"),
    (64, 128, 512, -1, "uint4b8", "fp16"),
    (5, 64, 4112, -1, "uint4b8", "bf16"),      # K % 32 == 16
    (1, 8, 16, -1, "uint4", "fp16"),           # smallest legal layer (one group of 16)
    (2, 16, 32, -1, "uint4", "bf16"),          # one group of 32
    (300, 384, 512, 128, "uint4b8", "bf16"),
    (77, 200, 1088, 64, "uint4", "fp16"),
    (40, 136, 4112, -1, "uint4b8", "bf16"),
    (513, 1024, 2048, 32, "uint4", "bf16"),
    (129, 256, 1024, 256, "uint4", "fp16"),
    (12, 256, 1024, 32, "uint4", "bf16"),      # G = 32 between 9 and 16 tokens with zero points: fused kernel
    (13, 264, 2048, 32, "uint4b8", "bf16"),    # ... without them: small-M kernel, two token tiles
    (14, 200, 4112, -1, "uint4", "fp16"),      # two token tiles, a 16-value K tail in the last box
    (24, 136, 128, 32, "uint4", "bf16"),       # one MMA hand-off: the second issuer has none
    (48, 200, 64, -1, "uint4b8", "fp16"),      # one 64-wide block
]


def _problem(M, N, K, G, qt, dt, seed=0):
    return synth.Problem(M, N, K, G, qt, dt, seed=seed)


@pytest.fixture(scope="module")
def cases():
    out = {}
    for sh in SHAPES:
        p = _problem(*sh)
        x = synth.make_inputs(p)
        w_ref = orc.dequant(x.q, x.scales, x.zeros, p.group_size, p.dtype)
        out[sh] = (p, x, w_ref, orc.gemm(x.A, w_ref, p.dtype))
    return out


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_pack_is_bit_exact(cases, sh):
    p, x, _, _ = cases[sh]
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    torch.cuda.synchronize()
    assert np.array_equal(w.words(), orc.pack_q(x.q, w.ldq))
    # scale and zero sections are the inputs transposed, padded with zeros
    lds, ldz = (p.N + 7) // 8 * 8, (p.N // 8 + 3) // 4 * 4
    ng = p.ngroups
    sc = to_host_bits(w.buf[w.so: w.so + ng * lds * 2].view(TORCH[p.dtype])).reshape(ng, lds)
    assert np.array_equal(sc[:, :p.N], x.scales.T) and np.all(sc[:, p.N:] == 0)
    if x.zeros is not None:
        z = w.buf[w.zo: w.zo + ng * ldz * 4].view(torch.int32).cpu().numpy().reshape(ng, ldz)
        assert np.array_equal(z[:, :p.N // 8], x.zeros.T) and np.all(z[:, p.N // 8:] == 0)
    assert np.array_equal(orc.unpack_q(w.words(), p.K), x.q)


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_dequant_is_bit_exact(cases, sh):
    p, x, w_ref, _ = cases[sh]
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    got = to_host_bits(w.dequant())
    assert np.array_equal(got, w_ref)


def _paths_for(M):
    paths = ["fused_tmem", "fused_smem", "dense"]
    if M <= 64:
        paths.insert(0, "decode")
    return paths


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_parity_all_paths(cases, sh):
    p, x, _, C_ref = cases[sh]
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    Wd = w.dequant()
    for path in _paths_for(p.M) + ["auto"]:
        C = run_gemm(w, x.A, path=path, Wdense=Wd if path in ("dense",) else None)
        Cv = orc.values(C, p.dtype)
        assert np.all(np.isfinite(Cv)), path
        err = orc.rel_error(Cv, C_ref)
        assert err <= TOL[p.dtype], (path, err)
    assert_device_status_ok()


@pytest.mark.parametrize("path", ["decode", "fused", "dense"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_one_hot_activations_return_dequantised_weights_exactly(path, dtype):
    # C[m, n] = w[n, k_m] exactly: one product with 1.0 and one rounding of an
    # already representable value.
    M, N, K, G = 24, 256, 1024, 64
    p = _problem(M, N, K, G, "uint4", dtype)
    q, s, z = synth.make_weights(p)
    km = (np.arange(M) * 37 + 5) % K
    A = np.zeros((M, K), dtype=np.uint16)
    A[np.arange(M), km] = 0x3F80 if dtype == "bf16" else 0x3C00
    w = DeviceWeight(p, q, s, z)
    w_ref = orc.dequant(q, s, z, G, dtype)
    C = run_gemm(w, A, path=path, Wdense=w.dequant() if path == "dense" else None)
    assert np.array_equal(C, w_ref[:, km].T)


@pytest.mark.parametrize("path,M", [("decode", 16), ("fused_tmem", 16), ("fused_tmem", 40), ("fused_smem", 16),
                                    ("dense", 16)])
def test_integer_valued_gemm_is_exact(path, M):
    # scale 1, A in {-1, 0, 1}: every partial sum is an integer below 2^24, so the
    # fp32 accumulation is exact in any order (also split between the tensor-memory
    # kernel's two accumulators at 40 tokens) and C = rne_dtype(exact).
    N, K = 192, 512
    p = _problem(M, N, K, -1, "uint4b8", "bf16")
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    s = np.full((N, 1), 0x3F80, dtype=np.uint16)
    a_int = rng.integers(-1, 2, (M, K))
    A = orc.round_to(a_int.astype(np.float64), "bf16")
    w = DeviceWeight(p, q, s, None)
    C = run_gemm(w, A, path=path, Wdense=w.dequant() if path == "dense" else None)
    exact = (a_int @ (q.astype(np.int64) - 8).T).astype(np.float64)
    assert np.array_equal(C, orc.round_to(exact, "bf16"))


def test_uint4_with_zero_points_8_matches_uint4b8_on_gpu():
    p8 = _problem(8, 256, 1024, 128, "uint4b8", "bf16")
    q, s, _ = synth.make_weights(p8)
    A = synth.make_activations(p8)
    pz = _problem(8, 256, 1024, 128, "uint4", "bf16")
    zeros = np.full((256 // 8, 1024 // 128), 0x88888888, dtype=np.uint32).view(np.int32)
    a = run_gemm(DeviceWeight(p8, q, s, None), A)
    b = run_gemm(DeviceWeight(pz, q, s, zeros), A)
    assert np.array_equal(a, b)


def test_every_decode_m_up_to_64():
    N, K = 256, 1536
    p = _problem(64, N, K, 128, "uint4", "bf16")
    x = synth.make_inputs(p)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    C_ref = orc.linear(x.A, x.q, x.scales, x.zeros, 128, "bf16")
    for M in range(1, 65):
        C = run_gemm(w, x.A[:M], path="decode")
        assert orc.rel_error(orc.values(C, "bf16"), C_ref[:M]) <= TOL["bf16"], M


def test_every_fused_m_from_17_to_72():
    # 32- and 64-token tiles with two MMA issuers, an odd number of hand-offs
    # (17 blocks of 64) and the 128-token tile just above
    N, K = 136, 1088
    p = _problem(72, N, K, 64, "uint4", "bf16")
    x = synth.make_inputs(p)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    C_ref = orc.linear(x.A, x.q, x.scales, x.zeros, 64, "bf16")
    for M in range(17, 73):
        C = run_gemm(w, x.A[:M], path="fused_tmem")
        assert orc.rel_error(orc.values(C, "bf16"), C_ref[:M]) <= TOL["bf16"], M
    assert_device_status_ok()


def test_fused_whole_and_split_clusters():
    # 224 row tiles of 32 tokens on the GPU's SMs: clusters of two that take two
    # whole tiles next to clusters that split one tile's K (grid = 2 CTAs per SM).
    # (64-token tiles do so from K = 8192, through the activation ring: covered on
    # the full 70B layer by test_gpu_fullsize's sampled crossover test.)
    N, K, G = 28672, 1024, 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = _problem(64, N, K, G, "uint4", "bf16")
    x = synth.make_inputs(p)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    C_ref = orc.linear(x.A, x.q, x.scales, x.zeros, G, "bf16")
    for M in (17, 32, 33, 64):
        plan = B().launch_plan(M, N, K, G, "uint4", "bf16", "fused_tmem", False, sms)
        if M <= 32 and sms < N // 128 < 2 * sms:
            assert plan["k_split"] == 2 and plan["grid"] == 2 * sms
        C = run_gemm(w, x.A[:M], path="fused_tmem")
        assert orc.rel_error(orc.values(C, "bf16"), C_ref[:M]) <= TOL["bf16"], M
    assert_device_status_ok()


def test_outputs_outside_c_are_untouched():
    # C is written exactly over [M, N]: guard rows around it stay intact
    p = _problem(37, 200, 512, 64, "uint4", "fp16")
    x = synth.make_inputs(p)
    w = DeviceWeight(p, x.q, x.scales, x.zeros)
    for path in ("decode", "fused_tmem", "fused_smem"):
        big = torch.full((p.M + 2, p.N), 7.0, dtype=torch.float16, device="cuda")
        C = big[1:-1]
        A = to_dev_bits(x.A, "fp16")
        B().gemm_ex(A, w.Wq, w.scales, w.zeros, None, C, p.M, p.N, p.K, p.group_size, p.qtype,
                    p.dtype, path)
        torch.cuda.synchronize()
        assert torch.all(big[0] == 7.0) and torch.all(big[-1] == 7.0)
    assert_device_status_ok()
