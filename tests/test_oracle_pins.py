"""Pins of the CPU oracle against values and identities fixed outside it.

Every oracle routine is checked against something other than itself: numbers
the pages print (or that follow by hand from a formula they print, with the
working in tests/golden), library routines (numpy's float64->float16 cast,
torch's float32->bfloat16 cast and float64 matmul), exact special cases and a
brute-force Python loop.  The cases are chosen so that a dropped term, a wrong
sign, a wrong group or row index or a transposed operand fails at least one.
"""

import itertools
import os

import numpy as np
import pytest
import torch

import oracle as orc
from w4a16_int4_weight_gb300 import inputs as synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# --------------------------------------------------------------------------
# RNE converters
# --------------------------------------------------------------------------

def _random_doubles(n, seed, lo_exp, hi_exp):
    rng = np.random.default_rng(seed)
    mant = rng.random(n) + 1.0
    ex = rng.integers(lo_exp, hi_exp, n)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return sign * np.ldexp(mant, ex)


def test_fp16_rounding_matches_numpy_on_random_doubles():
    # numpy converts float64 -> float16 directly with round-to-nearest-even.
    x = _random_doubles(1_000_000, 1, -30, 18)  # subnormals .. overflow
    got = orc.round_to(x, "fp16")
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounding_matches_torch_on_float32_values():
    # torch casts float32 -> bfloat16 with RNE; float32 inputs make it a single rounding.
    x = _random_doubles(1_000_000, 2, -140, 128).astype(np.float32)
    got = orc.round_to(x.astype(np.float64), "bf16")
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rounding_is_nearest_with_ties_to_even(dtype):
    # Property from the definition of RNE, for arbitrary float64 inputs.
    lo, hi = (-26, 15) if dtype == "fp16" else (-134, 127)
    x = _random_doubles(200_000, 3, lo, hi)
    # add exact ties: midpoints between neighbouring representable values
    base = orc.round_to(x[:1000], dtype).astype(np.int64)
    nxt = (base + 1) & 0xFFFF
    v0 = orc.values(base.astype(np.uint16), dtype)
    v1 = orc.values(nxt.astype(np.uint16), dtype)
    ok = np.isfinite(v0) & np.isfinite(v1) & (np.sign(v0) == np.sign(v1))
    x = np.concatenate([x, ((v0 + v1) / 2)[ok]])
    r = orc.round_to(x, dtype).astype(np.int64)
    v = orc.values(r.astype(np.uint16), dtype)
    assert np.all(np.isfinite(v))
    mag = r & 0x7FFF
    up = orc.values(((r & 0x8000) | np.minimum(mag + 1, 0x7FFF)).astype(np.uint16), dtype)
    dn = orc.values(((r & 0x8000) | np.maximum(mag - 1, 0)).astype(np.uint16), dtype)
    d = np.abs(x - v)
    assert np.all(d <= np.abs(x - up))
    assert np.all(d <= np.abs(x - dn))
    tie = (d == np.abs(x - up)) | ((d == np.abs(x - dn)) & (mag > 0))
    assert np.all((mag[tie] & 1) == 0)


def test_rounding_boundary_cases():
    r16 = lambda v: int(orc.round_to(np.array([v]), "fp16")[0])
    rb = lambda v: int(orc.round_to(np.array([v]), "bf16")[0])
    # fp16
    assert r16(65504.0) == 0x7BFF            # max normal
    assert r16(65519.99) == 0x7BFF
    assert r16(65520.0) == 0x7C00            # halfway to 2^16 rounds to even -> inf
    assert r16(2.0 ** -24) == 0x0001         # min subnormal
    assert r16(2.0 ** -25) == 0x0000         # tie with 0 -> even (0)
    assert r16(1.5 * 2.0 ** -25) == 0x0001
    assert r16(2.0 ** -14) == 0x0400         # min normal
    assert r16(1.0 + 2.0 ** -11) == 0x3C00   # tie -> even
    assert r16(1.0 + 3 * 2.0 ** -11) == 0x3C02
    assert r16(-0.0) == 0x8000
    assert r16(float("inf")) == 0x7C00 and r16(float("-inf")) == 0xFC00
    assert (r16(float("nan")) & 0x7C00) == 0x7C00 and (r16(float("nan")) & 0x3FF)
    # bf16
    assert rb(1.0) == 0x3F80
    assert rb(1.0 + 2.0 ** -8) == 0x3F80     # tie -> even
    assert rb(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert rb(2.0 ** -133) == 0x0001         # min subnormal
    assert rb(2.0 ** -134) == 0x0000         # tie with 0 -> even
    assert rb(3.3895313892515355e38) == 0x7F7F   # max finite
    assert rb(3.4e38) == 0x7F80                  # beyond the halfway point -> inf
    assert rb(-2.0) == 0xC000


def test_value_decoders_against_libraries():
    bits = np.arange(0, 1 << 16, dtype=np.uint16)
    f16 = orc.values(bits, "fp16")
    ref16 = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref16)
    assert np.array_equal(f16[fin], ref16[fin])
    assert np.array_equal(np.isnan(f16), np.isnan(ref16))
    b16 = orc.values(bits, "bf16")
    refb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    fin = np.isfinite(refb)
    assert np.array_equal(b16[fin], refb[fin])
    assert np.array_equal(np.isnan(b16), np.isnan(refb))


# --------------------------------------------------------------------------
# Packed words
# --------------------------------------------------------------------------

def test_exllama_example_word_and_shift_table():
    g = {ln[0]: ln[1:] for ln in _read_lines("exllama_word.txt")}
    vals = np.array([[int(v) for v in g["values"]]], dtype=np.uint8)
    words = orc.pack_q(vals)
    assert words.shape == (1, 4)              # K/8 = 1 word, padded to 4
    assert int(words[0, 0]) == int(g["word"][0], 16)
    assert list(words[0, 1:]) == [0, 0, 0]
    assert orc.shift_table() == [int(s) for s in g["shifts"]]


def test_pack_places_each_value_by_itself():
    # a single nonzero nibble in K-position i lands at its table shift only
    shifts = [int(s) for s in dict((ln[0], ln[1:]) for ln in _read_lines("exllama_word.txt"))["shifts"]]
    for i in range(8):
        for v in (1, 7, 15):
            q = np.zeros((1, 8), dtype=np.uint8)
            q[0, i] = v
            assert int(orc.pack_q(q)[0, 0]) == v << shifts[i]


def test_pack_unpack_round_trip_exhaustive_small():
    N, K = 16, 48
    q = np.array([[(n + k) % 16 for k in range(K)] for n in range(N)], dtype=np.uint8)
    w = orc.pack_q(q)
    assert w.shape == (N, 8)                  # K/8 = 6 -> pitch 8 words
    assert np.all(w[:, 6:] == 0)
    assert np.array_equal(orc.unpack_q(w, K), q)


def test_pack_unpack_round_trip_random():
    q = synth.nibbles(7, 1, 64 * 512).reshape(64, 512)
    assert np.array_equal(orc.unpack_q(orc.pack_q(q), 512), q)


def test_unpack_reads_row_pitch():
    q = synth.nibbles(8, 1, 3 * 32).reshape(3, 32)
    w = orc.pack_q(q, ldq=12)
    assert w.shape == (3, 12)
    assert np.array_equal(orc.unpack_q(w, 32), q)


# --------------------------------------------------------------------------
# Dequantisation
# --------------------------------------------------------------------------

def _dequant_cases():
    lines = _read_lines("dequant_tables.txt")
    cases = []
    i = 0
    while i < len(lines):
        assert lines[i][0] == "case"
        _, name, dtype, qtype, sbits = lines[i]
        q = [int(v) for v in lines[i + 1][1:]]
        w = [float(v) for v in lines[i + 2][1:]]
        cases.append((name, dtype, qtype, int(sbits, 16), q, w))
        i += 3
    return cases


@pytest.mark.parametrize("case", _dequant_cases(), ids=lambda c: c[0])
def test_dequant_hand_tables(case):
    name, dtype, qtype, sbits, q, w = case
    qa = np.array([q], dtype=np.uint8)
    s = np.array([[sbits]], dtype=np.uint16)
    got = orc.values(orc.dequant(qa, s, None, -1, dtype), dtype)[0]
    assert list(got) == w
    # +0 when q equals the zero point and the scale is positive
    bits = orc.dequant(qa, s, None, -1, dtype)[0]
    assert all(int(b) == 0 for b, qq in zip(bits, q) if qq == 8)


def test_dequant_explicit_zero_points_hand_case():
    g = {ln[0]: ln[1:] for ln in _read_lines("zero_points.txt")}
    N, K, G = int(g["N"][0]), int(g["K"][0]), int(g["G"][0])
    dtype = g["dtype"][0]
    q = np.full((N, K), int(g["q_all"][0]), dtype=np.uint8)
    sb = np.array([[int(v, 16) for v in g["scale_bits"]]] * N, dtype=np.uint16)
    zw = np.array([[int(v, 16) for v in g["zeros_words"]]], dtype=np.uint32).view(np.int32)
    w = orc.values(orc.dequant(q, sb, zw, G, dtype), dtype)
    exp0 = [float(v) for v in g["w_group0"]]
    exp1 = [float(v) for v in g["w_group1"]]
    for n in range(N):
        assert np.all(w[n, :G] == exp0[n])
        assert np.all(w[n, G:] == exp1[n])


def test_uint4_with_all_zero_points_8_equals_uint4b8():
    p = synth.Problem(1, 64, 256, 64, "uint4b8", "bf16")
    q, s, _ = synth.make_weights(p)
    zeros = np.full((64 // 8, 256 // 64), 0x88888888, dtype=np.uint32).view(np.int32)
    a = orc.dequant(q, s, None, 64, "bf16")
    b = orc.dequant(q, s, zeros, 64, "bf16")
    assert np.array_equal(a, b)


def test_group_minus_one_is_one_group_spanning_k():
    p = synth.Problem(1, 16, 128, -1, "uint4b8", "fp16")
    q, s, _ = synth.make_weights(p)
    assert s.shape == (16, 1)
    assert np.array_equal(orc.dequant(q, s, None, -1, "fp16"), orc.dequant(q, s, None, 128, "fp16"))
    # and it equals per-row scaling: every element of row n uses s[n]
    w = orc.values(orc.dequant(q, s, None, -1, "fp16"), "fp16")
    sv = orc.values(s, "fp16")
    exact = (q.astype(np.float64) - 8.0) * sv
    assert np.array_equal(w, orc.values(orc.round_to(exact, "fp16"), "fp16"))


def test_group_index_uses_k_over_g():
    # Row-distinct, group-distinct power-of-two scales expose a wrong group index.
    N, K, G = 8, 128, 32
    q = np.full((N, K), 9, dtype=np.uint8)          # q - 8 = 1 -> w = scale
    sv = np.array([[2.0 ** -(n + 2 * g) for g in range(K // G)] for n in range(N)])
    s = orc.round_to(sv, "bf16")
    w = orc.values(orc.dequant(q, s, None, G, "bf16"), "bf16")
    for n in range(N):
        for k in range(K):
            assert w[n, k] == sv[n, k // G]


def test_zero_point_nibble_of_row():
    words = np.array([[0x76543210, 0x01234567], [0xFEDCBA98, 0x89ABCDEF]], dtype=np.uint32).view(np.int32)
    ng = 2
    for n in range(16):
        assert orc.zero_point(words, ng, n, 0) == (n if n < 8 else 8 + (n - 8))
    assert [orc.zero_point(words, ng, n, 1) for n in range(8)] == [7, 6, 5, 4, 3, 2, 1, 0]
    assert orc.zero_point(None, ng, 3, 1) == 8


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------

def test_gemm_one_hot_rows_select_weight_columns():
    M, N, K = 5, 24, 64
    p = synth.Problem(M, N, K, 32, "uint4b8", "bf16")
    q, s, _ = synth.make_weights(p)
    W = orc.dequant(q, s, None, 32, "bf16")
    km = [0, 17, 33, 63, 40]
    A = np.zeros((M, K), dtype=np.uint16)
    for m, k in enumerate(km):
        A[m, k] = 0x3F80  # 1.0
    C = orc.gemm(A, W, "bf16")
    Wv = orc.values(W, "bf16")
    for m, k in enumerate(km):
        assert np.array_equal(C[m], Wv[:, k])


def test_gemm_integer_case_is_exact():
    M, N, K = 7, 40, 96
    rng = np.random.default_rng(11)
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    s = np.full((N, 1), 0x3F80, dtype=np.uint16)   # scale 1
    a_int = rng.integers(-1, 2, (M, K))
    A = orc.round_to(a_int.astype(np.float64), "bf16")
    C = orc.linear(A, q, s, None, -1, "bf16")
    want = a_int @ (q.astype(np.int64) - 8).T          # exact integer arithmetic
    assert np.array_equal(C, want.astype(np.float64))


def test_gemm_matches_brute_force_python_loop():
    M, N, K = 2, 3, 32
    p = synth.Problem(M, N, K, 32, "uint4b8", "fp16")
    q, s, _ = synth.make_weights(p)
    zeros = np.array([[0x00000F53]], dtype=np.int32)  # rows 0,1,2 -> zero 3, 5, 15
    A = synth.make_activations(p)
    C = orc.linear(A, q, s, zeros, 32, "fp16")
    av = orc.values(A, "fp16")
    sv = orc.values(s, "fp16")
    zs = [3, 5, 15]
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                w = (int(q[n, k]) - zs[n]) * float(sv[n, 0])
                wr = float(np.float16(w))            # numpy: one RNE to fp16
                acc += float(av[m, k]) * wr
            assert abs(acc - C[m, n]) <= 1e-12 * max(1.0, abs(acc))


def test_gemm_matches_torch_float64_matmul():
    p = synth.WORKLOADS["gemv_m1_k512_n512_g128_u4b8_fp16"][0]
    x = synth.make_inputs(synth.Problem(8, p.N, p.K, p.group_size, p.qtype, p.dtype, p.scale_lo, p.scale_hi))
    W = orc.dequant(x.q, x.scales, x.zeros, p.group_size, p.dtype)
    C = orc.gemm(x.A, W, p.dtype)
    ta = torch.from_numpy(orc.values(x.A, p.dtype))
    tw = torch.from_numpy(orc.values(W, p.dtype))
    ref = (ta @ tw.T).numpy()
    assert np.max(np.abs(C - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_gemm_is_not_transposed():
    # C is [M, N] with C[m, n] = sum_k A[m, k] W[n, k]; a square case would hide a transpose
    M, N, K = 3, 5, 16
    A = orc.round_to(np.arange(M * K, dtype=np.float64).reshape(M, K) / 8.0, "bf16")
    W = orc.round_to((np.arange(N * K, dtype=np.float64).reshape(N, K) % 7) - 3.0, "bf16")
    C = orc.gemm(A, W, "bf16")
    want = (np.arange(M * K).reshape(M, K) / 8.0) @ ((np.arange(N * K).reshape(N, K) % 7) - 3.0).T
    assert C.shape == (M, N)
    assert np.array_equal(C, want)


def test_sampled_gemm_variants_agree_with_full():
    p = synth.Problem(6, 40, 128, 64, "uint4", "bf16")
    x = synth.make_inputs(p)
    W = orc.dequant(x.q, x.scales, x.zeros, 64, "bf16")
    full = orc.gemm(x.A, W, "bf16")
    rows = np.array([5, 0, 3])
    assert np.array_equal(orc.gemm_rows(x.A, W, rows, "bf16"), full[rows])
    ms, ns = np.array([0, 5, 2, 2]), np.array([39, 0, 7, 8])
    assert np.array_equal(orc.gemm_pairs(x.A, W, ms, ns, "bf16"), full[ms, ns])
    words = orc.pack_q(x.q)
    got = orc.linear_rows_packed(x.A, words, p.K, x.scales, x.zeros, rows, 64, "bf16")
    assert np.array_equal(got, full[rows])


# --------------------------------------------------------------------------
# Seeded inputs (shared by both sides; no layer arithmetic)
# --------------------------------------------------------------------------

def test_inputs_are_seeded_and_in_range():
    p = synth.Problem(4, 64, 256, 32, "uint4", "bf16")
    a = synth.make_inputs(p)
    b = synth.make_inputs(p)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.A, b.A)
    assert a.q.max() <= 15 and a.q.min() == 0 and a.q.max() == 15
    sv = orc.values(a.scales, "bf16")
    assert sv.min() >= 0.00199 and sv.max() <= 0.0201  # bf16 rounding of the ends
    av = orc.values(a.A, "bf16")
    assert abs(av.mean()) < 0.1 and 0.9 < av.std() < 1.1
    assert a.zeros.shape == (8, 8)
    # the SplitMix64 stream reproduces the published first output for seed 0
    # (state 0 -> first output 0xE220A8397B1DCDAF)
    key0 = np.uint64(0)
    from w4a16_int4_weight_gb300.inputs import _mix64, GOLDEN_GAMMA
    with np.errstate(over="ignore"):
        first = _mix64(np.array([key0 + GOLDEN_GAMMA], dtype=np.uint64))[0]
    assert int(first) == 0xE220A8397B1DCDAF


# --------------------------------------------------------------------------
# Bias (one value per output feature n, added to the GEMM output)
# --------------------------------------------------------------------------

def test_bias_hand_case():
    # M=2, N=3, K=16, uint4b8, G=-1, scale 0.25 everywhere, A = one-hot rows.
    # w[n][k] = (q - 8) * 0.25; row m of A selects k = 3 (m=0) and k = 9 (m=1).
    # q[n][3] = 10, 6, 8 -> w = 0.5, -0.5, 0; q[n][9] = 12, 8, 0 -> w = 1, 0, -2.
    # bias = (0.25, -1.5, 3): C = [[0.75, -2.0, 3.0], [1.25, -1.5, 1.0]] exactly.
    q = np.full((3, 16), 8, dtype=np.uint8)
    q[:, 3] = [10, 6, 8]
    q[:, 9] = [12, 8, 0]
    s = np.full((3, 1), 0x3E80, dtype=np.uint16)          # bf16 0.25
    A = np.zeros((2, 16), dtype=np.uint16)
    A[0, 3] = 0x3F80                                         # 1.0
    A[1, 9] = 0x3F80
    bias = np.array([0x3E80, 0xBFC0, 0x4040], dtype=np.uint16)   # 0.25, -1.5, 3.0
    C = orc.linear(A, q, s, None, -1, "bf16", bias=bias)
    assert np.array_equal(C, np.array([[0.75, -2.0, 3.0], [1.25, -1.5, 1.0]]))


def test_bias_with_zero_weights_is_the_bias():
    p = synth.Problem(5, 40, 64, 32, "uint4", "fp16")
    _, s, z = synth.make_weights(p)
    # every q equal to its row's zero point: w = 0 exactly
    q = np.empty((40, 64), dtype=np.uint8)
    for n in range(40):
        for g in range(2):
            q[n, 32 * g:32 * (g + 1)] = orc.zero_point(z, 2, n, g)
    A = synth.make_activations(p)
    bias = orc.round_to(np.linspace(-3, 3, 40), "fp16")
    C = orc.linear(A, q, s, z, 32, "fp16", bias=bias)
    assert np.array_equal(C, np.broadcast_to(orc.values(bias, "fp16"), (5, 40)))


def test_bias_is_added_per_output_feature():
    p = synth.Problem(6, 24, 128, 64, "uint4b8", "bf16")
    x = synth.make_inputs(p)
    bias = orc.round_to(np.arange(24, dtype=np.float64) * 0.125 - 1.0, "bf16")
    C0 = orc.linear(x.A, x.q, x.scales, None, 64, "bf16")
    C1 = orc.linear(x.A, x.q, x.scales, None, 64, "bf16", bias=bias)
    assert np.allclose(C1 - C0, np.broadcast_to(orc.values(bias, "bf16"), C0.shape), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Checkpoint word formats (GPTQ sequential, the MI300 [K, N/8] layout, ExLlama)
# --------------------------------------------------------------------------

def test_gptq_word_of_values_0_to_7_is_sequential():
    # the pages unpack GPTQ words with shifts 0, 4, ..., 28: values 0..7 -> 0x76543210
    q = np.arange(8, dtype=np.uint8)[None, :]
    assert orc.encode_q(q, "gptq")[0, 0] == 0x76543210
    assert orc.encode_q(q, "exllama")[0, 0] == 0x75316420


def test_kn_word_packs_eight_output_rows():
    # [K, N/8]: word (k, j) holds rows 8j..8j+7 of column k at bits 4i
    q = np.zeros((16, 8), dtype=np.uint8)
    q[8:16, 3] = np.arange(8)          # rows 8..15, K-value 3
    w = orc.encode_q(q, "kn")
    assert w.shape == (8, 2)
    assert w[3, 1] == 0x76543210 and w[3, 0] == 0 and np.count_nonzero(w) == 1


@pytest.mark.parametrize("fmt", ["gptq", "kn"])
def test_checkpoint_formats_round_trip(fmt):
    rng = np.random.default_rng(21)
    q = rng.integers(0, 16, (24, 48)).astype(np.uint8)
    assert np.array_equal(orc.decode_q(orc.encode_q(q, fmt), fmt, 24, 48), q)


def test_exllama_words_match_the_packed_section_without_padding():
    rng = np.random.default_rng(22)
    q = rng.integers(0, 16, (5, 40)).astype(np.uint8)    # K/8 = 5, ldq = 8
    assert np.array_equal(orc.encode_q(q, "exllama"), orc.pack_q(q, 8)[:, :5])


# --------------------------------------------------------------------------
# The parity metric: max|C - C_ref| / (max|C_ref| + 1e-6), the tolerance rule
# every GPU parity test applies
# --------------------------------------------------------------------------

def test_rel_error_hand_cases():
    # largest difference over the largest reference magnitude, not a mean or a per-element ratio
    assert orc.rel_error(np.array([1.0, 2.0]), np.array([1.0, 4.0])) == pytest.approx(2.0 / (4.0 + 1e-6), rel=1e-12)
    # signs: |(-3) - (-1)| = 2 over max|C_ref| = 1
    assert orc.rel_error(np.array([-3.0, 0.0]), np.array([-1.0, 0.0])) == pytest.approx(2.0 / (1.0 + 1e-6), rel=1e-12)
    # the worst element decides, wherever it sits in a 2-D result
    C_ref = np.array([[10.0, -20.0], [5.0, 1.0]])
    C = C_ref.copy()
    C[1, 1] += 0.5
    assert orc.rel_error(C, C_ref) == pytest.approx(0.5 / (20.0 + 1e-6), rel=1e-12)
    # identical results and an all-zero reference
    assert orc.rel_error(C_ref, C_ref) == 0.0
    assert orc.rel_error(np.array([1e-7]), np.array([0.0])) == pytest.approx(1e-7 / 1e-6, rel=1e-12)


def test_rel_error_reads_dtype_bits():
    # bf16 0x3F80 = 1.0 and 0x4000 = 2.0; fp16 0x3C00 = 1.0 and 0x4000 = 2.0
    got = np.array([0x3F80, 0x4000], dtype=np.uint16)
    assert orc.rel_error(got, np.array([1.0, 2.5]), "bf16") == pytest.approx(0.5 / (2.5 + 1e-6), rel=1e-12)
    got = np.array([0x3C00, 0x4000], dtype=np.uint16)
    assert orc.rel_error(got, np.array([1.0, 2.0]), "fp16") == 0.0


def test_rel_error_of_a_nan_output_fails_any_tolerance():
    # a NaN canary left in an output must not pass "err <= tol"
    err = orc.rel_error(np.array([1.0, np.nan]), np.array([1.0, 1.0]))
    assert not (err <= 1e-2)
    nan_bf16 = np.array([0x7FC0], dtype=np.uint16)
    assert not (orc.rel_error(nan_bf16, np.array([1.0]), "bf16") <= 1e-2)
