"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source - a rounding
rule, an exponent bias, a word order, a zero-point or scale index, a sign, a
dropped term, a transposed operand, a row pitch - builds it, routes every oracle
call to it and runs the pins of tests/test_oracle_pins.py until one fails.  A
mistake that no pin notices fails this test.  The mistakes are planted in the
oracle, on the CPU; nothing here touches the CUDA path.
"""

import pytest

import oracle.oracle as orc_mod
import test_oracle_pins as pins

MISTAKES = [
    ("rne ties away from zero",
     "if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;", "if (f >= 0.5) r += 1.0;"),
    ("rounding truncates",
     "if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;", "(void)f;"),
    ("fp16 subnormal scale", "ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    ("bf16 exponent bias in decode", "ldexp((double)(128 + m), e - 127 - 7)", "ldexp((double)(128 + m), e - 126 - 7)"),
    ("overflow one binade late", "if (field >= (1 << ebits) - 1) return", "if (field > (1 << ebits) - 1) return"),
    ("bf16 encode bias", "encode_rne(x, 7, 8, 127)", "encode_rne(x, 7, 8, 128)"),
    ("sequential word order instead of the shuffle",
     "static int value_shift(int i) { return 4 * (i / 2) + 16 * (i % 2); }",
     "static int value_shift(int i) { return 4 * i; }"),
    ("unpack ignores the row pitch", "words[n * ldq + k / 8] >>", "words[n * (K / 8) + k / 8] >>"),
    ("zero-point nibble order reversed",
     "return (int)((w >> (4 * (n % 8))) & 0xF);", "return (int)((w >> (4 * (7 - n % 8))) & 0xF);"),
    ("zero point of the first group only",
     "uint32_t w = (uint32_t)zeros[(n / 8) * ng + g];", "uint32_t w = (uint32_t)zeros[(n / 8) * ng];"),
    ("implicit zero 7", "if (!zeros) return 8;", "if (!zeros) return 7;"),
    ("zero subtracted the wrong way",
     "double v = (double)((int)q[n * K + k] - z) * s;", "double v = (double)(z - (int)q[n * K + k]) * s;"),
    ("scale dropped", "double v = (double)((int)q[n * K + k] - z) * s;", "double v = (double)((int)q[n * K + k] - z);"),
    ("scales read transposed",
     "double s = dt_value(scales[n * ng + g], dtype);", "double s = dt_value(scales[g * N + n], dtype);"),
    ("group index off by one", "int64_t g = k / G_eff;", "int64_t g = (k + 1) / G_eff % ng;"),
    ("dot product drops its last term",
     "for (int64_t k = 0; k < K; ++k) acc += a[k] * w[k];", "for (int64_t k = 0; k + 1 < K; ++k) acc += a[k] * w[k];"),
    ("dot product pairs reversed K",
     "for (int64_t k = 0; k < K; ++k) acc += a[k] * w[k];", "for (int64_t k = 0; k < K; ++k) acc += a[k] * w[K - 1 - k];"),
    ("sampled rows ignored",
     "a[i * K + k] = dt_value(A[rows[i] * K + k], dtype);", "a[i * K + k] = dt_value(A[i * K + k], dtype);"),
    ("sampled pairs read W reversed", "dt_value(W[ns[i] * K + k], dtype)", "dt_value(W[ns[i] * K + (K - 1 - k)], dtype)"),
    ("bias subtracted", "C[m * N + n] += dt_value(bias[n], dtype);", "C[m * N + n] -= dt_value(bias[n], dtype);"),
    ("GPTQ words read in reverse nibble order",
     "(src[n * (K / 8) + k / 8] >> (4 * (k % 8)))", "(src[n * (K / 8) + k / 8] >> (4 * (7 - k % 8)))"),
    ("[K, N/8] words read in reverse nibble order",
     "(src[k * (N / 8) + n / 8] >> (4 * (n % 8)))", "(src[k * (N / 8) + n / 8] >> (4 * (7 - n % 8)))"),
]


def _pin_calls():
    """Every pin of tests/test_oracle_pins.py with its parameters, in file order."""
    calls = []
    for name in dir(pins):
        fn = getattr(pins, name)
        if not (name.startswith("test_") and callable(fn)):
            continue
        line = fn.__code__.co_firstlineno
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((line, name, fn, {}))
            continue
        argname, values = marks[0].args[0], marks[0].args[1]
        for v in values:
            calls.append((line, name, fn, {argname: v}))
    calls.sort(key=lambda c: c[0])
    return [(name, fn, kw) for _, name, fn, kw in calls]


def test_an_unmodified_copy_passes_every_pin(tmp_path):
    # the control: the same build-and-route path with nothing planted
    lib = orc_mod.load_variant(orc_mod.build_variant(orc_mod.source(), str(tmp_path)))
    with orc_mod.using_library(lib):
        for name, fn, kw in _pin_calls():
            fn(**kw)


@pytest.mark.parametrize("mistake", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_each_planted_mistake_fails_a_pin(mistake, tmp_path):
    title, old, new = mistake
    text = orc_mod.source()
    assert text.count(old) == 1, f"the planted change must match exactly once: {old}"
    lib = orc_mod.load_variant(orc_mod.build_variant(text.replace(old, new), str(tmp_path)))
    caught = None
    with orc_mod.using_library(lib):
        for name, fn, kw in _pin_calls():
            try:
                fn(**kw)
            except AssertionError:
                caught = name
                break
    assert caught, f"no pin caught the planted mistake: {title}"
