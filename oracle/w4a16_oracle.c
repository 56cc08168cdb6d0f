/*
 * CPU oracle for the W4A16 int4-weight linear layer  C[M,N] = A[M,K] . dequant(W)^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or constant generator with
 * the CUDA path; it implements the same published definitions independently.
 *
 * Sources (the vLLM mixed-precision linear-kernel pages):
 *   - "rdna_hybrid_w4a16" (later revision), function dequantize_w4a16: the
 *     weight is (q - zero) * scale, rounded once in the activation dtype because
 *     q - zero is a small exact integer.
 *   - same page, _triton_w4a16_skinny_fmt_kernel docstring: ExLlama word order
 *     (8 K-values per 32-bit word in the order 0,2,4,6,1,3,5,7; unshuffle
 *     shifts 0,16,4,20,8,24,12,28), scales [N, K/G], zero points
 *     [N/8, K/G] int32 with row n at word n/8, bits 4*(n%8).
 *   - "triton_w4a16" (MI300 page), module docstring and apply_weights: uint4b8
 *     subtracts the constant 8, uint4 subtracts the explicit zero point;
 *     group_size -1 means one group spanning K.
 *   - both Triton kernels: the dequantised tile is fed to a dot product that
 *     accumulates in float32 and the result is cast to the output dtype; the
 *     oracle accumulates in float64 (the exact definition) and leaves the result
 *     in float64 for comparison.
 *
 * Pins (tests/test_oracle_pins.py): RNE converters against numpy/torch and a
 * nearest-value property; the pages' ExLlama example word 0x75316420 and
 * shift table; hand-written dequant tables (including an fp16 tie); uint4 with
 * every zero = 8 against uint4b8; group -1 against group K; one-hot and
 * integer-valued GEMMs with exact results; a brute-force Python triple loop;
 * torch's float64 matmul.  No function here is "parity unpinned".
 *
 * Arithmetic is float64 throughout; every loop is the plain definition with no
 * blocking or reordering beyond the k-innermost sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_FP16 0
#define ORC_BF16 1

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* IEEE-754 binary16 / bfloat16: exact decode and round-to-nearest-even encode */
/* ------------------------------------------------------------------------- */

double orc_f16_value(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0x1F) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);             /* subnormal: m * 2^-24 */
    else v = ldexp((double)(1024 + m), e - 15 - 10);         /* (1 + m/1024) 2^(e-15) */
    return sign ? -v : v;
}

double orc_bf16_value(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int m = h & 0x7F;
    double v;
    if (e == 0xFF) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -133);             /* subnormal: m * 2^-133 */
    else v = ldexp((double)(128 + m), e - 127 - 7);          /* (1 + m/128) 2^(e-127) */
    return sign ? -v : v;
}

/* Round |x| (finite, > 0) scaled to an integer significand, ties to even. */
static double rne_integer(double v) {
    double r = floor(v);
    double f = v - r;                    /* exact: v has at most 53 bits */
    if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    return r;
}

/* Generic encoder: mbits explicit mantissa bits, exponent bias, exponent field
 * width.  Implements IEEE round-to-nearest-even including subnormals, overflow
 * to infinity and NaN. */
static uint16_t encode_rne(double x, int mbits, int ebits, int bias) {
    uint16_t sign = signbit(x) ? (uint16_t)(1u << (mbits + ebits)) : 0;
    uint16_t exp_all = (uint16_t)(((1u << ebits) - 1) << mbits);
    if (isnan(x)) return (uint16_t)(sign | exp_all | (1u << (mbits - 1)));
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | exp_all);
    if (a == 0.0) return sign;
    int emin = 1 - bias;                                    /* smallest normal exponent */
    int e;
    frexp(a, &e);                                           /* a = f 2^e, f in [0.5, 1) */
    int E = e - 1;                                          /* a in [2^E, 2^(E+1)) */
    if (E < emin) {
        /* subnormal range: integer multiple of 2^(emin - mbits) */
        double r = rne_integer(ldexp(a, mbits - emin));
        return (uint16_t)(sign | (uint16_t)r);              /* r == 2^mbits gives the min normal */
    }
    double r = rne_integer(ldexp(a, mbits - E));            /* in [2^mbits, 2^(mbits+1)] */
    if (r == ldexp(1.0, mbits + 1)) { r = ldexp(1.0, mbits); E += 1; }
    int field = E + bias;
    if (field >= (1 << ebits) - 1) return (uint16_t)(sign | exp_all);   /* overflow */
    return (uint16_t)(sign | (uint16_t)(field << mbits) | (uint16_t)(r - ldexp(1.0, mbits)));
}

uint16_t orc_round_f16(double x) { return encode_rne(x, 10, 5, 15); }
uint16_t orc_round_bf16(double x) { return encode_rne(x, 7, 8, 127); }

static double dt_value(uint16_t h, int dtype) {
    return dtype == ORC_BF16 ? orc_bf16_value(h) : orc_f16_value(h);
}
static uint16_t dt_round(double x, int dtype) {
    return dtype == ORC_BF16 ? orc_round_bf16(x) : orc_round_f16(x);
}

void orc_values(const uint16_t* h, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = dt_value(h[i], dtype);
}
void orc_round(const double* x, int64_t n, int dtype, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = dt_round(x[i], dtype);
}

/* ------------------------------------------------------------------------- */
/* Packed int4 weight words                                                   */
/* ------------------------------------------------------------------------- */
/* A word holds 8 consecutive K values v0..v7 of one row, stored low-to-high in
 * the order v0, v2, v4, v6, v1, v3, v5, v7 (the pages' ExLlama shuffle:
 * v0 | v2<<4 | v4<<8 | v6<<12 | v1<<16 | v3<<20 | v5<<24 | v7<<28).  Value i of
 * the word therefore sits at bit offset 4*(i/2) + 16*(i%2).  Rows are ldq words
 * long (ldq >= K/8); words past K/8 are zero. */

static int value_shift(int i) { return 4 * (i / 2) + 16 * (i % 2); }

int orc_shift_table(int i) { return value_shift(i); }

void orc_pack_q(const uint8_t* q, int64_t N, int64_t K, int64_t ldq, uint32_t* words) {
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t j = 0; j < ldq; ++j) {
            uint32_t w = 0;
            if (j < K / 8)
                for (int i = 0; i < 8; ++i)
                    w |= (uint32_t)(q[n * K + 8 * j + i] & 0xF) << value_shift(i);
            words[n * ldq + j] = w;
        }
    }
}

void orc_unpack_q(const uint32_t* words, int64_t N, int64_t K, int64_t ldq, uint8_t* q) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            q[n * K + k] = (uint8_t)((words[n * ldq + k / 8] >> value_shift((int)(k % 8))) & 0xF);
}

/* ------------------------------------------------------------------------- */
/* Dequantisation: w = rne_dtype((q - zero) * scale)                          */
/* ------------------------------------------------------------------------- */
/* zero = 8 for uint4b8 (zeros == NULL); otherwise the raw nibble of row n in
 * word zeros[(n/8)*ng + g] at bits 4*(n%8).  g = k / G_eff.  (q - zero) is an
 * integer in [-15, 15] and the scale has at most 11 significant bits, so the
 * float64 product is exact and one rounding gives the dtype result. */

int orc_zero_point(const int32_t* zeros, int64_t ng, int64_t n, int64_t g) {
    if (!zeros) return 8;
    uint32_t w = (uint32_t)zeros[(n / 8) * ng + g];
    return (int)((w >> (4 * (n % 8))) & 0xF);
}

void orc_dequant(const uint8_t* q, const uint16_t* scales, const int32_t* zeros,
                 int64_t N, int64_t K, int64_t G_eff, int dtype, uint16_t* w) {
    int64_t ng = K / G_eff;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            int64_t g = k / G_eff;
            int z = orc_zero_point(zeros, ng, n, g);
            double s = dt_value(scales[n * ng + g], dtype);
            double v = (double)((int)q[n * K + k] - z) * s;
            w[n * K + k] = dt_round(v, dtype);
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Checkpoint word formats the pages read (all 4-bit values, 8 per int32):      */
/*  - GPTQ / compressed-tensors ("triton_w4a16" page, repack_w_q): [N][K/8],   */
/*    K-value 8j+i of row n at bits 4i of word j (sequential shifts 0..28).    */
/*  - the MI300 kernel's layout (same function, step 4): [K][N/8], N-value      */
/*    8j+i of row k at bits 4i of word j.                                      */
/*  - the ExLlama shuffle ("rdna_hybrid_w4a16", pack_int4_exllama_shuffle):   */
/*    [N][K/8], K-value 8j+i at value_shift(i) (orc_pack_q without padding).   */
/* Encoders from unpacked q [N][K] and decoders back to it.                     */
/* ------------------------------------------------------------------------- */
void orc_encode_gptq(const uint8_t* q, int64_t N, int64_t K, uint32_t* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 8; ++j) {
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i) w |= (uint32_t)(q[n * K + 8 * j + i] & 0xF) << (4 * i);
            out[n * (K / 8) + j] = w;
        }
}

void orc_decode_gptq(const uint32_t* src, int64_t N, int64_t K, uint8_t* q) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            q[n * K + k] = (uint8_t)((src[n * (K / 8) + k / 8] >> (4 * (k % 8))) & 0xF);
}

void orc_encode_kn(const uint8_t* q, int64_t N, int64_t K, uint32_t* out) {
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N / 8; ++j) {
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i) w |= (uint32_t)(q[(8 * j + i) * K + k] & 0xF) << (4 * i);
            out[k * (N / 8) + j] = w;
        }
}

void orc_decode_kn(const uint32_t* src, int64_t N, int64_t K, uint8_t* q) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            q[n * K + k] = (uint8_t)((src[k * (N / 8) + n / 8] >> (4 * (n % 8))) & 0xF);
}

void orc_encode_exllama(const uint8_t* q, int64_t N, int64_t K, uint32_t* out) {
    orc_pack_q(q, N, K, K / 8, out);
}

/* ------------------------------------------------------------------------- */
/* GEMM in float64:  C[m][n] = sum_k A[m][k] * W[n][k]                          */
/* ------------------------------------------------------------------------- */

static double dot_values(const double* a, const double* w, int64_t K) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += a[k] * w[k];
    return acc;
}

/* Selected rows of C: out[i][n] = C[rows[i]][n] = sum_k A[rows[i]][k] W[n][k].
 * Each operand row is decoded to exact float64 values once; the sum runs over
 * k in increasing order. */
/* Returns 0, or 1 when host memory for the float64 copies could not be had
 * (the output is then incomplete and must not be used). */
int orc_gemm_rows(const uint16_t* A, const uint16_t* W, const int64_t* rows, int64_t nrows,
                  int64_t N, int64_t K, int dtype, double* out) {
    double* a = (double*)malloc((size_t)(nrows * K > 0 ? nrows * K : 1) * sizeof(double));
    if (!a) return 1;
    int failed = 0;
    for (int64_t i = 0; i < nrows; ++i)
        for (int64_t k = 0; k < K; ++k) a[i * K + k] = dt_value(A[rows[i] * K + k], dtype);
#pragma omp parallel
    {
        double* w = (double*)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            if (!w) continue;
            for (int64_t k = 0; k < K; ++k) w[k] = dt_value(W[n * K + k], dtype);
            for (int64_t i = 0; i < nrows; ++i) out[i * N + n] = dot_values(a + i * K, w, K);
        }
        free(w);
    }
    free(a);
    return failed;
}

int orc_gemm(const uint16_t* A, const uint16_t* W, int64_t M, int64_t N, int64_t K,
             int dtype, double* C) {
    int64_t* rows = (int64_t*)malloc((size_t)(M > 0 ? M : 1) * sizeof(int64_t));
    if (!rows) return 1;
    for (int64_t m = 0; m < M; ++m) rows[m] = m;
    const int rc = orc_gemm_rows(A, W, rows, M, N, K, dtype, C);
    free(rows);
    return rc;
}

/* Selected elements: out[i] = C[ms[i]][ns[i]]. */
void orc_gemm_pairs(const uint16_t* A, const uint16_t* W, const int64_t* ms, const int64_t* ns,
                    int64_t npairs, int64_t K, int dtype, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < npairs; ++i) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += dt_value(A[ms[i] * K + k], dtype) * dt_value(W[ns[i] * K + k], dtype);
        out[i] = acc;
    }
}

/* Bias: C[m][n] += bias[n] (dtype bits), the value the pages add to the GEMM
 * output ("rdna_hybrid_w4a16", _rdna_hybrid_w4a16_apply_impl: the bias vector
 * of the linear layer, one value per output feature n).  C stays in float64. */
void orc_add_bias(double* C, int64_t M, int64_t N, const uint16_t* bias, int dtype) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) C[m * N + n] += dt_value(bias[n], dtype);
}

/* The whole layer in the pages' order on a packed weight: unpack -> dequant ->
 * GEMM over the selected rows of A.  Used as the timed CPU baseline. */
int orc_linear_rows(const uint16_t* A, const uint32_t* words, int64_t ldq, const uint16_t* scales,
                    const int32_t* zeros, const int64_t* rows, int64_t nrows, int64_t N, int64_t K,
                    int64_t G_eff, int dtype, double* out) {
    uint8_t* q = (uint8_t*)malloc((size_t)(N * K));
    uint16_t* w = (uint16_t*)malloc((size_t)(N * K) * sizeof(uint16_t));
    if (!q || !w) { free(q); free(w); return 1; }
    orc_unpack_q(words, N, K, ldq, q);
    orc_dequant(q, scales, zeros, N, K, G_eff, dtype, w);
    const int rc = orc_gemm_rows(A, w, rows, nrows, N, K, dtype, out);
    free(q);
    free(w);
    return rc;
}
