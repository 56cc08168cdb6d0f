/*
 * w4a16.h - C ABI of libw4a16, the GB300 (sm_103a) W4A16 int4-weight linear layer.
 *
 *     C[M,N] = A[M,K] . dequant(W)^T,     dequant(W)[n,k] = (q[n,k] - zero[n,g]) * scale[n,g]
 *
 * with g = k / G_eff.  The definitions follow the vLLM mixed-precision linear
 * kernel pages ("rdna_hybrid_w4a16", both revisions; "triton_w4a16" for MI300):
 *   - quant types (RDNAHybridW4A16LinearKernel.SUPPORTED_QUANT_TYPES): uint4b8
 *     is symmetric with the implicit zero 8; uint4 carries explicit zero points;
 *   - group sizes (TRITON_W4A16_SUPPORTED_GROUP_SIZES): -1, 32, 64, 128, 256,
 *     where -1 is one group spanning K (apply_weights resolves it to K);
 *   - shape rules (can_implement): K % 16 == 0 and K % G_eff == 0; N % 8 == 0
 *     when zero points are packed 8 per word along N (triton_w4a16_skinny_fmt_gemm);
 *   - scales [N, K/G_eff] in the activation dtype, "skinny layout, NOT transposed";
 *     zero points int32 [N/8, K/G_eff], row n's raw zero point in word n/8 at
 *     bits 4*(n%8) (_triton_w4a16_skinny_fmt_kernel docstring);
 *   - dequantisation (dequantize_w4a16): q - zero is a small exact integer, so
 *     the weight is rounded once, in the activation dtype;
 *   - the GEMM accumulates in float32 and casts the result to the activation
 *     dtype (both Triton kernels: tl.dot(..., out_dtype=tl.float32), then .to()).
 *
 * Conventions for every entry point
 *   - All device pointers are plain CUDA device addresses owned by the caller.
 *     The library allocates no device memory, ever; it keeps only host-side
 *     caches and one static device status word per kernel module.
 *   - `stream` is a cudaStream_t (0 = legacy default stream).  Every call that
 *     takes a stream only enqueues work on it and returns; results are ready
 *     when the stream is synchronised.
 *   - Arguments are validated on the host before anything is enqueued.  A
 *     rejected call returns a nonzero w4a16_status, enqueues nothing and leaves
 *     a message for w4a16_last_error_string() (per calling thread).
 *   - Kernels bound every wait on a barrier (about one second).  A wait that
 *     runs out records W4A16_ERR_DEVICE_TIMEOUT in the library's device status
 *     word and the kernel returns without hanging; w4a16_device_status() reads it.
 *     The outputs such a kernel could not complete are written as NaN, but the
 *     call that enqueued it has already returned W4A16_OK: a caller that must
 *     not consume such results checks w4a16_device_status() after a run.
 *   - dtype is the activation = scale = output type; fp16 or bf16.
 *   - Sizes are int64_t and must be < 2^31.
 *   - Calls may come from several host threads at once (the host caches are
 *     locked; a thread that has not used CUDA yet gets the current device's
 *     primary context made current).  The GEMM, dequant and pack entry points
 *     may be captured into a CUDA graph: they only launch kernels on `stream`,
 *     whose arguments (tensor maps included) are fixed at capture.
 *   - Results are deterministic: no kernel uses atomics to combine partial
 *     sums, and K-split partials are added in a fixed order.
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,     /* a shape, pointer, alignment or enum was rejected */
    W4A16_ERR_UNSUPPORTED = 2,     /* valid arguments outside what this library implements */
    W4A16_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed (message has details) */
    W4A16_ERR_DEVICE_TIMEOUT = 4   /* a kernel's bounded barrier wait ran out */
} w4a16_status;

typedef enum {
    W4A16_UINT4B8 = 0,             /* symmetric, zero = 8 implicit; zeros pointer must be NULL */
    W4A16_UINT4 = 1                /* asymmetric, explicit zero points [N/8, K/G_eff] int32 */
} w4a16_qtype;

typedef enum { W4A16_FP16 = 0, W4A16_BF16 = 1 } w4a16_dtype;

typedef enum {
    W4A16_PATH_AUTO = 0,           /* the M-router decides */
    W4A16_PATH_DECODE = 1,         /* small-M split-K kernel (tensor-core mma.sync, M <= 64) */
    W4A16_PATH_FUSED = 2,          /* fused dequant + tcgen05 GEMM; one of the two below by M */
    W4A16_PATH_DENSE = 3,          /* tcgen05 GEMM on a dense dequantised copy */
    W4A16_PATH_FUSED_TMEM = 4,     /* fused, dequantised tile written to tensor memory
                                      (tcgen05.mma A operand from TMEM; mid M) */
    W4A16_PATH_FUSED_SMEM = 5      /* fused, dequantised tile written to shared memory
                                      (both tcgen05.mma operands in SMEM; large M) */
} w4a16_path;

/*
 * Packed weight buffer ("store the weight once", rdna_hybrid_w4a16 page 1):
 *
 *   offset 0           q section: uint32 words [N][ldq], ldq = round_up(K/8, 4).
 *                      Word j of row n holds K-values k = 8j .. 8j+7 of that row,
 *                      value 8j+i at bit offset 4*(i/2) + 16*(i%2): low to high
 *                      the nibbles are v0,v2,v4,v6,v1,v3,v5,v7 (the pages'
 *                      ExLlama shuffle, unshuffle shifts 0,16,4,20,8,24,12,28).
 *                      Words j >= K/8 are zero.
 *   scales_off         scales, transposed: dtype [K/G_eff][lds], lds = round_up(N, 8);
 *                      element (g, n) is the scale of row n, group g.  Padding
 *                      elements (n >= N) are zero.
 *   zeros_off          zero points (uint4 only), transposed: int32 [K/G_eff][ldz],
 *                      ldz = round_up(N/8, 4); word (g, j) holds the zero points
 *                      of rows 8j .. 8j+7 of group g, row n at bits 4*(n%8).
 *                      Padding words are zero.
 *
 * The transposition puts the scales of 128 consecutive rows of one group in
 * 256 contiguous bytes, so the kernels fetch them with the same TMA bulk
 * copies that bring the weight tiles.  Each section starts on a 256-byte
 * boundary; total_bytes is a multiple of 256.  zeros_off is 0 for uint4b8.
 * Host-only; returns W4A16_ERR_INVALID_ARG on bad arguments.  Any output
 * pointer may be NULL.
 */
w4a16_status w4a16_packed_layout(int64_t N, int64_t K, int G, int qtype, int dtype,
                                 size_t* total_bytes, size_t* scales_off, size_t* zeros_off,
                                 int64_t* ldq_words);

/*
 * Source layouts w4a16_pack_ex reads (checkpoint formats on the pages).
 */
typedef enum {
    W4A16_Q_UNPACKED = 0,   /* uint8 [N][K], one value per byte (w4a16_pack's input) */
    W4A16_Q_GPTQ = 1,       /* int32 [N][K/8]: K-value 8j+i of row n at bits 4i of word j
                               (GPTQ / compressed-tensors; triton_w4a16 page, repack_w_q) */
    W4A16_Q_EXLLAMA = 2,    /* int32 [N][K/8]: K-value 8j+i at bits 4*(i/2) + 16*(i%2)
                               (rdna_hybrid_w4a16, pack_int4_exllama_shuffle) */
    W4A16_Q_KN = 3          /* int32 [K][N/8]: N-value 8j+i of K-row k at bits 4i of word j
                               (the MI300 kernel's layout, repack_w_q step 4); N % 8 == 0 */
} w4a16_qformat;

typedef enum {
    W4A16_LAYOUT_NG = 0,    /* scales [N][K/G_eff], zeros [N/8][K/G_eff] (compressed-tensors) */
    W4A16_LAYOUT_GN = 1     /* scales [K/G_eff][N], zeros [K/G_eff][N/8] (AutoGPTQ; the MI300
                               kernel's repacked form) */
} w4a16_param_layout;

/*
 * w4a16_pack - relayout one quantised weight into the packed buffer.
 * (Prior art: process_weights_after_loading -> pack_skinny_int4 /
 *  pack_int4_exllama_shuffle on the rdna_hybrid_w4a16 pages; repack_w_q on
 *  the triton_w4a16 page.)
 *   q        device uint8 [N][K], one value per byte in natural K order; only the
 *            low 4 bits of each byte are used.  8-byte aligned.
 *   scales   device dtype [N][K/G_eff] (the checkpoint layout).  2-byte aligned.
 *   zeros    device int32 [N/8][K/G_eff] for uint4 (N % 8 == 0), NULL for uint4b8.
 *   Wpacked  device buffer of total_bytes (w4a16_packed_layout), 256-byte aligned,
 *            must not overlap the inputs.  Fully overwritten, padding included.
 * Enqueues one or two kernels on `stream`.
 */
/*
 * w4a16_pack_ex - w4a16_pack from a checkpoint's own word format: the packed
 * buffer it writes is the one w4a16_pack writes from the same values (bit for
 * bit, padding included), without an unpacked [N][K] copy in between.
 *   qsrc          device words in `qformat` (w4a16_qformat); 4-byte aligned
 *                 (8-byte for W4A16_Q_UNPACKED).
 *   param_layout  w4a16_param_layout of scales and zeros.
 *   Other arguments as for w4a16_pack.  W4A16_ERR_INVALID_ARG for an unknown
 *   format or layout, or W4A16_Q_KN with N % 8 != 0.  Enqueues two or three
 *   kernels on `stream`.
 */
w4a16_status w4a16_pack_ex(const void* qsrc, int qformat, const void* scales, const int32_t* zeros,
                           int param_layout, void* Wpacked, int64_t N, int64_t K, int G, int qtype,
                           int dtype, void* stream);

w4a16_status w4a16_pack(const uint8_t* q, const void* scales, const int32_t* zeros,
                        void* Wpacked, int64_t N, int64_t K, int G, int qtype, int dtype,
                        void* stream);

/*
 * w4a16_gemm - C[M,N] = A[M,K] . dequant(W)^T, routed by M (the hybrid's
 * _rdna_hybrid_w4a16_apply_impl: a skinny split-K path for decode, a fused
 * dequant GEMM for prefill).
 *   A        device dtype [M][K], row-major, contiguous (row stride K).  16-byte aligned.
 *   Wq       device q section of a packed buffer (its offset 0).  16-byte aligned.
 *   scales   device scale section of the packed buffer (transposed [K/G_eff][lds],
 *            see above), or the caller's own array in that layout.  16-byte aligned.
 *   zeros    device zero-point section ([K/G_eff][ldz] int32) for uint4, NULL for
 *            uint4b8.  16-byte aligned.
 *   C        device dtype [M][N], row-major, written in full, must not overlap inputs.
 *            2-byte aligned.
 *   M        >= 0; M == 0 returns W4A16_OK and enqueues nothing.
 * Float32 accumulation, one final rounding (RNE) to dtype.
 */
w4a16_status w4a16_gemm(const void* A, const void* Wq, const void* scales, const int32_t* zeros,
                        void* C, int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                        void* stream);

/*
 * Option bit OR-ed into w4a16_gemm_ex's `path` argument.
 *
 * W4A16_OPT_STATIC_WEIGHTS: the caller promises that Wq, scales and zeros are
 * not written by any work that may still be running on the stream when this
 * call's kernel starts (true for weights packed once and then only read).
 * The kernels always start early behind the previous kernel on the stream
 * (programmatic dependent launch) and wait for it before touching memory;
 * with this bit the small-M kernel also fetches its weights during that wait,
 * hiding HBM latency across back-to-back layers.  Activations and outputs are
 * never touched before the previous kernel completes.
 */
#define W4A16_OPT_STATIC_WEIGHTS 0x100

/*
 * w4a16_gemm_ex - w4a16_gemm with an optional dense copy and a path choice.
 * Wdense is NULL or a device dtype [N][K] dequantised copy (w4a16_dequant
 * output), 16-byte aligned; the prefill "cached dense-dequant" path of the
 * later rdna_hybrid_w4a16 revision (_cache_dequant_weight) uses it when the
 * router sends large M there.  path is a w4a16_path, optionally OR-ed with
 * W4A16_OPT_STATIC_WEIGHTS; forcing DECODE requires M <= 64 and forcing DENSE
 * requires Wdense (else W4A16_ERR_INVALID_ARG).
 */
w4a16_status w4a16_gemm_ex(const void* A, const void* Wq, const void* scales,
                           const int32_t* zeros, const void* Wdense, void* C,
                           int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                           int path, void* stream);

/*
 * w4a16_linear - the linear layer with its bias: C[m,n] = rne_dtype(sum_k
 * A[m,k] * w[n,k] + bias[n]), the bias of the pages' apply path
 * (rdna_hybrid_w4a16, _rdna_hybrid_w4a16_apply_impl: a per-output-feature
 * vector, handed to the skinny kernel or added to the fused GEMM's output).
 * Here it is added to the fp32 accumulator in every kernel's epilogue, so the
 * output is rounded once (the pages' fused path adds it after rounding, in
 * the dtype: two roundings; both lie within the GEMM tolerance).
 *   bias     device dtype [N], 2-byte aligned, or NULL for none.
 *   lda      row pitch of A in elements: 0 (= K) or >= K and a multiple of 8
 *            (16-byte rows, as every kernel reads A by TMA); rows may be padded
 *            (the pages' stride_am).  The padding is never read.
 *   ldc      row pitch of C in elements: 0 (= N) or >= N.  Only [M][N] is written.
 *   Every other argument, the validation and the error behaviour are those of
 *   w4a16_gemm_ex, which is w4a16_linear with bias NULL and lda = ldc = 0.
 */
w4a16_status w4a16_linear(const void* A, int64_t lda, const void* Wq, const void* scales,
                          const int32_t* zeros, const void* bias, const void* Wdense, void* C,
                          int64_t ldc, int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                          int path, void* stream);

/*
 * w4a16_route - the kernel w4a16_gemm_ex(..., W4A16_PATH_AUTO, ...) runs for
 * these sizes (has_dense != 0 when a dense copy is supplied).  Host-only.
 * Returns W4A16_PATH_DECODE, _FUSED_TMEM, _FUSED_SMEM or _DENSE, or -1 on
 * invalid arguments.
 */
int w4a16_route(int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype, int has_dense);

/*
 * w4a16_launch_plan - how w4a16_gemm_ex / w4a16_linear would launch for these
 * sizes on a GPU with num_sms SMs.  Host-only: touches no device.
 *   path       W4A16_PATH_AUTO (resolved by the router, has_dense as in
 *              w4a16_route), _FUSED, or one kernel by name.
 *   info       receives the kernel (path, always a specific one), the tokens per
 *              CTA tile, the CTAs per cluster that split K (1 = none), the depth
 *              of the small-M kernel's TMA ring (0 for the other kernels), the
 *              CTAs launched and the small-M kernel's dynamic shared memory per
 *              CTA (0 for the other kernels).  For the tensor-memory kernel
 *              between one and two tiles per SM, k_split 2 with a grid of two
 *              CTAs per SM means clusters of two that take two whole tiles next
 *              to clusters that split one tile's K.
 * Returns W4A16_ERR_INVALID_ARG for arguments w4a16_gemm_ex would reject
 * (pointers aside), W4A16_ERR_UNSUPPORTED where it would be unsupported.
 */
typedef struct {
    int path;
    int token_tile;
    int k_split;
    int stages;
    int64_t grid;
    int64_t smem_bytes;
} w4a16_launch_info;
w4a16_status w4a16_launch_plan(int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                               int path, int has_dense, int num_sms, w4a16_launch_info* info);

/*
 * w4a16_dequant - dense copy W[n][k] = rne_dtype((q[n][k] - zero) * scale), the
 * pages' dequantize_w4a16.  Bit-exact: (q - zero) * scale is exact in float32,
 * so the single rounding to dtype is the only one.
 *   Wq, scales, zeros as for w4a16_gemm.
 *   W        device dtype [N][K] row-major, 16-byte aligned, written in full.
 */
w4a16_status w4a16_dequant(const void* Wq, const void* scales, const int32_t* zeros, void* W,
                           int64_t N, int64_t K, int G, int qtype, int dtype, void* stream);

/*
 * w4a16_gemm_dense - C[M,N] = A[M,K] . W[N,K]^T on a dense dtype weight (the
 * pages' rocm_unquantized_gemm_impl on the cached copy): a persistent tcgen05
 * GEMM, one CTA per SM, fp32 accumulation, one RNE rounding to the dtype.
 *   A 16-byte aligned [M][K]; W 16-byte aligned [N][K]; C [M][N]; K % 16 == 0.
 */
w4a16_status w4a16_gemm_dense(const void* A, const void* W, void* C, int64_t M, int64_t N,
                              int64_t K, int dtype, void* stream);

/* Message of the last rejected or failed call on this thread ("" if none). */
const char* w4a16_last_error_string(void);

/*
 * w4a16_device_status - synchronise the current device, read and clear the
 * library's device status words (every kernel module's word is read and
 * cleared on each call).  Returns W4A16_OK, W4A16_ERR_DEVICE_TIMEOUT (a kernel
 * gave up waiting; *site, if non-NULL, receives the wait site id of the first
 * module, in library order, whose word was set) or W4A16_ERR_CUDA.
 */
w4a16_status w4a16_device_status(int* site);

/*
 * w4a16_selftest_wait_timeout - exercise the failure-detection path on the
 * device.  Enqueues a one-warp kernel that waits, through the same bounded
 * barrier wait every kernel of the library uses, on an mbarrier that nothing
 * ever completes.  After the wait limit (about one second) the wait gives up,
 * records site W4A16_SELFTEST_SITE in the library's device status word and the
 * kernel returns: nothing faults, nothing hangs, and the device stays usable.
 * A following w4a16_device_status() returns W4A16_ERR_DEVICE_TIMEOUT with that
 * site (and clears it).  Returns W4A16_ERR_CUDA if the launch fails.
 */
#define W4A16_SELFTEST_SITE 90
w4a16_status w4a16_selftest_wait_timeout(void* stream);

/* Library version, e.g. 100 for 0.1.0. */
int w4a16_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
