// C ABI of libw4a16 (declarations and argument contracts: include/w4a16.h).
//
// Host side only: argument validation (the rules of the pages' can_implement
// and asserts), the M-router (_rdna_hybrid_w4a16_apply_impl's role), TMA
// tensor-map encoding, and kernel launches on the caller's stream.  Nothing
// here allocates device memory.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "w4a16.h"
#include "internal.h"

namespace {

using namespace w4a16;

thread_local char g_err[512] = "";

w4a16_status fail(w4a16_status code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

w4a16_status cuda_fail(cudaError_t e, const char* what) {
    // A failed launch also leaves the error in the runtime's per-thread "last
    // error"; clear it so that it is not reported again by a later, unrelated call.
    (void)cudaGetLastError();
    return fail(W4A16_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shape / enum checks shared by every entry point that takes a quantised weight.
w4a16_status check_weight(int64_t N, int64_t K, int G, int qtype, int dtype, LayerShape* s) {
    if (dtype != W4A16_FP16 && dtype != W4A16_BF16)
        return fail(W4A16_ERR_INVALID_ARG, "dtype %d is not fp16 (0) or bf16 (1)", dtype);
    if (qtype != W4A16_UINT4B8 && qtype != W4A16_UINT4)
        return fail(W4A16_ERR_INVALID_ARG, "quant type %d is not uint4b8 (0) or uint4 (1)", qtype);
    if (G != -1 && G != 32 && G != 64 && G != 128 && G != 256)
        return fail(W4A16_ERR_INVALID_ARG, "group size %d not supported; supported: -1, 32, 64, 128, 256", G);
    if (N < 1 || N > kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "N=%lld out of range", (long long)N);
    if (K < 16 || K > kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "K=%lld out of range", (long long)K);
    if (K % 16 != 0) return fail(W4A16_ERR_INVALID_ARG, "K=%lld must be divisible by 16", (long long)K);
    const int64_t g_eff = G == -1 ? K : G;
    if (K % g_eff != 0)
        return fail(W4A16_ERR_INVALID_ARG, "K=%lld must be divisible by group_size=%d", (long long)K, G);
    if (qtype == W4A16_UINT4 && N % 8 != 0)
        return fail(W4A16_ERR_INVALID_ARG, "N must be divisible by 8 for packed zero points, got %lld", (long long)N);
    if (s) {
        s->N = N;
        s->K = K;
        s->g_eff = g_eff;
        s->ng = K / g_eff;
        s->ldq = (K / 8 + 3) / 4 * 4;
        s->lds = (N + 7) / 8 * 8;
        s->ldz = (N / 8 + 3) / 4 * 4;
        s->bf16 = dtype == W4A16_BF16;
        s->zp = qtype == W4A16_UINT4;
        s->M = 0;
        s->lda = K;
        s->ldc = N;
    }
    return W4A16_OK;
}

w4a16_status check_qptrs(const void* Wq, const void* scales, const int32_t* zeros, int qtype) {
    if (!Wq || !aligned(Wq, 16)) return fail(W4A16_ERR_INVALID_ARG, "Wq must be a non-null 16-byte aligned device pointer");
    if (!scales || !aligned(scales, 16)) return fail(W4A16_ERR_INVALID_ARG, "scales must be a non-null 16-byte aligned device pointer (the packed scale section)");
    if (qtype == W4A16_UINT4) {
        if (!zeros || !aligned(zeros, 16)) return fail(W4A16_ERR_INVALID_ARG, "uint4 needs a non-null 16-byte aligned zeros pointer (the packed zero section)");
    } else if (zeros) {
        return fail(W4A16_ERR_INVALID_ARG, "zeros must be NULL for uint4b8 (the zero point is the constant 8)");
    }
    return W4A16_OK;
}

// --- TMA tensor maps -------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_get_current = nullptr;   // optional: without it, bind on every encode
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

w4a16_status get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else if (g_encode_err == cudaSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    });
    if (!g_encode) return cuda_fail(g_encode_err, "cuTensorMapEncodeTiled lookup");
    return W4A16_OK;
}

// The encoder needs a current context.  A host thread whose runtime calls so
// far made none current (cudaGetDevice does not; a launch would) has none, and
// the encoder then fails with CUDA_ERROR_INVALID_CONTEXT.  cudaSetDevice makes
// the device's primary context current in this thread, as a launch would.
w4a16_status ensure_current_context() {
    CUcontext ctx = nullptr;
    if (g_ctx_get_current && g_ctx_get_current(&ctx) == CUDA_SUCCESS && ctx) return W4A16_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "making the device's primary context current");
    return W4A16_OK;
}

// 2-D row-major tensor [rows][cols] of `elem` bytes, box [box_rows][box_cols].
// Encoded tensor maps, keyed by every input of the encoding (a map is a pure
// function of them), so that repeated calls on the same buffers - a layer's
// weight every step, a reused activation buffer - skip the driver encoder.
struct MapKey {
    const void* base;
    uint64_t cols, rows, stride;
    uint32_t box_cols, box_rows;
    int dt, swz;
    bool operator==(const MapKey& o) const {
        return base == o.base && cols == o.cols && rows == o.rows && stride == o.stride &&
               box_cols == o.box_cols && box_rows == o.box_rows && dt == o.dt && swz == o.swz;
    }
};
constexpr int kMapCacheSize = 4096;   // direct-mapped
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool valid = false;
};
MapEntry g_map_cache[kMapCacheSize];
std::mutex g_map_mu;

size_t map_slot(const MapKey& k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    for (uint64_t v : {k.cols, k.rows, k.stride, uint64_t(k.box_cols) << 32 | k.box_rows,
                       uint64_t(uint32_t(k.dt)) << 32 | uint32_t(k.swz)})
        h = (h ^ v) * 0x100000001B3ull;
    return size_t(h >> 52) % kMapCacheSize;
}

w4a16_status make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int elem,
                      uint64_t cols, uint64_t rows, uint64_t row_stride_bytes, uint32_t box_cols,
                      uint32_t box_rows, CUtensorMapSwizzle swz) {
    const MapKey key{base, cols, rows, row_stride_bytes, box_cols, box_rows, int(dt), int(swz)};
    const size_t slot = map_slot(key);
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        if (g_map_cache[slot].valid && g_map_cache[slot].key == key) {
            *m = g_map_cache[slot].map;
            return W4A16_OK;
        }
    }
    w4a16_status st = get_encoder();
    if (st) return st;
    st = ensure_current_context();
    if (st) return st;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    (void)elem;
    CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(W4A16_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d) for a %llux%llu tensor",
                    int(r), (unsigned long long)rows, (unsigned long long)cols);
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_map_cache[slot].key = key;
    g_map_cache[slot].map = *m;
    g_map_cache[slot].valid = true;
    return W4A16_OK;
}

// --- device properties ------------------------------------------------------
w4a16_status device_sms(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 0 && dev < 64 && cache[dev]) {
        *sms = cache[dev];
        return W4A16_OK;
    }
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    if (dev >= 0 && dev < 64) cache[dev] = v;
    *sms = v;
    return W4A16_OK;
}

// --- router -----------------------------------------------------------------
// Crossover points measured on GB300 (decode kernel vs the fused tcgen05
// kernels): decode wins up to M = 16 on every measured layer.  The fused kernel
// with the dequantised tile in tensor memory beats the one with both operands
// in shared memory at every measured M (1 .. 4096); the latter stays reachable
// as W4A16_PATH_FUSED_SMEM.  The dense copy wins over fused dequant only where
// the tensor pipe, not the dequantisation, limits the fused kernel: at 1024
// tokens the fused kernel is level or ahead (14336x4096: 85 vs 91 us; 28672x8192:
// 313 vs 319 us), from 2048 the dense one mostly leads (28672x8192 M=4096: 1220
// vs 1325 us).
constexpr int64_t kDecodeUpToM = 16;
constexpr int64_t kDenseFromM = 2048;

int fused_kernel_for(int64_t) { return W4A16_PATH_FUSED_TMEM; }

// The route depends on the shape only: whether a small-M launch plan exists
// (its shared memory fits) does not depend on the SM count, which only changes
// the plan's K split and ring depth, chosen at launch from the live count.
int route_impl(const LayerShape& s, bool has_dense) {
    const int64_t M = s.M;
    // From 9 tokens (two MMA column tiles) at G = 32 with zero points, the small-M
    // kernel's per-group rescale and zero-point reload cost more than the fused
    // kernel's dequantisation except on large layers (measured, M = 9..16:
    // 14336x4096 16.9-18.0 vs 15.4-15.5 us, 4096x4096 7.6-8.1 vs 6.9 us, but
    // 28672x8192 46.4-47.1 vs 50.0 us; without zero points the small-M kernel is
    // ahead or level on every layer measured, 28672x8192 38.6 vs 48.5 us).
    const bool small_groups_zp = s.ng > 1 && s.g_eff <= 32 && s.zp && s.N * s.K < (int64_t(1) << 27);
    if (M <= kDecodeUpToM && !(M > 8 && small_groups_zp) && decode_plan_exists(M, s.N, s.K, s.g_eff, s.ng, s.zp))
        return W4A16_PATH_DECODE;
    if (has_dense && M >= kDenseFromM) return W4A16_PATH_DENSE;
    return fused_kernel_for(M);
}

int token_tile_for(int64_t M) {
    if (M <= 64) return 64;
    if (M <= 128) return 128;
    return 256;
}

w4a16_status launch_tcgen05(const void* A, const void* Wsrc, bool dense, const void* scales,
                            const int32_t* zeros, const void* bias, void* C, const LayerShape& s,
                            cudaStream_t stream) {
    if (dense) {
        // persistent dense-copy GEMM: 256-token tiles, one CTA per SM
        int sms = 0;
        w4a16_status st = device_sms(&sms);
        if (st) return st;
        CUtensorMap maps[2];
        st = make_map(&maps[0], A, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.K), uint64_t(s.M),
                      uint64_t(s.lda) * 2, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st) return st;
        st = make_map(&maps[1], Wsrc, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.K), uint64_t(s.N),
                      uint64_t(s.K) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st) return st;
        cudaError_t e = launch_dense_gemm(maps, C, bias, s, sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "dense GEMM launch");
        return W4A16_OK;
    }
    const int bt = token_tile_for(s.M);
    CUtensorMap maps[5];
    w4a16_status st = make_map(&maps[0], A, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.K),
                               uint64_t(s.M), uint64_t(s.lda) * 2, 64, uint32_t(bt),
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (st) return st;
    {
        st = make_map(&maps[1], Wsrc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, uint64_t(s.ldq), uint64_t(s.N),
                      uint64_t(s.ldq) * 4, 8, 128, CU_TENSOR_MAP_SWIZZLE_32B);
        if (st) return st;
        st = make_map(&maps[2], scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.lds),
                      uint64_t(s.ng), uint64_t(s.lds) * 2, 128, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st) return st;
        if (s.zp) {
            st = make_map(&maps[3], zeros, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, uint64_t(s.ldz),
                          uint64_t(s.ng), uint64_t(s.ldz) * 4, 16, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st) return st;
        } else {
            maps[3] = maps[2];   // unused without zero points
        }
    }
    // the output leaves by TMA store when its base and row pitch are 16-byte aligned
    const bool c_tma = (reinterpret_cast<uintptr_t>(C) & 15) == 0 && (s.ldc * 2) % 16 == 0;
    if (c_tma) {
        st = make_map(&maps[4], C, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.N), uint64_t(s.M),
                      uint64_t(s.ldc) * 2, 128, uint32_t(bt), CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st) return st;
    } else {
        maps[4] = maps[0];   // unused
    }
    cudaError_t e = launch_prefill(maps, C, bias, s, bt, c_tma, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tcgen05 GEMM launch");
    return W4A16_OK;
}

w4a16_status launch_tmem_path(const void* A, const void* Wq, const void* scales,
                              const int32_t* zeros, const void* bias, void* C, const LayerShape& s,
                              bool static_weights, cudaStream_t stream) {
    int sms = 0;
    w4a16_status st = device_sms(&sms);
    if (st) return st;
    const int bt = tmem_gemm_token_tile(s.M);
    // weight stages of 256 K-values: 128-byte packed rows and the group rows they span
    const uint32_t gps = uint32_t(decode_scale_box_rows(s.g_eff, s.ng));
    CUtensorMap maps[5];
    st = make_map(&maps[0], A, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.K), uint64_t(s.M),
                  uint64_t(s.lda) * 2, 64, uint32_t(bt), CU_TENSOR_MAP_SWIZZLE_128B);
    if (st) return st;
    st = make_map(&maps[1], Wq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, uint64_t(s.ldq), uint64_t(s.N),
                  uint64_t(s.ldq) * 4, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st) return st;
    st = make_map(&maps[2], scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.lds), uint64_t(s.ng),
                  uint64_t(s.lds) * 2, 128, gps, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st) return st;
    if (s.zp) {
        st = make_map(&maps[3], zeros, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, uint64_t(s.ldz),
                      uint64_t(s.ng), uint64_t(s.ldz) * 4, 16, gps, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st) return st;
    } else {
        maps[3] = maps[2];   // unused without zero points
    }
    // the output leaves by TMA store when its base and row pitch are 16-byte aligned
    const bool c_tma = (reinterpret_cast<uintptr_t>(C) & 15) == 0 && (s.ldc * 2) % 16 == 0;
    if (c_tma) {
        st = make_map(&maps[4], C, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.N), uint64_t(s.M),
                      uint64_t(s.ldc) * 2, 128, uint32_t(bt), CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st) return st;
    } else {
        maps[4] = maps[0];   // unused
    }
    cudaError_t e = launch_tmem_gemm(maps, C, bias, s, sms, static_weights, c_tma, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-memory GEMM launch");
    return W4A16_OK;
}

w4a16_status launch_decode_path(const void* A, const void* Wq, const void* scales,
                                const int32_t* zeros, const void* bias, void* C, const LayerShape& s,
                                bool static_weights, cudaStream_t stream) {
    int sms = 0;
    w4a16_status st = device_sms(&sms);
    if (st) return st;
    const uint32_t gps = uint32_t(decode_scale_box_rows(s.g_eff, s.ng));
    CUtensorMap maps[4];
    st = make_map(&maps[0], Wq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, uint64_t(s.ldq), uint64_t(s.N),
                  uint64_t(s.ldq) * 4, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st) return st;
    // one token tile (M <= 8): [M][256] boxes; more: [M][64] boxes with the 128-byte
    // swizzle, four per K box (the small-M kernel's activation sub-boxes)
    st = s.M <= 8 ? make_map(&maps[1], A, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.K), uint64_t(s.M),
                             uint64_t(s.lda) * 2, 256, uint32_t(s.M), CU_TENSOR_MAP_SWIZZLE_NONE)
                  : make_map(&maps[1], A, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.K), uint64_t(s.M),
                             uint64_t(s.lda) * 2, 64, uint32_t(s.M), CU_TENSOR_MAP_SWIZZLE_128B);
    if (st) return st;
    st = make_map(&maps[2], scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, uint64_t(s.lds), uint64_t(s.ng),
                  uint64_t(s.lds) * 2, 128, gps, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st) return st;
    if (s.zp) {
        st = make_map(&maps[3], zeros, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, uint64_t(s.ldz), uint64_t(s.ng),
                      uint64_t(s.ldz) * 4, 16, gps, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st) return st;
    } else {
        maps[3] = maps[2];   // unused without zero points
    }
    cudaError_t e = launch_decode(maps, C, bias, s, sms, static_weights, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode GEMM launch");
    return W4A16_OK;
}

}  // namespace

extern "C" {

int w4a16_version(void) { return 100; }

w4a16_status w4a16_selftest_wait_timeout(void* stream) {
    cudaError_t e = launch_wait_timeout(W4A16_SELFTEST_SITE, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test kernel launch");
    return W4A16_OK;
}

const char* w4a16_last_error_string(void) { return g_err; }

w4a16_status w4a16_packed_layout(int64_t N, int64_t K, int G, int qtype, int dtype,
                                 size_t* total_bytes, size_t* scales_off, size_t* zeros_off,
                                 int64_t* ldq_words) {
    LayerShape s;
    w4a16_status st = check_weight(N, K, G, qtype, dtype, &s);
    if (st) return st;
    const size_t q_bytes = size_t(N) * size_t(s.ldq) * 4;
    const size_t so = round_up(q_bytes, 256);
    const size_t s_bytes = size_t(s.ng) * size_t(s.lds) * 2;
    size_t zo = 0, end = so + s_bytes;
    if (s.zp) {
        zo = round_up(end, 256);
        end = zo + size_t(s.ng) * size_t(s.ldz) * 4;
    }
    if (total_bytes) *total_bytes = round_up(end, 256);
    if (scales_off) *scales_off = so;
    if (zeros_off) *zeros_off = zo;
    if (ldq_words) *ldq_words = s.ldq;
    g_err[0] = '\0';
    return W4A16_OK;
}

w4a16_status w4a16_pack_ex(const void* qsrc, int qformat, const void* scales, const int32_t* zeros,
                           int param_layout, void* Wpacked, int64_t N, int64_t K, int G, int qtype,
                           int dtype, void* stream) {
    LayerShape s;
    w4a16_status st = check_weight(N, K, G, qtype, dtype, &s);
    if (st) return st;
    if (qformat < W4A16_Q_UNPACKED || qformat > W4A16_Q_KN)
        return fail(W4A16_ERR_INVALID_ARG, "unknown weight format %d", qformat);
    if (param_layout != W4A16_LAYOUT_NG && param_layout != W4A16_LAYOUT_GN)
        return fail(W4A16_ERR_INVALID_ARG, "unknown scale/zero layout %d", param_layout);
    if (qformat == W4A16_Q_KN && N % 8)
        return fail(W4A16_ERR_INVALID_ARG, "the [K][N/8] format needs N divisible by 8, got N=%lld", (long long)N);
    const size_t qalign = qformat == W4A16_Q_UNPACKED ? 8 : 4;
    if (!qsrc || !aligned(qsrc, qalign))
        return fail(W4A16_ERR_INVALID_ARG, "q must be a non-null %zu-byte aligned device pointer", qalign);
    if (!Wpacked || !aligned(Wpacked, 256)) return fail(W4A16_ERR_INVALID_ARG, "Wpacked must be a non-null 256-byte aligned device pointer");
    if (!scales || !aligned(scales, 2)) return fail(W4A16_ERR_INVALID_ARG, "scales must be a non-null 2-byte aligned device pointer");
    if (s.zp && (!zeros || !aligned(zeros, 4))) return fail(W4A16_ERR_INVALID_ARG, "uint4 needs a non-null 4-byte aligned zeros pointer");
    if (!s.zp && zeros) return fail(W4A16_ERR_INVALID_ARG, "zeros must be NULL for uint4b8 (the zero point is the constant 8)");
    size_t total, so, zo;
    w4a16_packed_layout(N, K, G, qtype, dtype, &total, &so, &zo, nullptr);
    uint8_t* base = static_cast<uint8_t*>(Wpacked);
    cudaError_t e = launch_pack(qsrc, qformat, scales, zeros, param_layout == W4A16_LAYOUT_GN, base,
                                base + so, s.zp ? base + zo : nullptr, s, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    g_err[0] = '\0';
    return W4A16_OK;
}

w4a16_status w4a16_pack(const uint8_t* q, const void* scales, const int32_t* zeros, void* Wpacked,
                        int64_t N, int64_t K, int G, int qtype, int dtype, void* stream) {
    return w4a16_pack_ex(q, W4A16_Q_UNPACKED, scales, zeros, W4A16_LAYOUT_NG, Wpacked, N, K, G,
                         qtype, dtype, stream);
}

int w4a16_route(int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype, int has_dense) {
    LayerShape s;
    if (check_weight(N, K, G, qtype, dtype, &s) != W4A16_OK) return -1;
    if (M < 0 || M > kMaxDim) return -1;
    s.M = M;
    return route_impl(s, has_dense != 0);
}

w4a16_status w4a16_launch_plan(int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                               int path, int has_dense, int num_sms, w4a16_launch_info* info) {
    LayerShape s;
    w4a16_status st = check_weight(N, K, G, qtype, dtype, &s);
    if (st) return st;
    if (!info) return fail(W4A16_ERR_INVALID_ARG, "info must not be NULL");
    if (M < 1 || M > kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "M=%lld out of range", (long long)M);
    if (num_sms < 1 || num_sms > 4096) return fail(W4A16_ERR_INVALID_ARG, "num_sms=%d out of range", num_sms);
    if (path < W4A16_PATH_AUTO || path > W4A16_PATH_FUSED_SMEM) return fail(W4A16_ERR_INVALID_ARG, "unknown path %d", path);
    s.M = M;
    if (path == W4A16_PATH_AUTO) path = route_impl(s, has_dense != 0);
    if (path == W4A16_PATH_FUSED) path = fused_kernel_for(M);
    constexpr int64_t kRows = 128;   // weight rows per CTA tile in every GEMM kernel
    const int64_t row_tiles = (N + kRows - 1) / kRows;
    w4a16_launch_info r = {path, 0, 1, 0, 0, 0};
    if (path == W4A16_PATH_DECODE) {
        if (M > kDecodeMaxM) return fail(W4A16_ERR_INVALID_ARG, "the decode path takes M <= %lld", (long long)kDecodeMaxM);
        int ks, stages, nt;
        size_t smem;
        if (!plan_decode(M, N, K, s.g_eff, s.ng, s.zp, num_sms, &ks, &stages, &smem, &nt))
            return fail(W4A16_ERR_UNSUPPORTED, "decode path: no launch plan fits for M=%lld, K=%lld", (long long)M, (long long)K);
        r.token_tile = 8 * nt;
        r.k_split = ks;
        r.stages = stages;
        r.grid = row_tiles * ks;
        r.smem_bytes = int64_t(smem);
    } else if (path == W4A16_PATH_FUSED_TMEM) {
        const int bt = tmem_gemm_token_tile(M);
        r.token_tile = bt;
        r.k_split = tmem_gemm_ksplit(M, N, K, num_sms);
        r.grid = tmem_gemm_grid(M, N, K, num_sms);
    } else if (path == W4A16_PATH_FUSED_SMEM) {
        const int bt = token_tile_for(M);
        r.token_tile = bt;
        r.grid = row_tiles * ((M + bt - 1) / bt);
    } else {   // W4A16_PATH_DENSE: persistent, one CTA per SM at most
        const int64_t tiles = row_tiles * ((M + 255) / 256);
        r.token_tile = 256;
        r.grid = tiles < num_sms ? tiles : num_sms;
    }
    *info = r;
    g_err[0] = '\0';
    return W4A16_OK;
}

w4a16_status w4a16_linear(const void* A, int64_t lda, const void* Wq, const void* scales,
                          const int32_t* zeros, const void* bias, const void* Wdense, void* C,
                          int64_t ldc, int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                          int path, void* stream) {
    LayerShape s;
    w4a16_status st = check_weight(N, K, G, qtype, dtype, &s);
    if (st) return st;
    if (M < 0 || M > kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "M=%lld out of range", (long long)M);
    const int opts = path & ~0xFF;
    path &= 0xFF;
    if (opts & ~W4A16_OPT_STATIC_WEIGHTS) return fail(W4A16_ERR_INVALID_ARG, "unknown option bits 0x%x", opts);
    if (path < W4A16_PATH_AUTO || path > W4A16_PATH_FUSED_SMEM) return fail(W4A16_ERR_INVALID_ARG, "unknown path %d", path);
    st = check_qptrs(Wq, scales, zeros, qtype);
    if (st) return st;
    if (!A || !aligned(A, 16)) return fail(W4A16_ERR_INVALID_ARG, "A must be a non-null 16-byte aligned device pointer");
    if (!C || !aligned(C, 2)) return fail(W4A16_ERR_INVALID_ARG, "C must be a non-null 2-byte aligned device pointer");
    if (Wdense && !aligned(Wdense, 16)) return fail(W4A16_ERR_INVALID_ARG, "Wdense must be 16-byte aligned");
    if (bias && !aligned(bias, 2)) return fail(W4A16_ERR_INVALID_ARG, "bias must be 2-byte aligned");
    if (lda == 0) lda = K;
    if (ldc == 0) ldc = N;
    if (lda < K || lda > kMaxDim || lda % 8)
        return fail(W4A16_ERR_INVALID_ARG, "lda=%lld must be >= K=%lld and a multiple of 8 (16-byte row pitch)", (long long)lda, (long long)K);
    if (ldc < N || ldc > kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "ldc=%lld must be >= N=%lld", (long long)ldc, (long long)N);
    s.lda = lda;
    s.ldc = ldc;
    s.M = M;
    if (path == W4A16_PATH_AUTO) path = route_impl(s, Wdense != nullptr);
    if (path == W4A16_PATH_FUSED) path = fused_kernel_for(M);
    if (path == W4A16_PATH_DENSE && !Wdense) return fail(W4A16_ERR_INVALID_ARG, "the dense path needs a dense copy (Wdense)");
    if (path == W4A16_PATH_DECODE) {
        if (M > kDecodeMaxM) return fail(W4A16_ERR_INVALID_ARG, "the decode path takes M <= %lld", (long long)kDecodeMaxM);
        if (M > 0 && !decode_plan_exists(M, N, K, s.g_eff, s.ng, s.zp))
            return fail(W4A16_ERR_UNSUPPORTED, "decode path: the activation slice for M=%lld, K=%lld does not fit in shared memory", (long long)M, (long long)K);
    }
    g_err[0] = '\0';
    if (M == 0) return W4A16_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool static_weights = (opts & W4A16_OPT_STATIC_WEIGHTS) != 0;
    if (path == W4A16_PATH_DECODE)
        return launch_decode_path(A, Wq, scales, zeros, bias, C, s, static_weights, cs);
    if (path == W4A16_PATH_DENSE) return launch_tcgen05(A, Wdense, true, nullptr, nullptr, bias, C, s, cs);
    if (path == W4A16_PATH_FUSED_SMEM) return launch_tcgen05(A, Wq, false, scales, zeros, bias, C, s, cs);
    return launch_tmem_path(A, Wq, scales, zeros, bias, C, s, static_weights, cs);
}

w4a16_status w4a16_gemm_ex(const void* A, const void* Wq, const void* scales,
                           const int32_t* zeros, const void* Wdense, void* C, int64_t M,
                           int64_t N, int64_t K, int G, int qtype, int dtype, int path,
                           void* stream) {
    return w4a16_linear(A, 0, Wq, scales, zeros, nullptr, Wdense, C, 0, M, N, K, G, qtype, dtype,
                        path, stream);
}

w4a16_status w4a16_gemm(const void* A, const void* Wq, const void* scales, const int32_t* zeros,
                        void* C, int64_t M, int64_t N, int64_t K, int G, int qtype, int dtype,
                        void* stream) {
    return w4a16_gemm_ex(A, Wq, scales, zeros, nullptr, C, M, N, K, G, qtype, dtype,
                         W4A16_PATH_AUTO, stream);
}

w4a16_status w4a16_dequant(const void* Wq, const void* scales, const int32_t* zeros, void* W,
                           int64_t N, int64_t K, int G, int qtype, int dtype, void* stream) {
    LayerShape s;
    w4a16_status st = check_weight(N, K, G, qtype, dtype, &s);
    if (st) return st;
    st = check_qptrs(Wq, scales, zeros, qtype);
    if (st) return st;
    if (!W || !aligned(W, 16)) return fail(W4A16_ERR_INVALID_ARG, "W must be a non-null 16-byte aligned device pointer");
    cudaError_t e = launch_dequant(static_cast<const uint32_t*>(Wq), scales, zeros, W, s,
                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
    g_err[0] = '\0';
    return W4A16_OK;
}

w4a16_status w4a16_gemm_dense(const void* A, const void* W, void* C, int64_t M, int64_t N,
                              int64_t K, int dtype, void* stream) {
    if (dtype != W4A16_FP16 && dtype != W4A16_BF16)
        return fail(W4A16_ERR_INVALID_ARG, "dtype %d is not fp16 (0) or bf16 (1)", dtype);
    if (M < 0 || M > kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "M=%lld out of range", (long long)M);
    if (N < 1 || N > kMaxDim) return fail(W4A16_ERR_INVALID_ARG, "N=%lld out of range", (long long)N);
    if (K < 16 || K > kMaxDim || K % 16) return fail(W4A16_ERR_INVALID_ARG, "K=%lld must be a positive multiple of 16", (long long)K);
    if (!A || !aligned(A, 16)) return fail(W4A16_ERR_INVALID_ARG, "A must be a non-null 16-byte aligned device pointer");
    if (!W || !aligned(W, 16)) return fail(W4A16_ERR_INVALID_ARG, "W must be a non-null 16-byte aligned device pointer");
    if (!C || !aligned(C, 2)) return fail(W4A16_ERR_INVALID_ARG, "C must be a non-null 2-byte aligned device pointer");
    g_err[0] = '\0';
    if (M == 0) return W4A16_OK;
    LayerShape s;
    s.M = M;
    s.N = N;
    s.K = K;
    s.g_eff = K;
    s.ng = 1;
    s.ldq = (K / 8 + 3) / 4 * 4;
    s.lds = (N + 7) / 8 * 8;
    s.ldz = (N / 8 + 3) / 4 * 4;
    s.bf16 = dtype == W4A16_BF16;
    s.zp = false;
    s.lda = K;
    s.ldc = N;
    return launch_tcgen05(A, W, true, nullptr, nullptr, nullptr, C, s, static_cast<cudaStream_t>(stream));
}

w4a16_status w4a16_device_status(int* site) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    // read and clear every module's word, then report the first set one
    const int words[5] = {take_status_decode(), take_status_prefill(), take_status_tmem_gemm(),
                          take_status_dense(), take_status_selftest()};
    int v = 0;
    for (int w : words) {
        if (w < 0) {
            v = -1;
            break;
        }
        if (v == 0 && w > 0) v = w;
    }
    if (site) *site = v > 0 ? v : 0;
    if (v < 0) return fail(W4A16_ERR_CUDA, "reading the device status word failed");
    if (v > 0) return fail(W4A16_ERR_DEVICE_TIMEOUT, "a kernel barrier wait timed out at site %d", v);
    return W4A16_OK;
}

}  // extern "C"
