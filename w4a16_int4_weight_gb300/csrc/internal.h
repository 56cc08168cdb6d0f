// Internal launch interface between the C ABI (w4a16_api.cu) and the kernel
// modules.  Arguments are already validated when these are called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <unordered_map>

namespace w4a16 {

// Dynamic shared memory a kernel may use: cudaFuncSetAttribute once per
// (kernel, device) and size increase, since the attribute is a per-function
// maximum that stays set.
inline cudaError_t ensure_smem(const void* func, int bytes) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> granted;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = uint64_t(reinterpret_cast<uintptr_t>(func)) * 64u + uint64_t(dev & 63);
    std::lock_guard<std::mutex> lk(mu);
    auto it = granted.find(key);
    if (it != granted.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) granted[key] = bytes;
    return e;
}

struct LayerShape {
    int64_t M, N, K;
    int64_t g_eff;   // group size with -1 resolved to K
    int64_t ng;      // K / g_eff
    int64_t ldq;     // packed row pitch in 32-bit words
    int64_t lds;     // transposed scale row pitch in elements: round_up(N, 8)
    int64_t ldz;     // transposed zero-point row pitch in words: round_up(N/8, 4)
    bool bf16;       // activation dtype
    bool zp;         // explicit zero points (uint4)
    int64_t lda = 0; // row pitch of A in elements (>= K, a multiple of 8)
    int64_t ldc = 0; // row pitch of C in elements (>= N)
};

// pack_dequant.cu.  qformat: the w4a16_qformat values; groups_first: scales
// [ng][N] and zeros [ng][N/8] (else [N][ng] and [N/8][ng]).
constexpr int kQUnpacked = 0, kQGptq = 1, kQExllama = 2, kQKn = 3;
cudaError_t launch_pack(const void* qsrc, int qformat, const void* scales, const int32_t* zeros,
                        bool groups_first, void* Wq, void* scales_dst, void* zeros_dst,
                        const LayerShape& s, cudaStream_t stream);
cudaError_t launch_dequant(const uint32_t* Wq, const void* scales, const int32_t* zeros,
                           void* W, const LayerShape& s, cudaStream_t stream);

// decode.cu: small-M split-K kernel, M <= kDecodeMaxM.
constexpr int64_t kDecodeMaxM = 64;
// maps: packed q [N][ldq] u32 box {32,128} SW128; A [M][K] box {256,M} (M <= 8) or {64,M} SW128;
// scales [ng][lds] box {128, decode_scale_box_rows}; zeros [ng][ldz] box {16, same}.
// prefetch_weights: the weights are not written by work still running on the
// stream, so they may be fetched before the previous grid completes.
// bias (all three GEMMs): [N] dtype added to the fp32 result before its rounding, or null.
cudaError_t launch_decode(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                          int num_sms, bool prefetch_weights, cudaStream_t stream);
int decode_scale_box_rows(int64_t g_eff, int64_t ng);
bool plan_decode(int64_t M, int64_t N, int64_t K, int64_t g_eff, int64_t ng, bool zp,
                 int num_sms, int* ks_out, int* stages_out, size_t* smem_out, int* nt_out);
// Whether any plan fits the shape (independent of the SM count).
bool decode_plan_exists(int64_t M, int64_t N, int64_t K, int64_t g_eff, int64_t ng, bool zp);

// prefill.cu: fused-dequant tcgen05 GEMM with the dequantised tile in shared memory.
// maps: A [M][K] box {64,BT} SW128; packed [N][ldq] box {8,128} SW32; scales [ng][lds]
// box {128,2}; zeros [ng][ldz] box {16,2}.
cudaError_t launch_prefill(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                           int token_tile, bool c_tma, cudaStream_t stream);   // maps[4]: C, when c_tma

// tmem_gemm.cu: fused-dequant tcgen05 GEMM with the weight tile in tensor memory.
// maps: A [M][K] box {64, BT} SW128 (BT = tmem_gemm_token_tile(M)); packed
// [N][ldq] box {32,128} SW128; scales [ng][lds] box {128, gps}; zeros [ng][ldz]
// box {16, gps}, gps = decode_scale_box_rows(g_eff, ng); maps[4]: C [M][N] box {128, BT},
// valid when c_tma (16-byte aligned base and row pitch).
int tmem_gemm_token_tile(int64_t M);
// CTAs per cluster that split K (1, 2, 4 or 8) for the tensor-memory kernel.
int tmem_gemm_ksplit(int64_t M, int64_t N, int64_t K, int num_sms);
// The K split, the number of clusters that take whole tiles instead (see
// tmem_gemm.cu), and the grid of a launch.
void tmem_gemm_split(int64_t M, int64_t N, int64_t K, int num_sms, int* ks, int* whole_pairs, int* red_in_ring);
int64_t tmem_gemm_grid(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_tmem_gemm(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                             int num_sms, bool prefetch_weights, bool c_tma, cudaStream_t stream);
int take_status_tmem_gemm();

// Status words of each module: read-and-clear (synchronous).
int take_status_decode();
int take_status_prefill();

// dense_gemm.cu: persistent dense-copy GEMM (one CTA per SM, two tensor-memory
// accumulators).  maps: A [M][K] box {64, 256} SW128; dense weight [N][K] box {64, 128} SW128.
cudaError_t launch_dense_gemm(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                              int num_sms, cudaStream_t stream);
int take_status_dense();

// selftest.cu: one warp waits on an mbarrier that nothing completes; the bounded
// wait gives up after its limit and records `site` in this module's status word.
cudaError_t launch_wait_timeout(int site, cudaStream_t stream);
int take_status_selftest();

}  // namespace w4a16
