// Internal launch interface between the C ABI (w4a16_api.cu) and the kernel
// modules.  Arguments are already validated when these are called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

struct LayerShape {
    int64_t M, N, K;
    int64_t g_eff;   // group size with -1 resolved to K
    int64_t ng;      // K / g_eff
    int64_t ldq;     // packed row pitch in 32-bit words
    bool bf16;       // activation dtype
    bool zp;         // explicit zero points (uint4)
};

// pack_dequant.cu
cudaError_t launch_pack(const uint8_t* q, const void* scales, const int32_t* zeros, void* Wq,
                        void* scales_dst, void* zeros_dst, const LayerShape& s,
                        cudaStream_t stream);
cudaError_t launch_dequant(const uint32_t* Wq, const void* scales, const int32_t* zeros,
                           void* W, const LayerShape& s, cudaStream_t stream);

// decode.cu: small-M split-K kernel, M <= kDecodeMaxM.
constexpr int64_t kDecodeMaxM = 64;
cudaError_t launch_decode(const CUtensorMap& tmap_q, const void* A, const void* scales,
                          const int32_t* zeros, void* C, const LayerShape& s,
                          int num_sms, cudaStream_t stream);

// prefill.cu: tcgen05 GEMM, fused-dequant (Wq != null) or dense (tmap_w dense).
cudaError_t launch_prefill(const CUtensorMap& tmap_a, const CUtensorMap& tmap_w,
                           const void* scales, const int32_t* zeros, void* C,
                           const LayerShape& s, bool dense, int token_tile,
                           cudaStream_t stream);

// Status words of each module: read-and-clear (synchronous).
int take_status_decode();
int take_status_prefill();

}  // namespace w4a16
