// Packer and dense dequantiser.  Both are single-pass HBM-bound kernels: one
// thread handles four packed words (32 K-values) of one row, so every global
// access is a 16-byte vector (the q read is four 8-byte vectors).
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kThreads = 256;

// Eight bytes (K-values v0..v7 of one row, low nibble each) -> one packed word
// with nibbles v0,v2,v4,v6,v1,v3,v5,v7 from low to high.
__device__ __forceinline__ uint32_t pack8(uint2 b) {
    const uint32_t e = b.x & 0x0F0F0F0Fu;   // v0 v1 v2 v3 (one per byte)
    const uint32_t f = b.y & 0x0F0F0F0Fu;   // v4 v5 v6 v7
    return (e & 0xFu) | (((e >> 16) & 0xFu) << 4) | ((f & 0xFu) << 8) |
           (((f >> 16) & 0xFu) << 12) | (((e >> 8) & 0xFu) << 16) | (((e >> 24) & 0xFu) << 20) |
           (((f >> 8) & 0xFu) << 24) | (((f >> 24) & 0xFu) << 28);
}

__global__ void __launch_bounds__(kThreads) pack_q_kernel(const uint8_t* __restrict__ q,
                                                          uint32_t* __restrict__ out, int64_t N,
                                                          int64_t K, int64_t ldq) {
    const int64_t k8 = K / 8, l4 = ldq / 4, total = N * l4;
    for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * kThreads) {
        const int64_t n = i / l4, j0 = (i % l4) * 4;
        const uint8_t* row = q + n * K;
        uint4 w;
        uint32_t* wv = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int64_t j = j0 + t;
            wv[t] = j < k8 ? pack8(__ldg(reinterpret_cast<const uint2*>(row + 8 * j))) : 0u;
        }
        *reinterpret_cast<uint4*>(out + n * ldq + j0) = w;
    }
}

// [rows][cols] (row-major) -> [cols][ld] with zero padding for r >= rows.  The
// output is written in full and in order (coalesced); the strided reads touch
// each input element once.  Scales and zero points are a small fraction of the
// weight, and this runs once per weight.
template <typename T>
__global__ void __launch_bounds__(kThreads) transpose_pad_kernel(const T* __restrict__ src,
                                                                 T* __restrict__ dst, int64_t rows,
                                                                 int64_t cols, int64_t ld) {
    const int64_t total = cols * ld;
    for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * kThreads) {
        const int64_t c = i / ld, r = i % ld;
        dst[i] = r < rows ? src[r * cols + c] : T(0);
    }
}

template <bool BF16, bool ZP>
__global__ void __launch_bounds__(kThreads) dequant_kernel(
    const uint32_t* __restrict__ wq, const uint16_t* __restrict__ scales,
    const int32_t* __restrict__ zeros, uint16_t* __restrict__ out, int64_t N, int64_t K,
    int64_t ldq, int64_t g_eff, int64_t lds, int64_t ldz) {
    const int64_t k8 = K / 8, l4 = (k8 + 3) / 4, total = N * l4;
    for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * kThreads) {
        const int64_t n = i / l4, j0 = (i % l4) * 4;
        const uint4 words = __ldg(reinterpret_cast<const uint4*>(wq + n * ldq + j0));
        const uint32_t* wv = reinterpret_cast<const uint32_t*>(&words);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int64_t j = j0 + t;
            if (j >= k8) break;
            const int64_t g = (8 * j) / g_eff;   // g_eff is a multiple of 8: one group per word
            const uint16_t sb = __ldg(scales + g * lds + n);
            int z = 8;
            if constexpr (ZP) z = (__ldg(zeros + g * ldz + n / 8) >> (4 * (n % 8))) & 0xF;
            const uint32_t s2 = uint32_t(sb) | (uint32_t(sb) << 16);
            uint32_t p[4];
            unpack_word<BF16>(wv[t], make_zero_const<BF16>(z), p);
            uint4 o;
            o.x = scale_pair<BF16>(p[0], s2);
            o.y = scale_pair<BF16>(p[1], s2);
            o.z = scale_pair<BF16>(p[2], s2);
            o.w = scale_pair<BF16>(p[3], s2);
            *reinterpret_cast<uint4*>(out + n * K + 8 * j) = o;
        }
    }
}

int grid_for(int64_t items) {
    int64_t blocks = (items + kThreads - 1) / kThreads;
    if (blocks > 152 * 32) blocks = 152 * 32;
    return blocks < 1 ? 1 : int(blocks);
}

}  // namespace

cudaError_t launch_pack(const uint8_t* q, const void* scales, const int32_t* zeros, void* Wq,
                        void* scales_dst, void* zeros_dst, const LayerShape& s,
                        cudaStream_t stream) {
    const int64_t items = s.N * (s.ldq / 4);
    pack_q_kernel<<<grid_for(items), kThreads, 0, stream>>>(q, static_cast<uint32_t*>(Wq), s.N,
                                                             s.K, s.ldq);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    transpose_pad_kernel<uint16_t><<<grid_for(s.ng * s.lds), kThreads, 0, stream>>>(
        static_cast<const uint16_t*>(scales), static_cast<uint16_t*>(scales_dst), s.N, s.ng, s.lds);
    e = cudaGetLastError();
    if (e != cudaSuccess || !s.zp) return e;
    transpose_pad_kernel<int32_t><<<grid_for(s.ng * s.ldz), kThreads, 0, stream>>>(
        zeros, static_cast<int32_t*>(zeros_dst), s.N / 8, s.ng, s.ldz);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* Wq, const void* scales, const int32_t* zeros,
                           void* W, const LayerShape& s, cudaStream_t stream) {
    const int64_t items = s.N * ((s.K / 8 + 3) / 4);
    const auto* sc = static_cast<const uint16_t*>(scales);
    auto* out = static_cast<uint16_t*>(W);
    const int grid = grid_for(items);
    if (s.bf16) {
        if (s.zp) dequant_kernel<true, true><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, s.N, s.K, s.ldq, s.g_eff, s.lds, s.ldz);
        else dequant_kernel<true, false><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, s.N, s.K, s.ldq, s.g_eff, s.lds, s.ldz);
    } else {
        if (s.zp) dequant_kernel<false, true><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, s.N, s.K, s.ldq, s.g_eff, s.lds, s.ldz);
        else dequant_kernel<false, false><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, s.N, s.K, s.ldq, s.g_eff, s.lds, s.ldz);
    }
    return cudaGetLastError();
}

}  // namespace w4a16
