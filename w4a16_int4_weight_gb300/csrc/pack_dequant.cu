// Packer and dense dequantiser.  Both are single-pass HBM-bound kernels.  A
// CTA walks whole rows (grid-stride over n); its threads stride over the row's
// packed words, so consecutive threads touch consecutive words: a warp reads
// 128 (dequant) or 1024 (pack) contiguous bytes and writes 512 (dequant) or
// 128 (pack), with no integer division in the loops.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // dequant: packed words per thread per iteration

// Eight bytes (K-values v0..v7 of one row, low nibble each) -> one packed word
// with nibbles v0,v2,v4,v6,v1,v3,v5,v7 from low to high.
__device__ __forceinline__ uint32_t pack8(uint2 b) {
    const uint32_t e = b.x & 0x0F0F0F0Fu;   // v0 v1 v2 v3 (one per byte)
    const uint32_t f = b.y & 0x0F0F0F0Fu;   // v4 v5 v6 v7
    return (e & 0xFu) | (((e >> 16) & 0xFu) << 4) | ((f & 0xFu) << 8) |
           (((f >> 16) & 0xFu) << 12) | (((e >> 8) & 0xFu) << 16) | (((e >> 24) & 0xFu) << 20) |
           (((f >> 8) & 0xFu) << 24) | (((f >> 24) & 0xFu) << 28);
}

// Row n of q (K bytes) -> row n of the packed section (ldq words, the words
// past K/8 zero).
__global__ void __launch_bounds__(kThreads) pack_q_kernel(const uint8_t* __restrict__ q,
                                                          uint32_t* __restrict__ out, int N, int K,
                                                          int ldq) {
    const int k8 = K / 8;
    for (int n = blockIdx.x; n < N; n += gridDim.x) {
        const uint8_t* row = q + int64_t(n) * K;
        uint32_t* orow = out + int64_t(n) * ldq;
        for (int j = threadIdx.x; j < ldq; j += kThreads)
            orow[j] = j < k8 ? pack8(__ldg(reinterpret_cast<const uint2*>(row) + j)) : 0u;
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
    for (int64_t c = blockIdx.x; c < cols; c += gridDim.x)
        for (int64_t r = threadIdx.x; r < ld; r += kThreads)
            dst[c * ld + r] = r < rows ? src[r * cols + c] : T(0);
}

// W[n][8j .. 8j+7] = rne((q - z) * s) for packed word j of row n.  gshift:
// log2(G_eff) when there are several groups (G_eff a power of two), 31 when
// one group spans K.
template <bool BF16, bool ZP>
__global__ void __launch_bounds__(kThreads) dequant_kernel(
    const uint32_t* __restrict__ wq, const uint16_t* __restrict__ scales,
    const int32_t* __restrict__ zeros, uint16_t* __restrict__ out, int N, int K, int ldq,
    int gshift, int64_t lds, int64_t ldz) {
    const int k8 = K / 8;
    for (int n = blockIdx.x; n < N; n += gridDim.x) {
        const uint32_t* qrow = wq + int64_t(n) * ldq;
        uint4* orow = reinterpret_cast<uint4*>(out + int64_t(n) * K);
        const int zsh = 4 * (n & 7);
        // four independent word loads per thread in flight, each warp-coalesced
        for (int j0 = threadIdx.x; j0 < k8; j0 += kUnroll * kThreads) {
            uint32_t w[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * kThreads;
                w[u] = j < k8 ? __ldg(qrow + j) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * kThreads;
                if (j >= k8) break;
                const int g = (8 * j) >> gshift;
                const uint32_t sb = __ldg(scales + int64_t(g) * lds + n);
                int z = 8;
                if constexpr (ZP) z = int(uint32_t(__ldg(zeros + int64_t(g) * ldz + (n >> 3))) >> zsh) & 0xF;
                const uint32_t s2 = __byte_perm(sb, 0u, 0x1010);
                uint32_t p[4];
                unpack_word<BF16>(w[u], make_zero_const<BF16>(z), p);
                uint4 o;
                o.x = scale_pair<BF16>(p[0], s2);
                o.y = scale_pair<BF16>(p[1], s2);
                o.z = scale_pair<BF16>(p[2], s2);
                o.w = scale_pair<BF16>(p[3], s2);
                orow[j] = o;
            }
        }
    }
}

// One CTA per row, at most 32 per SM of a 152-SM GPU (grid-stride beyond).
int grid_for(int64_t rows) {
    int64_t blocks = rows;
    if (blocks > 152 * 32) blocks = 152 * 32;
    return blocks < 1 ? 1 : int(blocks);
}

int group_shift(const LayerShape& s) {
    if (s.ng == 1) return 31;
    int sh = 0;
    while ((int64_t(1) << sh) < s.g_eff) ++sh;
    return sh;
}

}  // namespace

cudaError_t launch_pack(const uint8_t* q, const void* scales, const int32_t* zeros, void* Wq,
                        void* scales_dst, void* zeros_dst, const LayerShape& s,
                        cudaStream_t stream) {
    pack_q_kernel<<<grid_for(s.N), kThreads, 0, stream>>>(q, static_cast<uint32_t*>(Wq), int(s.N),
                                                           int(s.K), int(s.ldq));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    transpose_pad_kernel<uint16_t><<<grid_for(s.ng), kThreads, 0, stream>>>(
        static_cast<const uint16_t*>(scales), static_cast<uint16_t*>(scales_dst), s.N, s.ng, s.lds);
    e = cudaGetLastError();
    if (e != cudaSuccess || !s.zp) return e;
    transpose_pad_kernel<int32_t><<<grid_for(s.ng), kThreads, 0, stream>>>(
        zeros, static_cast<int32_t*>(zeros_dst), s.N / 8, s.ng, s.ldz);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* Wq, const void* scales, const int32_t* zeros,
                           void* W, const LayerShape& s, cudaStream_t stream) {
    const auto* sc = static_cast<const uint16_t*>(scales);
    auto* out = static_cast<uint16_t*>(W);
    const int grid = grid_for(s.N);
    const int N = int(s.N), K = int(s.K), ldq = int(s.ldq);
    const int64_t lds = s.lds, ldz = s.ldz;
    const int gsh = group_shift(s);
    if (s.bf16) {
        if (s.zp) dequant_kernel<true, true><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, N, K, ldq, gsh, lds, ldz);
        else dequant_kernel<true, false><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, N, K, ldq, gsh, lds, ldz);
    } else {
        if (s.zp) dequant_kernel<false, true><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, N, K, ldq, gsh, lds, ldz);
        else dequant_kernel<false, false><<<grid, kThreads, 0, stream>>>(Wq, sc, zeros, out, N, K, ldq, gsh, lds, ldz);
    }
    return cudaGetLastError();
}

}  // namespace w4a16
