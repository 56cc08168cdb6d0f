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

// ExLlama position of K-value i (0..7) within its word.
__device__ __forceinline__ int exl_shift(int i) { return 4 * (i >> 1) + 16 * (i & 1); }

// GPTQ / compressed-tensors words [N][K/8] (K-value 8j+i at bits 4i) -> the
// packed section: the eight nibbles of each word move to their ExLlama places.
__global__ void __launch_bounds__(kThreads) repack_gptq_kernel(const uint32_t* __restrict__ src,
                                                               uint32_t* __restrict__ out, int N,
                                                               int K, int ldq) {
    const int k8 = K / 8;
    for (int n = blockIdx.x; n < N; n += gridDim.x) {
        const uint32_t* srow = src + int64_t(n) * k8;
        uint32_t* orow = out + int64_t(n) * ldq;
        for (int j = threadIdx.x; j < ldq; j += kThreads) {
            uint32_t w = 0;
            if (j < k8) {
                const uint32_t v = __ldg(srow + j);
#pragma unroll
                for (int i = 0; i < 8; ++i) w |= ((v >> (4 * i)) & 0xFu) << exl_shift(i);
            }
            orow[j] = w;
        }
    }
}

// ExLlama words [N][K/8] -> the packed section: the same words, row pitch ldq.
__global__ void __launch_bounds__(kThreads) repack_exllama_kernel(const uint32_t* __restrict__ src,
                                                                  uint32_t* __restrict__ out, int N,
                                                                  int K, int ldq) {
    const int k8 = K / 8;
    for (int n = blockIdx.x; n < N; n += gridDim.x)
        for (int j = threadIdx.x; j < ldq; j += kThreads)
            out[int64_t(n) * ldq + j] = j < k8 ? __ldg(src + int64_t(n) * k8 + j) : 0u;
}

// The MI300 layout [K][N/8] (N-value 8c+i of row k at bits 4i) -> the packed
// section.  Item (j, c): the eight source words of K-values 8j..8j+7 at column
// c give output word j of rows 8c..8c+7.  Consecutive threads take consecutive
// columns, so the source reads are coalesced.
__global__ void __launch_bounds__(kThreads) repack_kn_kernel(const uint32_t* __restrict__ src,
                                                             uint32_t* __restrict__ out, int N, int K,
                                                             int ldq) {
    const int n8 = N / 8, k8 = K / 8;
    const int64_t items = int64_t(ldq) * n8;
    for (int64_t it = int64_t(blockIdx.x) * kThreads + threadIdx.x; it < items;
         it += int64_t(gridDim.x) * kThreads) {
        const int j = int(it / n8), c = int(it % n8);
        uint32_t v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = j < k8 ? __ldg(src + int64_t(8 * j + t) * n8 + c) : 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t w = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) w |= ((v[t] >> (4 * i)) & 0xFu) << exl_shift(t);
            out[int64_t(8 * c + i) * ldq + j] = w;
        }
    }
}

// [rows][cols] (row-major) -> [rows][ld] with zero padding for c >= cols.
template <typename T>
__global__ void __launch_bounds__(kThreads) copy_pad_kernel(const T* __restrict__ src,
                                                            T* __restrict__ dst, int64_t rows,
                                                            int64_t cols, int64_t ld) {
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x)
        for (int64_t c = threadIdx.x; c < ld; c += kThreads)
            dst[r * ld + c] = c < cols ? src[r * cols + c] : T(0);
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
        // four independent word loads per thread in flight, each warp-coalesced.
        // Packed words are read and the dense rows written once, both with the
        // streaming (evict-first) cache policy: together 74 -> 88 % of HBM on
        // 14336 x 4096 (29.4 -> 24.6 us), either one alone changed nothing.
        for (int j0 = threadIdx.x; j0 < k8; j0 += kUnroll * kThreads) {
            uint32_t w[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * kThreads;
                w[u] = j < k8 ? __ldcs(qrow + j) : 0u;
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
                __stcs(&orow[j], o);
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

cudaError_t launch_pack(const void* qsrc, int qformat, const void* scales, const int32_t* zeros,
                        bool groups_first, void* Wq, void* scales_dst, void* zeros_dst,
                        const LayerShape& s, cudaStream_t stream) {
    auto* out = static_cast<uint32_t*>(Wq);
    const int N = int(s.N), K = int(s.K), ldq = int(s.ldq);
    switch (qformat) {
        case kQUnpacked:
            pack_q_kernel<<<grid_for(s.N), kThreads, 0, stream>>>(static_cast<const uint8_t*>(qsrc), out, N, K, ldq);
            break;
        case kQGptq:
            repack_gptq_kernel<<<grid_for(s.N), kThreads, 0, stream>>>(static_cast<const uint32_t*>(qsrc), out, N, K, ldq);
            break;
        case kQExllama:
            repack_exllama_kernel<<<grid_for(s.N), kThreads, 0, stream>>>(static_cast<const uint32_t*>(qsrc), out, N, K, ldq);
            break;
        default: {
            const int64_t items = s.ldq * (s.N / 8);
            int64_t blocks = (items + kThreads - 1) / kThreads;
            if (blocks > 152 * 32) blocks = 152 * 32;
            repack_kn_kernel<<<int(blocks < 1 ? 1 : blocks), kThreads, 0, stream>>>(static_cast<const uint32_t*>(qsrc), out, N, K, ldq);
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // scales -> [ng][lds], zero points -> [ng][ldz]: transposed from the
    // [N][ng] / [N/8][ng] layout, copied from [ng][N] / [ng][N/8]
    const auto* sc = static_cast<const uint16_t*>(scales);
    auto* scd = static_cast<uint16_t*>(scales_dst);
    if (groups_first) copy_pad_kernel<uint16_t><<<grid_for(s.ng), kThreads, 0, stream>>>(sc, scd, s.ng, s.N, s.lds);
    else transpose_pad_kernel<uint16_t><<<grid_for(s.ng), kThreads, 0, stream>>>(sc, scd, s.N, s.ng, s.lds);
    e = cudaGetLastError();
    if (e != cudaSuccess || !s.zp) return e;
    auto* zd = static_cast<int32_t*>(zeros_dst);
    if (groups_first) copy_pad_kernel<int32_t><<<grid_for(s.ng), kThreads, 0, stream>>>(zeros, zd, s.ng, s.N / 8, s.ldz);
    else transpose_pad_kernel<int32_t><<<grid_for(s.ng), kThreads, 0, stream>>>(zeros, zd, s.N / 8, s.ng, s.ldz);
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
