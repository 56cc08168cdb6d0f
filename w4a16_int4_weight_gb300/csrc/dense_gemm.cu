// Dense-copy GEMM (the pages' cached dense-dequant path: _cache_dequant_weight,
// then a plain dot on the dtype copy), persistent on GB300's tensor cores:
//
//   one CTA per SM walks tiles t = blockIdx.x, + gridDim.x, ... of
//   [128 weight rows x 256 tokens], token tiles fastest (CTAs working at the
//   same time share weight tiles through L2).
//   warp 8     TMA producer: per 64-wide K block the activation tile
//              [256 tokens x 64] and the weight tile [128 rows x 64] (128-byte
//              swizzle) into a 4-stage ring that runs on across tiles, so a tile's
//              first loads overlap the previous tile's last MMAs.
//   warp 9     allocates all 512 tensor-memory columns (two 256-column fp32
//              accumulators) and issues tcgen05.mma (one thread): A = weight tile
//              (M = 128), B = activation tile (N = 256).  Tile i accumulates in
//              buffer i % 2.
//   warps 0-7  epilogue: tcgen05.ld of buffer i % 2 (lane = weight row, column =
//              token), bias, RNE to the dtype, stores of C[token][row] (32 lanes
//              write 32 consecutive columns), then release the buffer: the
//              epilogue of tile i overlaps the MMAs of tile i + 1.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace dense {

constexpr int kBM = 128;                  // weight rows per tile (UMMA M)
constexpr int kBT = 256;                  // tokens per tile (UMMA N)
constexpr int kBK = 64;                   // K per stage: one 128-byte swizzle row of 16-bit values
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = (kEpiWarps + 2) * 32;
constexpr int kActBytes = kBT * kBK * 2;  // 32 KB
constexpr int kWtBytes = kBM * kBK * 2;   // 16 KB
constexpr int kStageBytes = kActBytes + kWtBytes;
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kBytes = kBarOff + 256 + 1024;   // + barriers, + alignment slack
constexpr int kTmemCols = 2 * kBT;             // two accumulators: the whole SM's tensor memory

struct Params {
    uint16_t* C;
    const uint16_t* bias;   // [N] dtype, added before the final rounding; may be null
    int64_t ldc;            // row pitch of C in elements (>= N)
    int M, N;
    int nkb;                // ceil(K / kBK)
    int tiles_m;            // ceil(M / kBT)
    int tiles;              // tiles_m * ceil(N / kBM)
};

__device__ int g_status;

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1) dense_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                                 const __grid_constant__ CUtensorMap tmap_w,
                                                                 const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    auto act_tile = [&](int s) { return smem + s * kStageBytes; };
    auto wt_tile = [&](int s) { return smem + s * kStageBytes + kActBytes; };
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);   // stage landed
    uint64_t* empty = full + kStages;                               // MMAs done with the stage
    uint64_t* acc_full = empty + kStages;                           // [2] tile accumulated
    uint64_t* acc_empty = acc_full + 2;                             // [2] epilogue done reading
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    int* status = &g_status;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kEpiWarps);
        }
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ---------------- TMA producer: one ring across all of this CTA's tiles ----------------
        if (lane == 0) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_w);
            grid_dependency_wait();   // activations may come from the previous kernel
            int g = 0;                // blocks issued so far
            bool ok = true;
            for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
                const int n0 = (t / p.tiles_m) * kBM, m0 = (t % p.tiles_m) * kBT;
                for (int kb = 0; kb < p.nkb; ++kb, ++g) {
                    const int s = g % kStages;
                    if (g >= kStages) ok = mbar_wait(&empty[s], uint32_t(g / kStages - 1) & 1u, status, 50);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&full[s], kActBytes + kWtBytes);
                    tma_load_2d(act_tile(s), &tmap_a, &full[s], kb * kBK, m0);
                    tma_load_2d(wt_tile(s), &tmap_w, &full[s], kb * kBK, n0);
                }
            }
            // copies still in flight must land before the CTA can retire
            for (int b = max(0, g - kStages); b < g; ++b)
                mbar_wait(&full[b % kStages], uint32_t(b / kStages) & 1u, status, 51);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BF16, kBM, kBT);
            int g = 0;
            bool ok = true;
            int i = 0;                // tiles of this CTA so far
            for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++i) {
                const int a = i & 1;
                // the epilogue of tile i - 2 must have read this buffer
                if (i >= 2) ok = mbar_wait(&acc_empty[a], uint32_t(i / 2 - 1) & 1u, status, 52);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + uint32_t(a * kBT);
                for (int kb = 0; kb < p.nkb; ++kb, ++g) {
                    const int s = g % kStages;
                    ok = mbar_wait(&full[s], uint32_t(g / kStages) & 1u, status, 53);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a_desc = smem_desc_sw128(wt_tile(s));
                    const uint64_t b_desc = smem_desc_sw128(act_tile(s));
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)   // 16 K-values = 32 bytes = 2 descriptor units
                        umma_f16_ss(d, a_desc + 2 * k, b_desc + 2 * k, idesc, (kb | k) != 0);
                    umma_commit(&empty[s]);
                }
                if (ok) umma_commit(&acc_full[a]);
            }
        }
    } else {
        // ---------------- epilogue warps ----------------
        // warp w reads TMEM lanes 32*(w%4).. (its rows) and half w/4 of the tile's columns
        const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
        const int rl = 32 * (warp & 3) + lane;
        int i = 0;
        bool dead = false;   // a wait timed out: this and every later tile of the CTA become NaN
        for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++i) {
            const int a = i & 1;
            const int n = (t / p.tiles_m) * kBM + rl;
            const int m0 = (t % p.tiles_m) * kBT;
            const bool row_ok = n < p.N;
            if (!dead) dead = !__all_sync(0xffffffffu, mbar_wait(&acc_full[a], uint32_t(i / 2) & 1u, status, 54));
            if (dead) {   // no tensor-memory reads: the issuer has stopped or is late
                if (row_ok) {
                    for (int c = (warp >> 2) * (kBT / 2); c < ((warp >> 2) + 1) * (kBT / 2); ++c)
                        if (m0 + c < p.M) p.C[size_t(m0 + c) * p.ldc + n] = nan_bits<BF16>();
                }
                continue;
            }
            tc_fence_after();
            const float b = p.bias && row_ok ? to_f32<BF16>(p.bias[n]) : 0.f;
#pragma unroll 1
            for (int c = (warp >> 2) * (kBT / 64); c < ((warp >> 2) + 1) * (kBT / 64); ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + uint32_t(a * kBT) + lane_base + uint32_t(32 * c), r);
                tmem_ld_wait();
                if (row_ok) {
                    const int tok0 = m0 + 32 * c;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = tok0 + j;
                        if (tok < p.M) p.C[size_t(tok) * p.ldc + n] = from_f32<BF16>(__uint_as_float(r[j]) + b);
                    }
                }
            }
            // every load of buffer a by this warp has completed (tmem_ld_wait above)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace dense

// maps: A [M][K] box {64, 256} SW128; dense weight [N][K] box {64, 128} SW128.
cudaError_t launch_dense_gemm(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                              int num_sms, cudaStream_t stream) {
    using namespace dense;
    Params p;
    p.C = static_cast<uint16_t*>(C);
    p.bias = static_cast<const uint16_t*>(bias);
    p.ldc = s.ldc;
    p.M = int(s.M);
    p.N = int(s.N);
    p.nkb = int((s.K + kBK - 1) / kBK);
    p.tiles_m = int((s.M + kBT - 1) / kBT);
    const int64_t tiles = int64_t(p.tiles_m) * ((s.N + kBM - 1) / kBM);
    if (tiles > int64_t(0x7fffffff)) return cudaErrorInvalidValue;   // beyond any C that fits in memory
    p.tiles = int(tiles);
    const int grid = int(tiles < num_sms ? tiles : num_sms);
    auto kern = s.bf16 ? dense_gemm_kernel<true> : dense_gemm_kernel<false>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), kBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kBytes, stream>>>(maps[0], maps[1], p);
    return cudaGetLastError();
}

int take_status_dense() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, dense::g_status, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(dense::g_status, &z, sizeof(int));
    return v;
}

}  // namespace w4a16
