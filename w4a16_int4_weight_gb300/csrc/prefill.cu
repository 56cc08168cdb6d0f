// Large-M ("prefill") W4A16 GEMM on the 5th-generation tensor cores.
//
// The pages' prefill kernel (_triton_w4a16_skinny_fmt_kernel, both revisions)
// loads a packed weight tile per K step, unpacks it, forms (q - z).to(dtype) *
// scale and feeds a dot product with fp32 accumulation.  Here the same tile
// algebra runs as a warp-specialised tcgen05 pipeline:
//
//   warp 8     TMA producer: per 64-wide K block, the activation tile
//              [BT tokens x 64] (128-byte swizzle) and the packed weight tile
//              [128 rows x 8 words] (32-byte swizzle) with its scale and
//              zero-point rows, into a 4-stage ring.
//   warps 0-7  dequantisers: thread i owns half of weight row
//              i % 128 (32 K-values), unpacks with LOP3 magic-number unpacks,
//              forms rne((q - z) * s) exactly as the pages do, and stores the
//              bf16/fp16 tile in the 128-byte-swizzled K-major layout the tensor
//              core reads.  After the K loop the same warps are the epilogue.
//   warp 9     allocates TMEM and issues tcgen05.mma (one thread): the weight
//              tile is the MMA's A operand (M = 128 weight rows), the activation
//              tile the B operand (N = BT tokens), fp32 accumulator in TMEM, so
//              each dequantised weight feeds BT multiply-adds.
//   epilogue   tcgen05.ld of the accumulator (lane = weight row, column =
//              token), RNE to the dtype, stores of C[token][row]: the 32 lanes
//              of a warp write 32 consecutive output columns.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kBM = 128;                  // weight rows per CTA (UMMA M)
constexpr int kBK = 64;                   // K per stage: one 128-byte swizzle row of 16-bit values
constexpr int kStages = 4;
constexpr int kDqWarps = 8;               // dequantiser / epilogue warps
constexpr int kProducerWarp = kDqWarps;
constexpr int kMmaWarp = kDqWarps + 1;
constexpr int kThreads = (kDqWarps + 2) * 32;
constexpr int kWtBytes = kBM * 128;       // 16 KB dequantised weight tile
constexpr int kPkBytes = kBM * 32;        // 4 KB packed tile (8 words per row)
constexpr int kScBytes = 2 * kBM * 2;     // scales of two groups x 128 rows
constexpr int kZpBytes = 2 * 16 * 4;      // zero-point words of two groups x 128 rows

__device__ int g_status;
__device__ __forceinline__ int* p_status() { return &g_status; }

struct Params {
    uint16_t* C;
    const uint16_t* bias;   // [N] dtype, added before the final rounding; may be null
    int64_t ldc;            // row pitch of C in elements (>= N)
    int M, N, K, g_eff, ng;
    int nkb;   // ceil(K / kBK)
    int c_tma; // tmap_c describes C (16-byte aligned base and row pitch): the tile leaves by TMA store
};

template <int BT>
struct Layout {
    static constexpr int kActBytes = BT * 128;
    static constexpr int kStageBytes =
        (kActBytes + kWtBytes + kPkBytes + kScBytes + kZpBytes + 1023) / 1024 * 1024;
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kBytes = kBarOff + 256 + 1024;   // + barriers, + alignment slack
};

template <bool BF16, bool ZP, int BT>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                              const __grid_constant__ CUtensorMap tmap_w,
                                                              const __grid_constant__ CUtensorMap tmap_s,
                                                              const __grid_constant__ CUtensorMap tmap_z,
                                                              const __grid_constant__ CUtensorMap tmap_c,
                                                              const Params p) {
    using L = Layout<BT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    auto act_tile = [&](int s) { return smem + s * L::kStageBytes; };
    auto wt_tile = [&](int s) { return smem + s * L::kStageBytes + L::kActBytes; };
    auto pk_tile = [&](int s) { return smem + s * L::kStageBytes + L::kActBytes + kWtBytes; };
    auto sc_tile = [&](int s) {   // [2 groups][128 rows] of dtype bits
        return reinterpret_cast<uint16_t*>(pk_tile(s) + kPkBytes);
    };
    auto zp_tile = [&](int s) {   // [2 groups][16 words]
        return reinterpret_cast<uint32_t*>(pk_tile(s) + kPkBytes + kScBytes);
    };
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* dq_full = full + kStages;
    uint64_t* empty = dq_full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // token tiles vary fastest, so the CTAs that share a weight tile run together
    // and read it from L2 after the first
    const int tiles_m = (p.M + BT - 1) / BT;
    const int n0 = int(blockIdx.x / tiles_m) * kBM;
    const int m0 = int(blockIdx.x % tiles_m) * BT;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&dq_full[s], kDqWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, BT);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = *tmem_slot;

    if (warp == kProducerWarp) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            tma_prefetch_desc(&tmap_a);
            tma_prefetch_desc(&tmap_w);
            grid_dependency_wait();   // activations may come from the previous kernel
            int issued = 0;
            bool ok = true;
            for (int kb = 0; kb < p.nkb && ok; ++kb) {
                const int s = kb % kStages;
                if (kb >= kStages)
                    ok = mbar_wait(&empty[s], uint32_t(kb / kStages - 1) & 1u, p_status(), 10);
                if (!ok) break;
                mbar_arrive_expect_tx(&full[s], L::kActBytes + kPkBytes + kScBytes + (ZP ? kZpBytes : 0));
                tma_load_2d(act_tile(s), &tmap_a, &full[s], kb * kBK, m0);
                // the K block's first group and the one after it (used when G = 32)
                const int g0 = (kb * kBK) / p.g_eff;
                tma_load_2d(pk_tile(s), &tmap_w, &full[s], kb * (kBK / 8), n0);
                tma_load_2d(sc_tile(s), &tmap_s, &full[s], n0, g0);
                if constexpr (ZP) tma_load_2d(zp_tile(s), &tmap_z, &full[s], n0 / 8, g0);
                ++issued;
            }
            // copies still in flight must land before the CTA can retire
            for (int kb = max(0, issued - kStages); kb < issued; ++kb)
                mbar_wait(&full[kb % kStages], uint32_t(kb / kStages) & 1u, p_status(), 11);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(BF16, kBM, BT);
            bool ok = true;
            for (int kb = 0; kb < p.nkb && ok; ++kb) {
                const int s = kb % kStages;
                const uint32_t par = uint32_t(kb / kStages) & 1u;
                ok = mbar_wait(&full[s], par, p_status(), 12);
                if (ok) ok = mbar_wait(&dq_full[s], par, p_status(), 13);
                if (!ok) break;
                tc_fence_after();
                const uint64_t a_desc = smem_desc_sw128(wt_tile(s));
                const uint64_t b_desc = smem_desc_sw128(act_tile(s));
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)   // 16 K-values = 32 bytes = 2 descriptor units
                    umma_f16_ss(tmem_d, a_desc + 2 * k, b_desc + 2 * k, idesc, (kb | k) != 0);
                umma_commit(&empty[s]);
            }
            if (ok) umma_commit(acc_full);
        }
    } else {
        // ---------------- dequantisers (warps 0-7), then epilogue ----------------
        const int row = tid & (kBM - 1);     // weight row within the tile
        const int half = tid >> 7;           // K-values 32*half .. +31 of each block
        bool ok = true;
        {
            for (int kb = 0; kb < p.nkb; ++kb) {
                const int s = kb % kStages;
                // warp-uniform outcome: the warp leaves the loop together or not at all
                ok = __all_sync(0xffffffffu, mbar_wait(&full[s], uint32_t(kb / kStages) & 1u, p_status(), 14));
                if (!ok) break;
                // 32-byte-swizzled packed row: 16-byte chunk h sits at chunk h ^ ((row / 4) % 2)
                const uint4 wq = *reinterpret_cast<const uint4*>(
                    pk_tile(s) + row * 32 + ((half ^ ((row >> 2) & 1)) << 4));
                const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
                // the 32 K-values lie in one group: every group size is a multiple of
                // 32, or there is one group; the tile's second group row is the
                // K block's second half when G = 32
                const int gl = (p.g_eff == 32 && p.ng > 1) ? half : 0;
                const uint32_t sv = sc_tile(s)[gl * kBM + row];
                const uint32_t s2 = sv | (sv << 16);
                int z = 8;
                if constexpr (ZP) z = (zp_tile(s)[gl * 16 + (row >> 3)] >> (4 * (row & 7))) & 0xF;
                const ZeroConst zc = make_zero_const<BF16>(z);
                uint8_t* dst = wt_tile(s) + row * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t q[4];
                    unpack_word<BF16>(words[j], zc, q);
                    uint4 o;
                    o.x = scale_pair<BF16>(q[0], s2);
                    o.y = scale_pair<BF16>(q[1], s2);
                    o.z = scale_pair<BF16>(q[2], s2);
                    o.w = scale_pair<BF16>(q[3], s2);
                    // 16-byte chunk c of this 128-byte row goes to chunk c ^ (row % 8)
                    const int c = 4 * half + j;
                    *reinterpret_cast<uint4*>(dst + ((c ^ (row & 7)) << 4)) = o;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&dq_full[s]);
            }
        }
        // ---------------- epilogue ----------------
        if (ok) ok = mbar_wait(acc_full, 0u, p_status(), 15);
        ok = __all_sync(0xffffffffu, ok);   // tcgen05.ld below is warp-collective
        tc_fence_after();
        // A failed wait leaves the tile incomplete: its outputs become NaN, written
        // directly (shared memory may still receive copies that were in flight).
        auto nan_tile = [&]() {
            const int n_out = n0 + 32 * (warp & 3) + lane;
            if (n_out >= p.N) return;
            for (int c = (warp >> 2) * (BT / 2); c < ((warp >> 2) + 1) * (BT / 2); ++c) {
                const int tok = m0 + c;
                if (tok < p.M) p.C[size_t(tok) * p.ldc + n_out] = nan_bits<BF16>();
            }
        };
        if (p.c_tma && named_barrier_or(1, kDqWarps * 32, !ok)) {
            nan_tile();
        } else if (p.c_tma) {
            // Stage the output tile [BT tokens][128 rows] in the dtype in the operand
            // ring (the tensor core's reads of it completed before acc_full), then one
            // TMA store that clips rows >= N and tokens >= M.
            static_assert(kStages * L::kStageBytes >= BT * kBM * 2, "output tile fits the operand ring");
            uint16_t* stg = reinterpret_cast<uint16_t*>(smem);
            {
                const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
                const int rl = 32 * (warp & 3) + lane;
                const int n_out = n0 + rl;
                const float b = p.bias && n_out < p.N ? to_f32<BF16>(p.bias[n_out]) : 0.f;
#pragma unroll 1
                for (int c = (warp >> 2) * (BT / 64); c < ((warp >> 2) + 1) * (BT / 64); ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tmem_d + lane_base + uint32_t(32 * c), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        stg[(32 * c + j) * kBM + rl] = from_f32<BF16>(__uint_as_float(r[j]) + b);
                }
                fence_proxy_async_smem();
            }
            named_barrier_sync(1, kDqWarps * 32);
            if (warp == 0 && lane == 0) {
                tma_store_2d(&tmap_c, stg, n0, m0);
                bulk_commit_group();
                bulk_wait_read_all();   // the tile must stay until the store has read it
            }
        } else if (!ok) {
            nan_tile();
        } else {
            // warp w reads TMEM lanes 32*(w%4).. (its rows) and half w/4 of the columns
            const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
            const int n_out = n0 + 32 * (warp & 3) + lane;
            const bool row_ok = n_out < p.N;
            const float b = p.bias && row_ok ? to_f32<BF16>(p.bias[n_out]) : 0.f;
#pragma unroll 1
            for (int c = (warp >> 2) * (BT / 64); c < ((warp >> 2) + 1) * (BT / 64); ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem_d + lane_base + uint32_t(32 * c), r);
                tmem_ld_wait();
                if (row_ok) {
                    const int tok0 = m0 + 32 * c;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int tok = tok0 + j;
                        if (tok < p.M) p.C[size_t(tok) * p.ldc + n_out] = from_f32<BF16>(__uint_as_float(r[j]) + b);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tmem_d, BT);
}

template <bool BF16, bool ZP, int BT>
cudaError_t launch_t(const CUtensorMap* maps, const Params& p, cudaStream_t stream) {
    auto kern = prefill_kernel<BF16, ZP, BT>;
    constexpr int smem = Layout<BT>::kBytes;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    const int64_t ctas = int64_t((p.N + kBM - 1) / kBM) * ((p.M + BT - 1) / BT);
    if (ctas > int64_t(0x7fffffff)) return cudaErrorInvalidValue;   // beyond any C that fits in memory
    const dim3 grid(static_cast<unsigned>(ctas));
    kern<<<grid, kThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], p);
    return cudaGetLastError();
}

template <int BT>
cudaError_t launch_bt(const CUtensorMap* maps, const Params& p, bool bf16, bool zp, cudaStream_t stream) {
    if (bf16) return zp ? launch_t<true, true, BT>(maps, p, stream) : launch_t<true, false, BT>(maps, p, stream);
    return zp ? launch_t<false, true, BT>(maps, p, stream) : launch_t<false, false, BT>(maps, p, stream);
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                           int token_tile, bool c_tma, cudaStream_t stream) {
    Params p;
    p.c_tma = c_tma ? 1 : 0;
    p.C = static_cast<uint16_t*>(C);
    p.bias = static_cast<const uint16_t*>(bias);
    p.ldc = s.ldc;
    p.M = int(s.M);
    p.N = int(s.N);
    p.K = int(s.K);
    p.g_eff = int(s.g_eff);
    p.ng = int(s.ng);
    p.nkb = int((s.K + kBK - 1) / kBK);
    switch (token_tile) {
        case 64: return launch_bt<64>(maps, p, s.bf16, s.zp, stream);
        case 128: return launch_bt<128>(maps, p, s.bf16, s.zp, stream);
        default: return launch_bt<256>(maps, p, s.bf16, s.zp, stream);
    }
}

int take_status_prefill() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof(int));
    return v;
}

}  // namespace w4a16
