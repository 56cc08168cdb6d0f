// Fused-dequant W4A16 GEMM with the dequantised weight tile held in tensor memory.
//
// Same algebra as the pages' fused kernel (_triton_w4a16_skinny_fmt_kernel:
// per K step, (q - z).to(dtype) * scale, then a dot with fp32 accumulation),
// arranged for sm_103a so that no dequantised byte crosses shared memory:
//
//   warp 8     weight producer (TMA): per 256-wide K stage, the packed tile
//              [128 rows x 128 B] (128-byte swizzle) and the scale and zero-point
//              rows of the groups it spans.  Whole 128-byte row segments keep
//              DRAM reads in full lines.
//   warp 10    activation producer (TMA): per 64-wide K block, the tile
//              [BT tokens x 64] (128-byte swizzle).
//   warps 0-7  dequantisers: thread = (TMEM lane = weight row, half of a 64-wide
//              K block); one LOP3 per value pair (magic-number unpack), exact
//              subtraction of the zero point, one rounding multiply by the scale,
//              then tcgen05.st of the 16 bf16/fp16 pairs straight into the
//              block's tensor-memory stage.  They convert block i+1 while the
//              store of block i drains, and run the epilogue after the K loop.
//   warp 9     allocates tensor memory; one thread issues
//              tcgen05.mma.cta_group::1.kind::f16 with A = the weight stage in
//              TMEM (M = 128 weight rows), B = the activation tile in shared
//              memory (N = BT tokens), fp32 accumulator in TMEM.
//   warp 11    (32- and 64-token tiles) a second issuer: the two take alternate
//              MMA units, each into its own accumulator, and the epilogue adds
//              the two.
//
// Three rings: weight stages (shared memory, released by the dequantisers once
// read), activation stages (shared memory, released by the MMA) and
// tensor-memory A stages (32 columns = one 64-wide K block of 128 rows as
// 16-bit pairs, released by the MMA).  Tensor memory: columns [0, BT) hold the
// accumulator ([0, 2 BT) the two issuers' accumulators), every further
// allocated column an A stage.
//
// Small row counts split K over a thread-block cluster (KS CTAs, whole weight
// stages each): partial accumulators are pushed through distributed shared
// memory to the CTA that owns each row block, by stores that complete on that
// CTA's mbarrier, and summed there.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace tgemm {

constexpr int kBM = 128;                  // weight rows per CTA (UMMA M, TMEM lanes)
constexpr int kBK = 64;                   // K per MMA block / activation stage / TMEM stage
constexpr int kWK = 256;                  // K per weight stage (128 bytes of a packed row)
constexpr int kSubPerW = kWK / kBK;       // MMA blocks per weight stage
constexpr int kMaxGps = kWK / 32;         // group rows per weight stage (G >= 32)
constexpr int kDqWarps = 8;
constexpr int kWProducerWarp = kDqWarps;
constexpr int kMmaWarp = kDqWarps + 1;
constexpr int kAProducerWarp = kDqWarps + 2;
constexpr int kMmaWarp2 = kDqWarps + 3;   // second MMA issuer (32- and 64-token tiles)
// MMA-issuing threads per token tile (see Layout::kIssuers) and threads per CTA.
constexpr int issuers_for(int bt) { return bt == 32 || bt == 64 ? 2 : 1; }
constexpr int threads_for(int bt) { return (kDqWarps + 2 + issuers_for(bt)) * 32; }
constexpr int kPkBytes = kBM * kWK / 2;                         // 16 KB packed tile
constexpr int kScBytes = kMaxGps * kBM * 2;                     // scale rows
constexpr int kZpBytes = kMaxGps * (kBM / 8) * 4;               // zero-point rows
constexpr int kWStageBytes = (kPkBytes + kScBytes + kZpBytes + 1023) / 1024 * 1024;

struct Params {
    uint16_t* C;
    const uint16_t* bias;   // [N] dtype, added before the final rounding; may be null
    int64_t ldc;            // row pitch of C in elements (>= N)
    int* status;
    int M, N, K, g_eff, ng;
    int gps;           // group rows per weight stage: min(8, 256 / g_eff), 1 for one group
    int nkb;           // ceil(K / kBK) MMA blocks
    int nws;           // ceil(K / kWK) weight stages
    int ks;            // CTAs per cluster (K split); 1 = whole K per CTA
    int whole_pairs;   // with ks > 1: the first whole_pairs clusters take ks whole tiles
                       // (one per CTA, no split), the others split one tile's K
    int red_in_ring;   // the split's reduction buffer is the activation ring (launched
                       // without the buffer's own shared memory; see the epilogue)
    int prefetch_weights;
    int c_tma;         // tmap_c describes C (16-byte aligned base and row pitch): whole-K tiles
                       // leave through one TMA store of a shared-memory tile
};

// Tensor-memory columns per CTA (a power of two for tcgen05.alloc): the
// accumulator (BT <= 128 columns) and four 32-column A stages; two CTAs per SM
// share the 512 columns.
constexpr int kTmemColsPerCta = 256;
constexpr int kTmemStagesPerCta = 4;

// Ring depths per token tile (16, 32, 64 or 128 tokens): two CTAs per SM (one
// with the split-K buffer at BT >= 64), 64-128 KB of packed weights in flight
// per SM.  From 32 to 64 tokens, three weight stages and three or four activation
// units: with two units the activation copy for unit u + 2 was requested only
// when the dequantisers started unit u, and dequantiser warp 0 waited for it
// (70B MLP, 32 / 64 tokens: 50.4 -> 48.5 / 51.4 -> 49.5 us; 14336 x 4096 at
// 64 tokens: 19.3 -> 18.9 us).
template <int BT>
struct Layout {
    static_assert(BT == 16 || BT == 32 || BT == 64 || BT == 128, "token tile");
    // The MMA issuer takes K blocks in units of kUnit = 2: one wait and two
    // commits per unit, which halves its fixed cost per block (a wait costs the
    // single issuing thread 130-220 cycles, a commit ~44; measured faster than
    // one-block units at every token tile, most at 128 tokens: 66 -> 58 us on
    // the 70B MLP).
    static constexpr int kUnit = 2;
    static constexpr int kWStages = BT <= 16 ? 4 : BT <= 64 ? 3 : 2;
    static constexpr int kAUnits = BT <= 32 ? 4 : BT <= 64 ? 3 : 2;   // activation unit-slots
    static constexpr int kTmemCols = kTmemColsPerCta;
    static constexpr int kTmemStages = kTmemStagesPerCta;             // 32-column block stages
    static constexpr int kTUnits = kTmemStages / kUnit;               // tensor-memory unit-slots
    // MMA-issuing threads, each with its own accumulator, taking alternate units.
    // One thread pays ~540 cycles per unit in waits, commits and fences beside
    // the eight MMAs, and the tensor pipe idled while it did; a second issuer
    // overlaps them.  Measured on GB300: 32 and 64 tokens 2-7 % faster (70B MLP
    // 48.5 -> 46.5 us at 32 tokens); 16-token tiles (zero points, G = 32) 1.5 %
    // slower, so they keep one; 128-token tiles leave no tensor memory for a
    // second accumulator.
    static constexpr int kIssuers = issuers_for(BT);
    static_assert(kIssuers == 1 || kTUnits == 2, "issuer i owns tensor-memory unit-slot i");
    static_assert(kIssuers * BT + 32 * kTmemStages <= kTmemCols, "tensor-memory budget");
    static_assert((kTmemStages & (kTmemStages - 1)) == 0, "power-of-two tensor-memory ring");
    static_assert(kUnit == 2 && kSubPerW % kUnit == 0 && kTUnits >= 2, "two-block units tile a weight stage");
    static constexpr int kActBytes = BT * kBK * 2;                    // one activation tile
    static constexpr int kAUnitBytes = kUnit * kActBytes;
    static constexpr int kActOff = kWStages * kWStageBytes;
    static constexpr int kBarOff = kActOff + kAUnits * kAUnitBytes;
    static constexpr int kRedOff = kBarOff + 512;                 // split-K reduction buffer
    static constexpr int kRedBytes = kBM * BT * 4;                // [ks][kBM/ks][BT] fp32
    static constexpr int kBytesNoRed = kRedOff + 1024;
    static constexpr int kBytesRed = kRedOff + kRedBytes + 1024;
    static constexpr bool kSplitFits = kBytesRed <= 227 * 1024;
    static_assert(2 * (kWStages + kAUnits + kTUnits) * 8 + 16 + 4 <= 512, "barrier area");
};

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem desc]^T, kind::f16.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The register budget allows two CTAs per SM (the launch plan assumes two).
// Three thinner CTAs per SM at BT <= 64 (two weight and two A stages) and
// splitting 128-token tiles over clusters both measured slower; so did one CTA
// per SM with 256-token tiles, at every M up to 4096.
template <bool BF16, bool ZP, int BT>
__global__ void __launch_bounds__(threads_for(BT), 2) tmem_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                                const __grid_constant__ CUtensorMap tmap_w,
                                                                const __grid_constant__ CUtensorMap tmap_s,
                                                                const __grid_constant__ CUtensorMap tmap_z,
                                                                const __grid_constant__ CUtensorMap tmap_c,
                                                                const Params p) {
    using L = Layout<BT>;
    constexpr int kWStages = L::kWStages;
    constexpr int kUnit = L::kUnit;
    constexpr int kAUnits = L::kAUnits;
    constexpr int kTmemStages = L::kTmemStages;
    constexpr int kTUnits = L::kTUnits;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    auto pk_tile = [&](int s) { return smem + s * kWStageBytes; };
    auto sc_tile = [&](int s) { return reinterpret_cast<uint16_t*>(pk_tile(s) + kPkBytes); };
    auto zp_tile = [&](int s) { return reinterpret_cast<uint32_t*>(pk_tile(s) + kPkBytes + kScBytes); };
    auto act_tile = [&](int slot, int g) {
        return smem + L::kActOff + slot * L::kAUnitBytes + g * L::kActBytes;
    };
    uint64_t* w_full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);   // weight stage landed
    uint64_t* w_empty = w_full + kWStages;                               // weight stage read
    uint64_t* a_full = w_empty + kWStages;                               // activation unit landed
    uint64_t* a_empty = a_full + kAUnits;                                // MMA done with it
    uint64_t* dq_full = a_empty + kAUnits;                               // TMEM unit written
    uint64_t* t_empty = dq_full + kTUnits;                               // MMA done with it
    uint64_t* acc_full = t_empty + kTUnits;
    uint64_t* red_bar = acc_full + 1;                                    // split K: partials pushed here
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_bar + 1);
    float* red = reinterpret_cast<float*>(smem + (p.red_in_ring ? L::kActOff : L::kRedOff));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // blockIdx.x = cluster * ks + rank in the cluster: the ks CTAs of a cluster are
    // consecutive.  Tile t = n tile * token tiles + token tile (token tiles vary
    // fastest so that the CTAs sharing a weight tile run together and read it from
    // L2 after the first).  Clusters below whole_pairs take ks whole tiles, one per
    // CTA (ks tiles per cluster); the others split one tile's K ks ways.
    const int tiles_m = (p.M + BT - 1) / BT;
    const int cl = int(blockIdx.x) / p.ks, cr = int(blockIdx.x) % p.ks;
    const bool whole = cl < p.whole_pairs;
    const int ks = whole ? 1 : p.ks;              // this CTA's K split
    const int rank = whole ? 0 : cr;
    const int tile = whole ? cl * p.ks + cr : p.whole_pairs * p.ks + (cl - p.whole_pairs);
    const int n0 = (tile / tiles_m) * kBM;
    const int m0 = (tile % tiles_m) * BT;
    // this CTA's weight stages [ws_lo, ws_hi) and MMA blocks [kb_lo, kb_hi)
    const int ws_lo = (rank * p.nws) / ks;
    const int ws_hi = ((rank + 1) * p.nws) / ks;
    const int nws = ws_hi - ws_lo;
    const int kb_lo = ws_lo * kSubPerW;
    const int kb_hi = min(ws_hi * kSubPerW, p.nkb);
    const int nkb = max(kb_hi - kb_lo, 0);
    const int nunits = (nkb + kUnit - 1) / kUnit;                     // MMA units of kUnit blocks

    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], kDqWarps);
        }
        for (int s = 0; s < kAUnits; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int t = 0; t < kTUnits; ++t) {
            mbar_init(&dq_full[t], kDqWarps);
            mbar_init(&t_empty[t], 1);
        }
        mbar_init(acc_full, L::kIssuers);
        mbar_init(red_bar, 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (ks > 1) {
        // Peers store this CTA's rows of their partial tiles (kBM x BT fp32 in
        // all) only after the cluster barrier, i.e. after red_bar is initialised.
        // (Clusters of whole tiles use neither the barrier nor red_bar.)
        if (tid == 0) mbar_arrive_expect_tx(red_bar, uint32_t(kBM * BT * 4));
        if (!p.red_in_ring) cluster_arrive_relaxed();
    }
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_d = tmem;                    // accumulator of issuer 0: columns [0, BT)
    const uint32_t tmem_d2 = tmem + BT;              // issuer 1 (two issuers): [BT, 2 BT)
    const uint32_t tmem_a = tmem + L::kIssuers * BT; // A stages: 32 columns each
    bool ok = true;

    if (warp == kWProducerWarp) {
        // --------------------------- weight producer ---------------------------
        if (lane == 0) {
            tma_prefetch_desc(&tmap_w);
            tma_prefetch_desc(&tmap_s);
            const uint32_t tx = kPkBytes + uint32_t(p.gps) * (kBM * 2 + (ZP ? (kBM / 8) * 4 : 0));
            // With one token tile every weight byte is read once: evict-first L2
            // policy.  With more, the token tiles of a row tile read it from L2.
            const bool once = tiles_m == 1;
            const uint64_t pol = l2_evict_first_policy();
            auto load_w = [&](int w) {
                const int s = w % kWStages, ws = ws_lo + w;
                const int g0 = (ws * kWK) / p.g_eff;   // first group of the stage
                mbar_arrive_expect_tx(&w_full[s], tx);
                if (once) {
                    tma_load_2d_hint(pk_tile(s), &tmap_w, &w_full[s], ws * (kWK / 8), n0, pol);
                    tma_load_2d_hint(sc_tile(s), &tmap_s, &w_full[s], n0, g0, pol);
                    if constexpr (ZP) tma_load_2d_hint(zp_tile(s), &tmap_z, &w_full[s], n0 / 8, g0, pol);
                } else {
                    tma_load_2d(pk_tile(s), &tmap_w, &w_full[s], ws * (kWK / 8), n0);
                    tma_load_2d(sc_tile(s), &tmap_s, &w_full[s], n0, g0);
                    if constexpr (ZP) tma_load_2d(zp_tile(s), &tmap_z, &w_full[s], n0 / 8, g0);
                }
            };
            const int first = min(kWStages, nws);
            if (!p.prefetch_weights) grid_dependency_wait();
            for (int w = 0; w < first; ++w) load_w(w);
            int issued = first;
            for (; issued < nws; ++issued) {
                const int s = issued % kWStages;
                if (!mbar_wait(&w_empty[s], uint32_t(issued / kWStages - 1) & 1u, p.status, 30)) break;
                load_w(issued);
            }
            // no copy may be in flight when the CTA exits
            for (int w = max(0, issued - kWStages); w < issued; ++w)
                mbar_wait(&w_full[w % kWStages], uint32_t(w / kWStages) & 1u, p.status, 31);
        }
    } else if (warp == kAProducerWarp) {
        // ------------------------- activation producer -------------------------
        if (lane == 0) {
            tma_prefetch_desc(&tmap_a);
            grid_dependency_wait();   // activations may come from the previous kernel
            int issued = 0;
            for (; issued < nunits; ++issued) {
                const int s = issued % kAUnits;
                if (issued >= kAUnits &&
                    !mbar_wait(&a_empty[s], uint32_t(issued / kAUnits - 1) & 1u, p.status, 32))
                    break;
                const int nb = min(kUnit, nkb - kUnit * issued);
                mbar_arrive_expect_tx(&a_full[s], uint32_t(nb * L::kActBytes));
                for (int g = 0; g < nb; ++g)
                    tma_load_2d(act_tile(s, g), &tmap_a, &a_full[s], (kb_lo + kUnit * issued + g) * kBK, m0);
                if (issued == 0) grid_launch_dependents();
            }
            if (nunits == 0) grid_launch_dependents();
            for (int u = max(0, issued - kAUnits); u < issued; ++u)
                mbar_wait(&a_full[u % kAUnits], uint32_t(u / kAUnits) & 1u, p.status, 33);
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ------------------------------ MMA issuers -----------------------------
        // Issuer i takes units i, i + kIssuers, ... into its own accumulator.
        const int first = (L::kIssuers == 2 && warp == kMmaWarp2) ? 1 : 0;
        if (lane == 0 && (warp == kMmaWarp || L::kIssuers == 2)) {
            constexpr uint32_t idesc = idesc_f16(BF16, kBM, BT);
            const uint32_t acc_d = first == 0 ? tmem_d : tmem_d2;
            bool good = true;
            for (int u = first; u < nunits && good; u += L::kIssuers) {
                const int s = u % kAUnits, tu = u % kTUnits;
                // dq_full completes only after dequant warp 0 has seen the unit's
                // activation tiles land (a_full), so one wait covers both.  The
                // issuer sleeps in it rather than polling, which leaves its
                // scheduler's issue slots to the dequantisers there (1-5 % at
                // 24-128 tokens).
                good = mbar_wait_sleep(&dq_full[tu], uint32_t(u / kTUnits) & 1u, p.status, 35);
                if (!good) break;
                tc_fence_after();
                const int nb = min(kUnit, nkb - kUnit * u);
#pragma unroll
                for (int g = 0; g < kUnit; ++g) {
                    if (g < nb) {
                        const int i = kUnit * u + g;                  // block, TMEM stage i % T
                        const uint32_t a_col = uint32_t(32 * (i & (kTmemStages - 1)));
                        const uint64_t b_desc = smem_desc_sw128(act_tile(s, g));
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k)   // 16 K-values: 8 TMEM columns, 32 smem bytes
                            umma_f16_ts(acc_d, tmem_a + a_col + uint32_t(8 * k), b_desc + 2 * k, idesc,
                                        (u != first || g != 0 || k != 0) ? 1u : 0u);
                    }
                }
                umma_commit(&a_empty[s]);    // frees the activation unit
                umma_commit(&t_empty[tu]);   // frees the tensor-memory unit
            }
            // (an issuer without units arrives at once: nothing of its own is in flight)
            if (good && nkb > 0) umma_commit(acc_full);
        }
    } else {
        // ------------------------------ dequantisers ------------------------------
        // Thread = (weight row = TMEM lane, half of each 64-wide block).  One
        // weight stage (4 blocks) per iteration, block index j a compile-time
        // constant, so per-thread offsets are precomputed and no register array
        // is copied.  The 32 K-values of a (row, half) lie in one group: every
        // group size is a multiple of 32, or there is one group.
        const int row = tid & (kBM - 1);
        const int half = tid >> 7;
        const uint32_t t_addr = tmem_a + (uint32_t(32 * (warp & 3)) << 16) + uint32_t(16 * half);
        const int gshift = p.ng > 1 ? __ffs(p.g_eff) - 1 : 31;   // 31: one group
        int pk_off[kSubPerW], sc_off[kSubPerW], zp_off[kSubPerW];
#pragma unroll
        for (int j = 0; j < kSubPerW; ++j) {
            pk_off[j] = row * 128 + (((2 * j + half) ^ (row & 7)) << 4);
            const int gl = (j * kBK + 32 * half) >> gshift;
            sc_off[j] = gl * kBM + row;
            zp_off[j] = gl * (kBM / 8) + (row >> 3);
        }
        const int zp_shift = 4 * (row & 7);
        uint32_t ca[16], cb[16];
        auto convert = [&](const uint8_t* stg, int j, uint32_t (&cols)[16]) {
            const uint4 wq = *reinterpret_cast<const uint4*>(stg + pk_off[j]);
            const uint32_t sv = reinterpret_cast<const uint16_t*>(stg + kPkBytes)[sc_off[j]];
            const uint32_t s2 = __byte_perm(sv, 0u, 0x1010);
            int z = 8;
            if constexpr (ZP)
                z = int(reinterpret_cast<const uint32_t*>(stg + kPkBytes + kScBytes)[zp_off[j]] >> zp_shift);
            const ZeroConst zc = make_zero_const<BF16>(z);
            const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint32_t q[4];
                unpack_word<BF16>(words[jj], zc, q);
#pragma unroll
                for (int e = 0; e < 4; ++e) cols[4 * jj + e] = scale_pair<BF16>(q[e], s2);
            }
        };
        // Hand-off of MMA unit u (blocks kUnit*u ..): before its first store, wait
        // until the MMAs that last read its tensor-memory slot are complete; after
        // its last store, wait for the stores, and (warp 0) for the unit's
        // activation tiles, then signal the issuer.
        auto unit_free = [&](int u) -> bool {
            const int tu = u % kTUnits;
            return u < kTUnits ||
                   __all_sync(0xffffffffu, mbar_wait(&t_empty[tu], uint32_t(u / kTUnits + 1) & 1u, p.status, 37));
        };
        auto unit_done = [&](int u) -> bool {
            tmem_st_wait();
            tc_fence_before();
            if (warp == 0 &&
                !__all_sync(0xffffffffu, mbar_wait(&a_full[u % kAUnits], uint32_t(u / kAUnits) & 1u, p.status, 34)))
                return false;
            __syncwarp();
            if (lane == 0) mbar_arrive(&dq_full[u % kTUnits]);
            return true;
        };
        // block li (local index) into its 32-column tensor-memory stage
        auto put = [&](int li, const uint32_t (&cols)[16]) {
            tc_fence_after();
            tmem_st_32x32b_x16(t_addr + uint32_t(32 * (li & (kTmemStages - 1))), cols);
        };
        for (int w = 0; w < nws && ok; ++w) {
            const int s = w % kWStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&w_full[s], uint32_t(w / kWStages) & 1u, p.status, 36))) {
                ok = false;
                break;
            }
            const uint8_t* stg = pk_tile(s);
            const int b0 = w * kSubPerW;                        // first block of the stage
            const int nj = min(kSubPerW, nkb - b0);
            if (nj == kSubPerW) {
                // units (0,1) and (2,3) of the stage
                const int u0 = b0 / 2;
                convert(stg, 0, ca);
                convert(stg, 1, cb);
                ok = unit_free(u0);
                if (ok) {
                    put(b0, ca);
                    put(b0 + 1, cb);
                    ok = unit_done(u0);
                }
                convert(stg, 2, ca);
                convert(stg, 3, cb);
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[s]);   // the stage has been read
                ok = ok && unit_free(u0 + 1);
                if (ok) {
                    put(b0 + 2, ca);
                    put(b0 + 3, cb);
                    ok = unit_done(u0 + 1);
                }
            } else {
                // the last stage of a K range that ends inside it
#pragma unroll
                for (int j = 0; j < kSubPerW; ++j) {
                    if (j < nj) {
                        const int li = b0 + j, u = li / kUnit;
                        convert(stg, j, ca);
                        if (j == nj - 1) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&w_empty[s]);
                        }
                        if (li % kUnit == 0) ok = ok && unit_free(u);
                        if (ok) {
                            put(li, ca);
                            tmem_st_wait();   // ca is reused by the next block
                        }
                        if (li % kUnit == kUnit - 1 || j == nj - 1) ok = ok && unit_done(u);
                    }
                }
            }
        }
        // ------------------------------ epilogue ------------------------------
        if (ok && nkb > 0) ok = mbar_wait(acc_full, 0u, p.status, 25);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
    }

    // Epilogue: warp w reads TMEM lanes 32*(w%4).. and column half w/4 of the tile
    // (tiles narrower than 32 tokens use warps 0-3 only).
    constexpr int kHalves = BT >= 32 ? 2 : 1;
    constexpr int kColsPerWarp = BT / kHalves;
    const bool epi = warp < 4 * kHalves;
    // The tile's fp32 sums for TMEM lanes of this warp, columns col .. col + 15:
    // the two issuers' accumulators added when the second one holds units.
    const bool two_acc = L::kIssuers == 2 && nunits > 1;
    auto load_acc = [&](int col, uint32_t (&r)[16]) {
        const uint32_t off = (uint32_t(32 * (warp & 3)) << 16) + uint32_t(col);
        tmem_ld_32x32b_x16(tmem_d + off, r);
        if (two_acc) {
            uint32_t r2[16];
            tmem_ld_32x32b_x16(tmem_d2 + off, r2);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(r2[j]));
        } else {
            tmem_ld_wait();
        }
    };
    const int row = 32 * (warp & 3) + lane;
    const int c0 = (warp >> 2) * kColsPerWarp;
    // the bias of an output row, 0 without one
    auto bias_of = [&](int n) { return p.bias && n < p.N ? to_f32<BF16>(p.bias[n]) : 0.f; };
    // A failed wait leaves the tile incomplete: its outputs become NaN, written
    // directly (shared memory may still receive copies that were in flight).
    auto nan_tile = [&]() {
        const int n = n0 + row;
        if (n >= p.N) return;
        for (int c = 0; c < kColsPerWarp; ++c) {
            const int tok = m0 + c0 + c;
            if (tok < p.M) p.C[size_t(tok) * p.ldc + n] = nan_bits<BF16>();
        }
    };
    if (ks == 1 && p.c_tma) {
        // Stage the output tile [BT tokens][128 rows] in the dtype in the activation
        // ring (the tensor core's last reads of it completed before acc_full), then
        // one TMA store; it clips rows >= N and tokens >= M.  Two-byte stores of
        // 32 lanes straight to global memory took ~2 us of a 27 us tile.
        static_assert(L::kAUnits * L::kAUnitBytes >= BT * kBM * 2, "output tile fits the activation ring");
        uint16_t* stg = reinterpret_cast<uint16_t*>(smem + L::kActOff);
        if (epi && named_barrier_or(1, 4 * kHalves * 32, !(ok && nkb > 0))) {
            nan_tile();
        } else if (epi) {
            {
                const float b = bias_of(n0 + row);
#pragma unroll 1
                for (int c = 0; c < kColsPerWarp; c += 16) {
                    uint32_t r[16];
                    load_acc(c0 + c, r);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        stg[(c0 + c + j) * kBM + row] = from_f32<BF16>(__uint_as_float(r[j]) + b);
                }
                fence_proxy_async_smem();
            }
            named_barrier_sync(1, 4 * kHalves * 32);
            if (warp == 0 && lane == 0) {
                tma_store_2d(&tmap_c, stg, n0, m0);
                bulk_commit_group();
                bulk_wait_read_all();   // the tile must stay until the store has read it
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
        return;
    }
    if (ks == 1) {
        if (epi && !(ok && nkb > 0)) {
            nan_tile();
        } else if (epi) {
            const int n = n0 + row;
            const float b = bias_of(n);
#pragma unroll 1
            for (int c = 0; c < kColsPerWarp; c += 16) {
                uint32_t r[16];
                load_acc(c0 + c, r);
                if (n < p.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = m0 + c0 + c + j;
                        if (tok < p.M) p.C[size_t(tok) * p.ldc + n] = from_f32<BF16>(__uint_as_float(r[j]) + b);
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
        return;
    }
    // Split K: push the partial tile to the owner of each row block (rows_per rows)
    // with stores that complete on the owner's red_bar; an owner waits for its own
    // rows only (a cluster-wide release barrier costs about a microsecond).  Every
    // row's columns are always sent, zeros after a failed wait, so that red_bar
    // completes.
    const int rows_per = kBM / ks;
    if (p.red_in_ring) {
        // The buffer is the activation ring: every thread here is past the
        // dequantisers' wait for the accumulator (the MMAs, the ring's last
        // readers, have completed; the producers' copies all landed) before the
        // CTA arrives, and peers store into it only after all have arrived.
        static_assert(L::kRedBytes <= L::kAUnits * L::kAUnitBytes, "the reduction buffer fits the activation ring");
        __syncthreads();
        cluster_arrive();
    }
    cluster_wait();   // every CTA's red_bar is initialised
    if (epi) {
        const int owner = row / rows_per;
        const uint32_t dst = cluster_map(
            smem_u32(red) + uint32_t((rank * rows_per + (row - owner * rows_per)) * BT * 4), uint32_t(owner));
        const uint32_t bar = cluster_map(smem_u32(red_bar), uint32_t(owner));
#pragma unroll 1
        for (int c = 0; c < kColsPerWarp; c += 16) {
            uint32_t r[16] = {};   // a CTA without K blocks contributes zeros
            if (ok && nkb > 0) load_acc(c0 + c, r);
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                st_async_f32x4(dst + uint32_t((c0 + c + j) * 4), __uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                               __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]), bar);
        }
    }
    // Once red_bar completes no peer writes here any more, so the CTA may retire.
    // (the peers' sends can follow one of their own timed-out waits, so this wait
    // is longer than any other)
    const bool got = mbar_wait_limit(red_bar, 0u, p.status, 38, 3 * kWaitLimitNs);
    const int any_failed = __syncthreads_or(!ok || !got);
    // this CTA owns rows [rank*rows_per, (rank+1)*rows_per) of the tile
    const int items = rows_per * BT;
    for (int it = tid; it < items; it += threads_for(BT)) {
        const int rl = it % rows_per, col = it / rows_per;
        float sum = 0.f;
        for (int c = 0; c < ks; ++c) sum += red[(size_t(c) * rows_per + rl) * BT + col];
        const int n = n0 + rank * rows_per + rl, tok = m0 + col;
        if (n < p.N && tok < p.M)
            p.C[size_t(tok) * p.ldc + n] = any_failed ? nan_bits<BF16>() : from_f32<BF16>(sum + bias_of(n));
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
}

}  // namespace tgemm
}  // namespace w4a16
