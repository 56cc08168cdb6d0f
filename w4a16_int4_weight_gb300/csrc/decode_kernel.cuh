// Small-M ("decode") W4A16 GEMM kernel: C[M,N] = A[M,K] . dequant(W)^T for M <= 64.
//
// The pages' skinny split-K decode kernel (wvSplitK_int4_g, called from
// _rdna_hybrid_w4a16_apply_impl for M <= MAX_SKINNY_BATCH_SIZE) is only named
// there; this is a GB300 design of the same job:
//
//  * Work split.  A CTA owns 128 weight rows and a contiguous run of 256-wide
//    K boxes; the KS CTAs that share a row tile form one thread-block cluster
//    and split K between them.  Their fp32 partials are pushed through
//    distributed shared memory to the CTA that owns each row, by stores that
//    complete on the owner's mbarrier (no cluster-wide release barrier), so
//    no global workspace and no atomics are used.
//  * Data movement.  A producer warp streams, per K box and on one mbarrier,
//    the packed weight box [128 rows x 32 words] (128-byte swizzle), the
//    activation box [M x 256] (zero-filled past K) and the box's scales and zero
//    points from the transposed scale / zero sections: three or four TMA
//    operations per 16 KB of weights.  Consumer warps release a stage through
//    a second mbarrier, so no CTA-wide barrier sits in the K loop.
//  * Math.  Each consumer warp owns 16 rows.  A packed word (8 consecutive
//    K-values of a row) is unpacked with one LOP3 per value pair into 16-bit
//    floats (magic-number trick) and the zero point is subtracted exactly,
//    giving the integers q - z; they are the A operand of mma.m16n8k16 (weights
//    as MMA rows, tokens as MMA columns).  A thread's word covers 8 physical
//    K-values and MMA step s uses values 4s..4s+3 of the words of a thread quad:
//    a permutation of K applied to both operands, which leaves the dot product
//    unchanged.  A quad's words span 32 consecutive K, inside one quantisation
//    group (G >= 32), so the scale is applied once per group:
//        C[n, m] = sum_g s[n,g] * sum_{k in g} A[m,k] (q[n,k] - z[n,g]).
//    (The pages round each dequantised weight to the dtype before the dot; the
//    result differs from this only by those roundings, well inside the output
//    tolerance; w4a16_dequant keeps the exact per-weight rounding.)
#pragma once

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {
namespace decode {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + one producer warp
constexpr int kBN = 16 * kConsumerWarps;               // weight rows per CTA
constexpr int kBoxK = 256;               // K-values per box (32 words = 128 bytes per row)
constexpr int kWBytes = kBN * 128;       // 16 KB packed weight box
constexpr int kMaxStages = 8;
constexpr int kMaxGps = 8;               // groups per box at G = 32
constexpr int kBarBytes = 256;           // mbarriers: full[kMaxStages], empty[kMaxStages], red
// The owner of split-K rows waits for its peers' partials longer than any
// other wait: a peer sends even after one of its own waits gave up, which can
// happen one wait limit after the owner reached this point.
constexpr uint64_t kReductionWaitLimitNs = 3 * kWaitLimitNs;

struct Params {
    uint16_t* C;
    const uint16_t* bias;   // [N] dtype, added before the final rounding; may be null
    int64_t ldc;            // row pitch of C in elements (>= N)
    int* status;      // device status word (first timed-out wait site)
    int M, N, K, g_eff;
    int nboxes;       // ceil(K / kBoxK)
    int ks;           // CTAs per cluster (K split)
    int stages;       // ring depth (<= kMaxStages)
    int gps;          // scale-tile rows per box
    int a_slot;       // bytes of the activation box slot: one token tile: [M rows][256
                      // values] in 1024-byte units; more: four 64-value sub-boxes
                      // [8 NT rows][128 B] (128-byte swizzle), 1024 NT bytes each
    int mpr;          // columns of the reduction buffer: two per stored pair of MMA columns
    int stage_bytes;  // bytes per stage (multiple of 1024): weights, activations, gps scale
                      // rows of 256 bytes and, with zero points, gps rows of 64 bytes
    int red_off;      // byte offset of the cluster reduction buffer
    int prefetch_weights;   // weights may be read before the previous grid completes
};

struct StageView {
    uint8_t* w;        // [128 rows][128 B], 128-byte swizzle
    uint8_t* a;        // activation slot (see Params::a_slot)
    uint16_t* sc;      // [gps][128]
    uint32_t* zp;      // [gps][16]
};

__device__ __forceinline__ StageView stage_view(uint8_t* base, const Params& p, int s) {
    StageView v;
    v.w = base + s * p.stage_bytes;
    v.a = v.w + kWBytes;
    v.sc = reinterpret_cast<uint16_t*>(v.a + p.a_slot);
    v.zp = reinterpret_cast<uint32_t*>(v.sc + p.gps * kBN);
    return v;
}

// Every weight byte is read once per call: the copies carry the evict-first L2
// policy (70B MLP M = 1: 29.4 -> 28.7 us; fp16 26.8 -> 26.0 us).
template <bool ZP>
__device__ __forceinline__ void load_weights(const StageView& v, const CUtensorMap* tq,
                                             const CUtensorMap* ts, const CUtensorMap* tz,
                                             uint64_t* bar, int box, int n0, int g_eff) {
    const int g0 = box * kBoxK / g_eff;
    const uint64_t pol = l2_evict_first_policy();
    tma_load_2d_hint(v.w, tq, bar, box * 32, n0, pol);
    tma_load_2d_hint(v.sc, ts, bar, n0, g0, pol);
    if constexpr (ZP) tma_load_2d_hint(v.zp, tz, bar, n0 / 8, g0, pol);
}

// Two token tiles or more: four [M][64] copies (128-byte swizzle) into the
// sub-boxes; one tile: one [M][256] copy.
template <int NT>
__device__ __forceinline__ void load_acts(const StageView& v, const CUtensorMap* ta,
                                          uint64_t* bar, int box) {
    if constexpr (NT >= 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) tma_load_2d(v.a + i * (1024 * NT), ta, bar, box * kBoxK + 64 * i, 0);
    } else {
        tma_load_2d(v.a, ta, bar, box * kBoxK, 0);
    }
}

// WPG: 32-wide word steps per quantisation group (1, 2, 4 for G = 32, 64, 128);
// 8 when a group spans whole boxes (G >= 256, or one group spanning K).
template <int NT, bool BF16, bool ZP, int WPG>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tmap_q,
                                                          const __grid_constant__ CUtensorMap tmap_a,
                                                          const __grid_constant__ CUtensorMap tmap_s,
                                                          const __grid_constant__ CUtensorMap tmap_z,
                                                          const Params p) {
    constexpr int MP = 8 * NT;                      // padded token count of the MMA column tiles
    // Two token tiles or more: activations in 128-byte-swizzled sub-boxes and MMA
    // columns permuted (below); one tile: plain rows, column g = token g.
    constexpr bool SWZ = NT >= 2;
    // Independent accumulator chains per token tile.  Two chains shorten the MMA
    // dependency chain but cost a merge per group; measured on GB300 (70B MLP and
    // 11008x4096 layers, M = 1 and 8), one chain is faster at 32-wide groups
    // (2.5-5 %) and for fp16 at 64-wide groups (2.6 %), two elsewhere (bf16 at
    // G = 64: 4.6 %).
    constexpr int NSETS = (NT == 1 && (WPG >= 4 || (BF16 && WPG == 2))) ? 2 : 1;
    constexpr int GPB = 8 / WPG;                    // groups per box (1 in the large-group mode)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* red_bar = empty + kMaxStages;   // split K: the partials pushed into this CTA
    float* red = reinterpret_cast<float*>(smem + p.red_off);   // [ks][kBN/ks][mpr]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = int(blockIdx.x) % p.ks;   // rank inside the cluster (cluster = (ks,1,1))
    const int n0 = (int(blockIdx.x) / p.ks) * kBN;
    const int b_lo = (rank * p.nboxes) / p.ks;
    const int b_hi = ((rank + 1) * p.nboxes) / p.ks;
    const int nb = b_hi - b_lo;
    const int k_hi = min(p.K, b_hi * kBoxK);

    if (tid == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(red_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (p.ks > 1) {
        // The peers' partials for this CTA's rows: kBN rows x (pairs of token
        // columns below M) x 8 bytes, whatever the split.  Peers store only after
        // the cluster barrier, i.e. after every CTA has initialised red_bar.
        if (tid == 0) mbar_arrive_expect_tx(red_bar, uint32_t(kBN * 4 * p.mpr));
        cluster_arrive_relaxed();
    }

    bool failed = false;
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    const int g = lane >> 2, t = lane & 3;
    const int r0 = warp * 16 + g, r1 = r0 + 8;   // rows within the tile; r % 8 == g

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            const uint32_t stage_tx = kWBytes + uint32_t(p.M) * (kBoxK * 2u) +
                                      uint32_t(p.gps) * kBN * 2u + (ZP ? uint32_t(p.gps) * 64u : 0u);
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_a);
            const int first = min(p.stages, nb);
            // With static weights the packed weights, scales and zero points are
            // requested before the previous grid in the stream has finished; the
            // activations (and, without that promise, everything) only after it.
            if (p.prefetch_weights) {
                for (int i = 0; i < first; ++i) {
                    mbar_arrive_expect_tx(&full[i], stage_tx);
                    load_weights<ZP>(stage_view(smem, p, i), &tmap_q, &tmap_s, &tmap_z, &full[i],
                                     b_lo + i, n0, p.g_eff);
                }
            }
            grid_dependency_wait();
            for (int i = 0; i < first; ++i) {
                const StageView v = stage_view(smem, p, i);
                if (!p.prefetch_weights) {
                    mbar_arrive_expect_tx(&full[i], stage_tx);
                    load_weights<ZP>(v, &tmap_q, &tmap_s, &tmap_z, &full[i], b_lo + i, n0, p.g_eff);
                }
                load_acts<NT>(v, &tmap_a, &full[i], b_lo + i);
            }
            // the next kernel in the stream may start its own prologue now
            grid_launch_dependents();
            int issued = first;
            int s = first % p.stages;                        // ring slot of box `issued`
            uint32_t wrap = uint32_t(first / p.stages) & 1u;  // its pass over the ring, mod 2
            for (; issued < nb; ++issued) {
                if (!mbar_wait(&empty[s], wrap ^ 1u, p.status, 3)) break;
                const StageView v = stage_view(smem, p, s);
                mbar_arrive_expect_tx(&full[s], stage_tx);
                load_weights<ZP>(v, &tmap_q, &tmap_s, &tmap_z, &full[s], b_lo + issued, n0, p.g_eff);
                load_acts<NT>(v, &tmap_a, &full[s], b_lo + issued);
                if (++s == p.stages) { s = 0; wrap ^= 1u; }
            }
            // copies still in flight must land before the CTA retires
            for (int i = max(0, issued - p.stages); i < issued; ++i)
                mbar_wait(&full[i % p.stages], uint32_t(i / p.stages) & 1u, p.status, 2);
        }
        // The other lanes wait here for lane 0 (blocked, not polling the
        // reduction barrier below for the whole K loop).
        __syncwarp();
    } else {
        // ------------------------------ consumers -----------------------------
        float accg[NSETS][NT][4];
#pragma unroll
        for (int c = 0; c < NSETS; ++c)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) accg[c][j][e] = 0.f;
        float s0 = 0.f, s1 = 0.f;
        ZeroConst zc0 = make_zero_const<BF16>(8), zc1 = zc0;
        int g_end = -1;   // large-group mode: K where the group whose sums accg holds ends

        // acc += scale * group sum.  In the per-group modes the next group's first
        // MMAs overwrite accg (zero accumulator input), so nothing is cleared here.
        auto flush = [&]() {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[e] = accg[0][j][e];
#pragma unroll
                    for (int c = 1; c < NSETS; ++c) v[e] += accg[c][j][e];
                }
                acc[j][0] = fmaf(s0, v[0], acc[j][0]);
                acc[j][1] = fmaf(s0, v[1], acc[j][1]);
                acc[j][2] = fmaf(s1, v[2], acc[j][2]);
                acc[j][3] = fmaf(s1, v[3], acc[j][3]);
            }
        };
        auto load_group = [&](const StageView& v, int gl) {
            s0 = to_f32<BF16>(v.sc[gl * kBN + r0]);
            s1 = to_f32<BF16>(v.sc[gl * kBN + r1]);
            if constexpr (ZP) {
                zc0 = make_zero_const<BF16>((v.zp[gl * 16 + (r0 >> 3)] >> (4 * g)) & 0xF);
                zc1 = make_zero_const<BF16>((v.zp[gl * 16 + (r1 >> 3)] >> (4 * g)) & 0xF);
            }
        };
        // Per-thread shared-memory offsets that do not depend on the stage.  Word
        // ws*4 + t of row r0 sits in 16-byte chunk ws ^ (r0 % 8) = ws ^ g (128-byte
        // swizzle), at byte r0*128 + ((ws ^ g) << 4) + 4t = wofs ^ (ws << 4) with g in
        // bits 4-6 of wofs; row r1 = r0 + 8 is 1024 bytes further.
        const int wofs = r0 * 128 + (g << 4) + (t << 2);
        // MMA column g of tile j is token 8j + g with one token tile.  With more, it is
        // token 8j + col_tok, col_tok = (g >> 1) | ((g & 1) << 2): a quarter-warp
        // (g = 2p, 2p + 1) then reads two tokens 4 apart, whose 16-byte chunks the
        // 128-byte swizzle of the sub-boxes puts on different banks (tokens 1 apart
        // share them; 2-5 % at 16 tokens, nothing at 8 or fewer, where plain rows keep
        // the stage smaller).  Columns whose token is past M reach only outputs that
        // are never stored: their lanes read sub-box rows the copy did not write, or
        // token M - 1 (plain rows, a broadcast).
        const int col_tok = SWZ ? (g >> 1) | ((g & 1) << 2) : g;
        // activation offsets of tile j: plain rows, K-values 8t .. 8t+7 of step ws at
        // ws * 64; sub-boxes, at (ws / 2) * 1024 NT for even / odd steps
        int aoff[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if constexpr (SWZ) {
                // chunk (ws % 2) * 4 + t of row tok sits at chunk ^ (tok % 8), tok % 8 = col_tok
                const int tok = 8 * j + col_tok;
                aoff[j][0] = tok * 128 + ((t ^ col_tok) << 4);
                aoff[j][1] = tok * 128 + (((4 | t) ^ col_tok) << 4);
            } else {
                aoff[j][0] = min(8 * j + col_tok, p.M - 1) * (kBoxK * 2) + (t << 4);
                aoff[j][1] = 0;
            }
        }

        // One K box; CHECK: the box may end early at k_hi (the last box of a K range).
        auto run_box = [&](const StageView& v, int box_k, auto check_tag) {
            constexpr bool CHECK = decltype(check_tag)::value;
#pragma unroll
            for (int gi = 0; gi < GPB; ++gi) {
                if (CHECK && box_k + gi * WPG * 32 >= k_hi) break;
                if constexpr (WPG < 8) load_group(v, gi);
#pragma unroll
                for (int w = 0; w < WPG; ++w) {
                    const int ws = gi * WPG + w;
                    if (CHECK && box_k + ws * 32 >= k_hi) break;
                    const uint8_t* wp = v.w + (wofs ^ (ws << 4));
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(wp);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(wp + 1024);
                    uint32_t q0[4], q1[4];
                    unpack_word<BF16>(w0, zc0, q0);
                    unpack_word<BF16>(w1, zc1, q1);
                    const uint32_t a_s0[4] = {q0[0], q1[0], q0[1], q1[1]};
                    const uint32_t a_s1[4] = {q0[2], q1[2], q0[3], q1[3]};
                    // activation K-values kw + 8t .. +7 of each token row
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const uint8_t* ap = SWZ ? v.a + (ws >> 1) * (1024 * NT) + aoff[j][ws & 1]
                                                : v.a + ws * 64 + aoff[j][0];
                        const uint4 b = *reinterpret_cast<const uint4*>(ap);
                        // step st = 2w + s of the group goes to set st % NSETS; a set's
                        // first step in a group starts from zero (per-group modes)
                        if (WPG < 8 && w == 0) {
                            mma_m16n8k16<BF16, true>(accg[0][j], a_s0, b.x, b.y);
                            if constexpr (NSETS == 2) mma_m16n8k16<BF16, true>(accg[1][j], a_s1, b.z, b.w);
                            else mma_m16n8k16<BF16>(accg[0][j], a_s1, b.z, b.w);
                        } else {
                            mma_m16n8k16<BF16>(accg[0][j], a_s0, b.x, b.y);
                            mma_m16n8k16<BF16>(accg[NSETS - 1][j], a_s1, b.z, b.w);
                        }
                    }
                }
                if constexpr (WPG < 8) flush();
            }
        };

        int stage = 0;
        uint32_t wrap = 0;   // pass over the ring, mod 2: the phase parity to wait for
        for (int i = 0; i < nb; ++i) {
            const bool got = __all_sync(0xffffffffu, mbar_wait_sleep(&full[stage], wrap, p.status, 1));
            if (!got) { failed = true; break; }
            const StageView v = stage_view(smem, p, stage);
            const int box_k = (b_lo + i) * kBoxK;
            if constexpr (WPG == 8) {
                // boxes advance by 256 and a group here spans a multiple of 256 (or all of K)
                if (box_k >= g_end) {
                    if (g_end >= 0) flush();
#pragma unroll
                    for (int c = 0; c < NSETS; ++c)
#pragma unroll
                        for (int j = 0; j < NT; ++j)
#pragma unroll
                            for (int e = 0; e < 4; ++e) accg[c][j][e] = 0.f;
                    g_end = g_end < 0 ? (box_k / p.g_eff + 1) * p.g_eff : g_end + p.g_eff;
                    load_group(v, 0);
                }
            }
            if (box_k + kBoxK <= k_hi) run_box(v, box_k, std::false_type{});
            else run_box(v, box_k, std::true_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == p.stages) { stage = 0; wrap ^= 1u; }
        }
        if constexpr (WPG == 8) {
            if (g_end >= 0) flush();
        }
    }

    // C fragment: (row g, columns 2t, 2t+1) and (row g + 8, same columns); column
    // 2t + e of tile j is token 8j + 2t + e (one token tile) or 8j + t + 4e (more)
    const bool consumer = warp < kConsumerWarps;
    // the bias of an output row, 0 without one
    auto bias_of = [&](int n) { return p.bias && n < p.N ? to_f32<BF16>(p.bias[n]) : 0.f; };
    // A failed wait leaves the result incomplete: those outputs become NaN.
    const uint16_t nan_out = nan_bits<BF16>();
    if (p.ks == 1) {
        if (consumer) {
            const float b0 = bias_of(n0 + r0), b1 = bias_of(n0 + r1);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = SWZ ? 8 * j + t + 4 * (e & 1) : 8 * j + 2 * t + (e & 1);
                    const int n = n0 + (e < 2 ? r0 : r1);
                    if (tok < p.M && n < p.N)
                        p.C[size_t(tok) * p.ldc + n] =
                            failed ? nan_out : from_f32<BF16>(acc[j][e] + (e < 2 ? b0 : b1));
                }
            }
        }
        __syncthreads();   // the producer's final waits end before the CTA retires
        return;
    }
    // Split K: each partial goes to the CTA that owns its row, into slot `rank` of
    // that CTA's reduction buffer, by a store that completes on the owner's
    // red_bar; an owner waits for its own rows only (no cluster-wide release,
    // which costs about a microsecond).
    const int rows_per = kBN / p.ks;
    cluster_wait();   // every CTA's red_bar is initialised
    if (consumer) {
        const uint32_t red_s = smem_u32(red), bar_s = smem_u32(red_bar);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // (row, columns 2t and 2t+1) as one 8-byte store
                // the pair holds tokens 8j + 2t, + 1 (one token tile) or 8j + t, + 4;
                // pairs whose first token is past M are never summed
                if ((SWZ ? 8 * j + t : 8 * j + 2 * t) >= p.M) continue;
                const int col = 8 * j + 2 * t;
                const int row = h == 0 ? r0 : r1;
                const int owner = row / rows_per;
                const uint32_t off = uint32_t(((rank * rows_per + (row - owner * rows_per)) * p.mpr + col) * 4);
                st_async_f32x2(cluster_map(red_s + off, uint32_t(owner)), acc[j][2 * h], acc[j][2 * h + 1],
                               cluster_map(bar_s, uint32_t(owner)));
            }
        }
    }
    // Once red_bar completes no peer writes here any more, so the CTA may retire.
    const bool got = mbar_wait_sleep(red_bar, 0u, p.status, 4, kReductionWaitLimitNs);
    const int any_failed = __syncthreads_or(failed || !got);
    const int items = rows_per * p.M;
    for (int it = tid; it < items; it += kThreads) {
        const int rl = it % rows_per, tok = it / rows_per;
        const int col = SWZ ? 8 * (tok >> 3) + 2 * (tok & 3) + ((tok >> 2) & 1) : tok;   // its reduction column
        float sum = 0.f;
        for (int c = 0; c < p.ks; ++c) sum += red[(c * rows_per + rl) * p.mpr + col];
        const int n = n0 + rank * rows_per + rl;
        if (n < p.N) p.C[size_t(tok) * p.ldc + n] = any_failed ? nan_out : from_f32<BF16>(sum + bias_of(n));
    }
}

template <int NT, bool BF16, bool ZP, int WPG>
cudaError_t launch_one(const CUtensorMap* maps, const Params& p, int grid, size_t smem,
                       cudaStream_t stream) {
    auto kern = decode_kernel<NT, BF16, ZP, WPG>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], p);
}

template <bool BF16, bool ZP, int WPG>
cudaError_t launch_nt(int nt, const CUtensorMap* maps, const Params& p, int grid, size_t smem,
                      cudaStream_t stream) {
    switch (nt) {
        case 1: return launch_one<1, BF16, ZP, WPG>(maps, p, grid, smem, stream);
        case 2: return launch_one<2, BF16, ZP, WPG>(maps, p, grid, smem, stream);
        case 4: return launch_one<4, BF16, ZP, WPG>(maps, p, grid, smem, stream);
        default: return launch_one<8, BF16, ZP, WPG>(maps, p, grid, smem, stream);
    }
}

template <bool BF16>
cudaError_t launch_dtype(bool zp, int wpg, int nt, const CUtensorMap* maps, const Params& p,
                         int grid, size_t smem, cudaStream_t stream) {
#define W4A16_DECODE_WPG(W)                                                                       \
    case W:                                                                                      \
        return zp ? launch_nt<BF16, true, W>(nt, maps, p, grid, smem, stream)                   \
                  : launch_nt<BF16, false, W>(nt, maps, p, grid, smem, stream);
    switch (wpg) {
        W4A16_DECODE_WPG(1)
        W4A16_DECODE_WPG(2)
        W4A16_DECODE_WPG(4)
        W4A16_DECODE_WPG(8)
        default: return cudaErrorInvalidValue;
    }
#undef W4A16_DECODE_WPG
}

// Defined in decode_bf16.cu / decode_fp16.cu (one dtype per translation unit).
cudaError_t launch_bf16(bool zp, int wpg, int nt, const CUtensorMap* maps, const Params& p,
                        int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_fp16(bool zp, int wpg, int nt, const CUtensorMap* maps, const Params& p,
                        int grid, size_t smem, cudaStream_t stream);

}  // namespace decode
}  // namespace w4a16
