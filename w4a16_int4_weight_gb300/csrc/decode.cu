// Small-M ("decode") W4A16 GEMM: C[M,N] = A[M,K] . dequant(W)^T for M <= 64.
//
// The pages' skinny split-K decode kernel (wvSplitK_int4_g, called from
// _rdna_hybrid_w4a16_apply_impl for M <= MAX_SKINNY_BATCH_SIZE) is only named
// there; this is a GB300 design of the same job:
//
//  * Work split.  A CTA owns 128 weight rows and a contiguous range of 256-wide
//    K boxes; the KS CTAs that share a row tile form one thread-block cluster
//    and split K between them.  Their fp32 partial tiles are summed through
//    distributed shared memory, so no global workspace and no atomics are used.
//  * Weight stream.  One thread issues TMA box loads ([128 rows x 32 words],
//    128-byte swizzle) into a ring of up to four 16 KB stages; for the
//    decode shapes every box of a CTA is in flight at once.
//  * Math.  Each warp owns 16 rows.  The packed word of a row (8 consecutive
//    K-values) is unpacked with one LOP3 per value pair into 16-bit floats and
//    the zero point is subtracted exactly, giving the integers q - z.  They are
//    the A operand of mma.m16n8k16 (weights as MMA rows, tokens as MMA columns,
//    "swap AB"), so the tensor pipe absorbs the multiply-adds.  A thread's word
//    covers 8 physical K-values; MMA step s of a word uses values 4s..4s+3 of
//    the four words of a thread quad, i.e. a permutation of K applied to both
//    operands, which leaves the dot product unchanged.  A quad's words span 32
//    consecutive K, inside one quantisation group (G >= 32), so the scale is
//    applied once per group to the fp32 group sum:
//        C[n, m] = sum_g s[n,g] * sum_{k in g} A[m,k] (q[n,k] - z[n,g]).
//    (The pages round each dequantised weight to the dtype before the dot; the
//    GEMM result differs from that only by those roundings, well inside the
//    output tolerance, and w4a16_dequant keeps the exact per-weight rounding.)
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBN = 128;                 // weight rows per CTA
constexpr int kBoxK = 256;               // K-values per TMA box (32 words = 128 bytes)
constexpr int kBoxBytes = kBN * 128;     // 16 KB
constexpr int kMaxStages = 4;

__device__ int g_status;

struct Params {
    const uint16_t* A;
    const uint16_t* scales;
    const int32_t* zeros;
    uint16_t* C;
    int M, N, K, g_eff, ng;
    int nboxes;      // ceil(K / kBoxK)
    int ks;          // CTAs per cluster (K split)
    int stages;      // ring depth (<= kMaxStages)
    int act_pitch;   // bytes per staged activation row
    int act_rows;    // rows of staged activations (M)
};

__device__ __forceinline__ uint32_t lds_u32(const uint8_t* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ uint4 lds_v4(const uint8_t* p) {
    return *reinterpret_cast<const uint4*>(p);
}

template <int NT, bool BF16, bool ZP>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tmap_q,
                                                          const Params p) {
    constexpr int MP = 8 * NT;   // padded token count of the MMA column tiles
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* wbuf = smem;                                           // stages x 16 KB
    uint8_t* act = wbuf + p.stages * kBoxBytes;                     // act_rows x act_pitch
    float* part = reinterpret_cast<float*>(act + p.act_rows * p.act_pitch);  // kBN x MP
    uint64_t* bars = reinterpret_cast<uint64_t*>(part + kBN * MP);  // kMaxStages

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = int(blockIdx.x) % p.ks;   // rank inside the cluster (cluster = (ks,1,1))
    const int n0 = (int(blockIdx.x) / p.ks) * kBN;
    const int b_lo = (rank * p.nboxes) / p.ks;
    const int b_hi = ((rank + 1) * p.nboxes) / p.ks;
    const int nb = b_hi - b_lo;
    const int k_lo = b_lo * kBoxK;
    const int k_hi = min(p.K, b_hi * kBoxK);

    if (tid == 0) {
        for (int s = 0; s < kMaxStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    int issued = 0;
    if (tid == 0) {
        tma_prefetch_desc(&tmap_q);
        for (; issued < min(p.stages, nb); ++issued) {
            mbar_arrive_expect_tx(&bars[issued], kBoxBytes);
            tma_load_2d(wbuf + issued * kBoxBytes, &tmap_q, &bars[issued], (b_lo + issued) * 32, n0);
        }
    }

    // Activations may be produced by the previous kernel in the stream: wait
    // for it (a no-op without programmatic dependent launch), then stage this
    // CTA's K range of A, zero past K up to the next multiple of 32.
    grid_dependency_wait();
    {
        const int span = ((k_hi - k_lo) + 31) & ~31;
        const int vec_per_row = span / 8;
        const int total = p.M * vec_per_row;
        for (int v = tid; v < total; v += kThreads) {
            const int tok = v / vec_per_row, c = v - tok * vec_per_row;
            const int k = k_lo + 8 * c;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (k < p.K)
                val = __ldg(reinterpret_cast<const uint4*>(p.A + size_t(tok) * p.K + k));
            *reinterpret_cast<uint4*>(act + tok * p.act_pitch + 16 * c) = val;
        }
    }
    __syncthreads();

    const int g = lane >> 2, t = lane & 3;
    const int r0 = warp * 16 + g, r1 = r0 + 8;
    const int nr0 = n0 + r0, nr1 = n0 + r1;
    const bool v0 = nr0 < p.N, v1 = nr1 < p.N;

    float acc[NT][4], accg[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[j][e] = accg[j][e] = 0.f;

    int cur_g = -1;
    float s0 = 0.f, s1 = 0.f;
    ZeroConst zc0 = make_zero_const<BF16>(8), zc1 = zc0;
    bool failed = false;

    for (int i = 0; i < nb; ++i) {
        const int stage = i % p.stages;
        const bool got = mbar_wait(&bars[stage], uint32_t(i / p.stages) & 1u, &g_status, 1);
        if (!__syncthreads_and(got)) { failed = true; break; }
        const uint8_t* wt = wbuf + stage * kBoxBytes;
        const int box_k = (b_lo + i) * kBoxK;
#pragma unroll
        for (int ws = 0; ws < 8; ++ws) {
            const int kw = box_k + ws * 32;
            if (kw >= k_hi) break;
            const int grp = kw / p.g_eff;
            if (grp != cur_g) {
                if (cur_g >= 0) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        acc[j][0] = fmaf(s0, accg[j][0], acc[j][0]);
                        acc[j][1] = fmaf(s0, accg[j][1], acc[j][1]);
                        acc[j][2] = fmaf(s1, accg[j][2], acc[j][2]);
                        acc[j][3] = fmaf(s1, accg[j][3], acc[j][3]);
                        accg[j][0] = accg[j][1] = accg[j][2] = accg[j][3] = 0.f;
                    }
                }
                cur_g = grp;
                s0 = v0 ? to_f32<BF16>(__ldg(p.scales + size_t(nr0) * p.ng + grp)) : 0.f;
                s1 = v1 ? to_f32<BF16>(__ldg(p.scales + size_t(nr1) * p.ng + grp)) : 0.f;
                if constexpr (ZP) {
                    const int z0 = v0 ? (__ldg(p.zeros + size_t(nr0 >> 3) * p.ng + grp) >> (4 * (nr0 & 7))) & 0xF : 8;
                    const int z1 = v1 ? (__ldg(p.zeros + size_t(nr1 >> 3) * p.ng + grp) >> (4 * (nr1 & 7))) & 0xF : 8;
                    zc0 = make_zero_const<BF16>(z0);
                    zc1 = make_zero_const<BF16>(z1);
                }
            }
            // word wi of the 32-word box row; 16-byte chunk wi/4 sits at chunk (wi/4) ^ (row % 8)
            const int wi = ws * 4 + t;
            const int chunk = ((wi >> 2) ^ g) << 4, within = (wi & 3) << 2;
            const uint32_t w0 = lds_u32(wt + r0 * 128 + chunk + within);
            const uint32_t w1 = lds_u32(wt + r1 * 128 + chunk + within);
            uint32_t q0[4], q1[4];
            unpack_word<BF16>(w0, zc0, q0);
            unpack_word<BF16>(w1, zc1, q1);
            const uint32_t a_s0[4] = {q0[0], q1[0], q0[1], q1[1]};
            const uint32_t a_s1[4] = {q0[2], q1[2], q0[3], q1[3]};
            const int koff = (kw - k_lo + 8 * t) * 2;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int tok = 8 * j + g;
                uint4 b = make_uint4(0u, 0u, 0u, 0u);
                if (tok < p.M) b = lds_v4(act + tok * p.act_pitch + koff);
                mma_m16n8k16<BF16>(accg[j], a_s0, b.x, b.y);
                mma_m16n8k16<BF16>(accg[j], a_s1, b.z, b.w);
            }
        }
        __syncthreads();   // every warp is done with this stage
        if (tid == 0 && issued < nb) {
            mbar_arrive_expect_tx(&bars[stage], kBoxBytes);
            tma_load_2d(wbuf + stage * kBoxBytes, &tmap_q, &bars[stage], (b_lo + issued) * 32, n0);
            ++issued;
        }
    }
    if (failed && tid == 0) {
        // let copies still in flight land before the CTA's shared memory goes away
        for (int i = max(0, issued - p.stages); i < issued; ++i)
            mbar_wait(&bars[i % p.stages], uint32_t(i / p.stages) & 1u, &g_status, 2);
    }
    if (cur_g >= 0) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            acc[j][0] = fmaf(s0, accg[j][0], acc[j][0]);
            acc[j][1] = fmaf(s0, accg[j][1], acc[j][1]);
            acc[j][2] = fmaf(s1, accg[j][2], acc[j][2]);
            acc[j][3] = fmaf(s1, accg[j][3], acc[j][3]);
        }
    }
    // C fragment: (row g, tokens 2t, 2t+1) and (row g + 8, same tokens)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int tok = 8 * j + 2 * t;
        part[r0 * MP + tok] = acc[j][0];
        part[r0 * MP + tok + 1] = acc[j][1];
        part[r1 * MP + tok] = acc[j][2];
        part[r1 * MP + tok + 1] = acc[j][3];
    }

    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    // CTA `rank` finishes rows [rank * kBN/ks, (rank+1) * kBN/ks) of the tile,
    // summing the partials of all CTAs of the cluster.
    const int rows_per = kBN / p.ks;
    const int row_base = rank * rows_per;
    const int items = rows_per * p.M;
    for (int it = tid; it < items; it += kThreads) {
        const int row = row_base + it % rows_per, tok = it / rows_per;
        float sum = 0.f;
        for (int c = 0; c < p.ks; ++c) {
            const float* peer = cluster.map_shared_rank(part, c);
            sum += peer[row * MP + tok];
        }
        const int n = n0 + row;
        if (n < p.N && !failed) p.C[size_t(tok) * p.N + n] = from_f32<BF16>(sum);
    }
    cluster.sync();   // peers may still be reading this CTA's partials
}

template <int NT, bool BF16, bool ZP>
cudaError_t launch_t(const CUtensorMap& tmap, const Params& p, int grid, size_t smem,
                     cudaStream_t stream) {
    auto kern = decode_kernel<NT, BF16, ZP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmap, p);
}

template <bool BF16, bool ZP>
cudaError_t launch_nt(int nt, const CUtensorMap& tmap, const Params& p, int grid, size_t smem,
                      cudaStream_t stream) {
    switch (nt) {
        case 1: return launch_t<1, BF16, ZP>(tmap, p, grid, smem, stream);
        case 2: return launch_t<2, BF16, ZP>(tmap, p, grid, smem, stream);
        case 4: return launch_t<4, BF16, ZP>(tmap, p, grid, smem, stream);
        default: return launch_t<8, BF16, ZP>(tmap, p, grid, smem, stream);
    }
}

}  // namespace

// Host-side plan: cluster size and ring depth for a shape; false if the
// activation slice cannot fit in shared memory.
bool plan_decode(int64_t M, int64_t N, int64_t K, int num_sms, int* ks_out, int* stages_out,
                 size_t* smem_out, int* nt_out) {
    if (M < 1 || M > kDecodeMaxM) return false;
    const int nt = M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8;
    const int64_t row_tiles = (N + kBN - 1) / kBN;
    const int64_t nboxes = (K + kBoxK - 1) / kBoxK;
    const int64_t target = 2LL * num_sms;
    int ks = 1;
    while (ks < 8 && row_tiles * ks < target && 2 * ks <= nboxes) ks *= 2;
    for (;;) {
        const int64_t boxes_per = (nboxes + ks - 1) / ks;
        const int64_t pitch = 512 * boxes_per + 64;
        for (int stages = int(boxes_per < kMaxStages ? boxes_per : kMaxStages); stages >= 1; --stages) {
            const size_t smem = size_t(stages) * kBoxBytes + size_t(M) * pitch +
                                size_t(kBN) * 8 * nt * 4 + kMaxStages * 8 + 1024;
            if (smem <= 227 * 1024 && (stages >= 2 || boxes_per == 1)) {
                *ks_out = ks;
                *stages_out = stages;
                *smem_out = smem;
                *nt_out = nt;
                return true;
            }
        }
        if (ks < 8 && 2 * ks <= nboxes) ks *= 2;
        else return false;
    }
}

cudaError_t launch_decode(const CUtensorMap& tmap_q, const void* A, const void* scales,
                          const int32_t* zeros, void* C, const LayerShape& s, int num_sms,
                          cudaStream_t stream) {
    int ks, stages, nt;
    size_t smem;
    if (!plan_decode(s.M, s.N, s.K, num_sms, &ks, &stages, &smem, &nt)) return cudaErrorInvalidValue;
    Params p;
    p.A = static_cast<const uint16_t*>(A);
    p.scales = static_cast<const uint16_t*>(scales);
    p.zeros = zeros;
    p.C = static_cast<uint16_t*>(C);
    p.M = int(s.M);
    p.N = int(s.N);
    p.K = int(s.K);
    p.g_eff = int(s.g_eff);
    p.ng = int(s.ng);
    p.nboxes = int((s.K + kBoxK - 1) / kBoxK);
    p.ks = ks;
    p.stages = stages;
    p.act_pitch = int(512 * ((p.nboxes + ks - 1) / ks) + 64);
    p.act_rows = int(s.M);
    const int grid = int((s.N + kBN - 1) / kBN) * ks;
    if (s.bf16) {
        return s.zp ? launch_nt<true, true>(nt, tmap_q, p, grid, smem, stream)
                    : launch_nt<true, false>(nt, tmap_q, p, grid, smem, stream);
    }
    return s.zp ? launch_nt<false, true>(nt, tmap_q, p, grid, smem, stream)
                : launch_nt<false, false>(nt, tmap_q, p, grid, smem, stream);
}

int take_status_decode() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof(int));
    return v;
}

}  // namespace w4a16
