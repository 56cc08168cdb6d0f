// Host side of the tensor-memory fused GEMM (kernel: tmem_gemm.cuh): token tile
// and K-split choice, instantiation and launch.
#include <mutex>

#include "tmem_gemm.cuh"

namespace w4a16 {
namespace {

__device__ int g_status;

int* status_ptr() {
    static std::mutex mu;
    static int* cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int*>(p);
    }
    return cache[dev];
}

constexpr int kSmemPerSm = 228 * 1024;     // shared memory per SM (sm_100 family)
constexpr int kSmemPerCtaReserved = 1024;  // the runtime's per-CTA reservation

int tmem_safe_smem(int bytes, int tmem_cols) {
    const int allowed = 512 / tmem_cols;
    const int floor_bytes = kSmemPerSm / (allowed + 1) - kSmemPerCtaReserved + 1;
    return bytes > floor_bytes ? bytes : floor_bytes;
}

template <bool BF16, bool ZP, int BT>
cudaError_t launch_t(const CUtensorMap* maps, const tgemm::Params& p, int grid_x, int grid_y,
                     cudaStream_t stream) {
    using L = tgemm::Layout<BT>;
    auto kern = tgemm::tmem_gemm_kernel<BF16, ZP, BT>;
    // tcgen05.alloc blocks while the SM's 512 columns are taken; CTAs of one
    // cluster wait for each other, so more resident CTAs than 512 / kTmemCols
    // could deadlock.  Ask for enough shared memory that no more fit.
    const int smem = tmem_safe_smem(p.ks > 1 && !p.red_in_ring ? L::kBytesRed : L::kBytesNoRed, L::kTmemCols);
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_x, grid_y);
    cfg.blockDim = dim3(tgemm::threads_for(BT));
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
    return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], p);
}

template <int BT>
cudaError_t launch_bt(const CUtensorMap* maps, const tgemm::Params& p, bool bf16, bool zp,
                      int gx, int gy, cudaStream_t stream) {
    if (bf16) return zp ? launch_t<true, true, BT>(maps, p, gx, gy, stream)
                        : launch_t<true, false, BT>(maps, p, gx, gy, stream);
    return zp ? launch_t<false, true, BT>(maps, p, gx, gy, stream)
              : launch_t<false, false, BT>(maps, p, gx, gy, stream);
}

}  // namespace

// Token tile: the smallest of 16/32/64 that covers M, else 128.  Above 128 tokens
// 128-wide tiles (two CTAs, 16 dequantising warps and two MMA pipelines per SM)
// measured faster than 256-wide ones (one CTA per SM, half the dequantisation per
// FLOP) at every M up to 4096 on GB300 (70B MLP M=256: 114 -> 94 us; M=4096:
// 1466 -> 1345 us).
int tmem_gemm_token_tile(int64_t M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    return 128;
}

namespace {

template <int BT>
int resident_ctas(bool split) {
    using L = tgemm::Layout<BT>;
    const int smem = tmem_safe_smem(split ? L::kBytesRed : L::kBytesNoRed, L::kTmemCols);
    int by_smem = kSmemPerSm / (smem + kSmemPerCtaReserved);
    int by_tmem = 512 / L::kTmemCols;
    int by_threads = 2048 / tgemm::threads_for(BT);
    return by_smem < by_tmem ? (by_smem < by_threads ? by_smem : by_threads)
                             : (by_tmem < by_threads ? by_tmem : by_threads);
}

int resident_for(int bt, bool split) {
    switch (bt) {
        case 16: return resident_ctas<16>(split);
        case 32: return resident_ctas<32>(split);
        case 64: return resident_ctas<64>(split);
        default: return resident_ctas<128>(split);
    }
}

bool split_fits(int bt) {
    switch (bt) {
        case 16: return tgemm::Layout<16>::kSplitFits;
        case 32: return tgemm::Layout<32>::kSplitFits;
        case 64: return tgemm::Layout<64>::kSplitFits;
        default: return tgemm::Layout<128>::kSplitFits;
    }
}

}  // namespace

// K split over a cluster (a power of two up to 8): doubled while all CTAs still
// fit on the GPU at once (the split's reduction buffer lowers residency), so
// that more dequantising warps share each SM.  Each CTA keeps >= 2 weight
// stages (512 K-values).
//
// Between one and two tiles per SM (32-token tiles, whose split buffer still
// leaves two CTAs per SM) no split fits and whole tiles leave the SMs unevenly
// loaded (70B MLP: 224 tiles, 72 SMs with two, 80 with one).  There clusters of
// two either take two whole tiles or split one tile's K, so many of each that
// the grid is exactly two CTAs per SM: whole_pairs = tiles - SMs, giving every
// SM about 1.5 tiles of work instead of up to 2.  At 64-token tiles the split
// buffer would leave one CTA per SM, so there the split CTAs reduce through the
// activation ring instead, behind a cluster barrier after the K loop: worth it
// from 32 weight stages (K >= 8192: 70B MLP 48.0 -> 46.2 us, 20480 x 8192
// 46.5 -> 40.0 us), not at 16 (24576 x 4096: 25.0 -> 25.9 us).  The barrier
// measured slower on every other split, and 128-token tiles slower too.
void tmem_gemm_split(int64_t M, int64_t N, int64_t K, int num_sms, int* ks_out, int* whole_pairs_out,
                     int* red_in_ring_out) {
    const int bt = tmem_gemm_token_tile(M);
    const int64_t tiles = ((N + tgemm::kBM - 1) / tgemm::kBM) * ((M + bt - 1) / bt);
    const int64_t nws = (K + tgemm::kWK - 1) / tgemm::kWK;
    *ks_out = 1;
    *whole_pairs_out = 0;
    *red_in_ring_out = 0;
    const bool mixed_range = tiles > num_sms && tiles < 2 * int64_t(num_sms) && nws >= 4;
    if (bt == 64 && mixed_range && nws >= 32 && resident_for(bt, false) >= 2) {
        *ks_out = 2;
        *whole_pairs_out = int(tiles - num_sms);
        *red_in_ring_out = 1;
        return;
    }
    if (!split_fits(bt)) return;
    const int64_t cap = int64_t(resident_for(bt, true)) * num_sms;
    int ks = 1;
    while (ks < 8 && tiles * ks * 2 <= cap && nws / (2 * ks) >= 2) ks *= 2;
    *ks_out = ks;
    if (ks == 1 && bt == 32 && resident_for(bt, true) >= 2 && mixed_range) {
        *ks_out = 2;
        *whole_pairs_out = int(tiles - num_sms);
    }
}

int tmem_gemm_ksplit(int64_t M, int64_t N, int64_t K, int num_sms) {
    int ks, wp, ring;
    tmem_gemm_split(M, N, K, num_sms, &ks, &wp, &ring);
    return ks;
}

int64_t tmem_gemm_grid(int64_t M, int64_t N, int64_t K, int num_sms) {
    int ks, wp, ring;
    tmem_gemm_split(M, N, K, num_sms, &ks, &wp, &ring);
    const int64_t tiles = ((N + tgemm::kBM - 1) / tgemm::kBM) * ((M + tmem_gemm_token_tile(M) - 1) / tmem_gemm_token_tile(M));
    // whole_pairs clusters of ks CTAs hold ks tiles each, the rest one tile each
    return int64_t(ks) * (wp + (tiles - int64_t(wp) * ks));
}

cudaError_t launch_tmem_gemm(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                             int num_sms, bool prefetch_weights, bool c_tma, cudaStream_t stream) {
    tgemm::Params p;
    p.C = static_cast<uint16_t*>(C);
    p.bias = static_cast<const uint16_t*>(bias);
    p.ldc = s.ldc;
    p.status = status_ptr();
    if (!p.status) return cudaErrorSymbolNotFound;
    p.M = int(s.M);
    p.N = int(s.N);
    p.K = int(s.K);
    p.g_eff = int(s.g_eff);
    p.ng = int(s.ng);
    p.nkb = int((s.K + tgemm::kBK - 1) / tgemm::kBK);
    p.nws = int((s.K + tgemm::kWK - 1) / tgemm::kWK);
    p.gps = decode_scale_box_rows(p.g_eff, p.ng);
    tmem_gemm_split(s.M, s.N, s.K, num_sms, &p.ks, &p.whole_pairs, &p.red_in_ring);
    p.prefetch_weights = prefetch_weights ? 1 : 0;
    p.c_tma = c_tma ? 1 : 0;
    const int bt = tmem_gemm_token_tile(s.M);
    const int64_t ctas = tmem_gemm_grid(s.M, s.N, s.K, num_sms);
    if (ctas > int64_t(0x7fffffff)) return cudaErrorInvalidValue;   // beyond any C that fits in memory
    const int gx = int(ctas);
    const int gy = 1;
    switch (bt) {
        case 16: return launch_bt<16>(maps, p, s.bf16, s.zp, gx, gy, stream);
        case 32: return launch_bt<32>(maps, p, s.bf16, s.zp, gx, gy, stream);
        case 64: return launch_bt<64>(maps, p, s.bf16, s.zp, gx, gy, stream);
        default: return launch_bt<128>(maps, p, s.bf16, s.zp, gx, gy, stream);
    }
}

int take_status_tmem_gemm() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof(int));
    return v;
}

}  // namespace w4a16
