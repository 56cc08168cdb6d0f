// Host side of the small-M kernel: launch planning (cluster split of K, ring
// depth, shared memory), dispatch to the per-dtype instantiations, and the
// module's device status word.  The kernel itself is in decode_kernel.cuh.
#include <mutex>

#include "decode_kernel.cuh"

namespace w4a16 {

namespace {

__device__ int g_status;

int stage_bytes_for(int64_t M) {
    using namespace decode;
    const int a_slot = int((M + 7) / 8 * 8) * 64;
    const int raw = kWBytes + (kBoxK / kSubK) * a_slot + kMaxGps * kBN * 2 + kMaxGps * 16 * 4;
    return (raw + 1023) / 1024 * 1024;
}

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

}  // namespace

// Groups a 256-wide K box can touch: 256 / G for G in {32, 64, 128}; one for
// G >= 256 (a multiple of 256) and for a single group spanning K (G = -1,
// which can be smaller than 32 only when K itself is).
int decode_scale_box_rows(int64_t g_eff, int64_t ng) {
    if (ng == 1 || g_eff >= decode::kBoxK) return 1;
    return int(decode::kBoxK / g_eff);
}

// Host-side plan for a shape: cluster size (K split), ring depth, shared memory.
// K is split over up to 8 CTAs until there are about three CTAs per SM; each
// ring stage holds one 256-wide K box.
bool plan_decode(int64_t M, int64_t N, int64_t K, int num_sms, int* ks_out, int* stages_out,
                 size_t* smem_out, int* nt_out) {
    using namespace decode;
    if (M < 1 || M > kDecodeMaxM) return false;
    const int nt = M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8;
    const int64_t row_tiles = (N + kBN - 1) / kBN;
    const int64_t nboxes = (K + kBoxK - 1) / kBoxK;
    const int64_t target = 3LL * num_sms;
    int ks = 1;
    while (ks < 8 && row_tiles * ks < target && 2 * ks <= nboxes) ks *= 2;
    const int64_t boxes_per = (nboxes + ks - 1) / ks;
    const int sb = stage_bytes_for(M);
    const size_t red = ks > 1 ? size_t(kBN) * 8 * nt * 4 : 0;
    // two stages keep a box in flight behind the one being consumed; more
    // stages only while they still leave room for three CTAs per SM
    int want = int(boxes_per < 2 ? boxes_per : 2);
    for (int s = 3; s <= kMaxStages && s <= boxes_per; ++s)
        if (size_t(s) * sb + red + 2048 <= 74 * 1024) want = s;
    for (int stages = want; stages >= 1; --stages) {
        const size_t smem = size_t(stages) * sb + 128 + red + 1024;
        if (smem <= 227 * 1024) {
            *ks_out = ks;
            *stages_out = stages;
            *smem_out = smem;
            *nt_out = nt;
            return true;
        }
    }
    return false;
}

cudaError_t launch_decode(const CUtensorMap* maps, void* C, const LayerShape& s, int num_sms,
                          bool prefetch_weights, cudaStream_t stream) {
    using namespace decode;
    int ks, stages, nt;
    size_t smem;
    if (!plan_decode(s.M, s.N, s.K, num_sms, &ks, &stages, &smem, &nt)) return cudaErrorInvalidValue;
    Params p;
    p.C = static_cast<uint16_t*>(C);
    p.status = status_ptr();
    if (!p.status) return cudaErrorSymbolNotFound;
    p.M = int(s.M);
    p.N = int(s.N);
    p.K = int(s.K);
    p.g_eff = int(s.g_eff);
    p.nboxes = int((s.K + kBoxK - 1) / kBoxK);
    p.ks = ks;
    p.stages = stages;
    p.gps = decode_scale_box_rows(s.g_eff, s.ng);
    if (p.gps < 1 || p.gps > kMaxGps) return cudaErrorInvalidValue;   // never expected
    p.a_slot = int((s.M + 7) / 8 * 8) * 64;
    p.stage_bytes = stage_bytes_for(s.M);
    p.red_off = stages * p.stage_bytes + 128;
    p.prefetch_weights = prefetch_weights ? 1 : 0;
    const int wpg = (s.ng == 1 || s.g_eff >= kBoxK) ? 8 : int(s.g_eff / 32);
    const int grid = int((s.N + kBN - 1) / kBN) * ks;
    return s.bf16 ? launch_bf16(s.zp, wpg, nt, maps, p, grid, smem, stream)
                  : launch_fp16(s.zp, wpg, nt, maps, p, grid, smem, stream);
}

int take_status_decode() {
    int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof(int));
    return v;
}

}  // namespace w4a16
