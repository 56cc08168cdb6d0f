// Host side of the small-M kernel: launch planning (cluster split of K, ring
// depth, shared memory), dispatch to the per-dtype instantiations, and the
// module's device status word.  The kernel itself is in decode_kernel.cuh.
#include <mutex>

#include "decode_kernel.cuh"

namespace w4a16 {

namespace {

__device__ int g_status;

// Activation box slot: 8 * NT token rows of 256 values.
int a_slot_for(int64_t M) { return 4096 * (M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8); }

int stage_bytes_for(int64_t M, int gps, bool zp) {
    using namespace decode;
    const int a_slot = a_slot_for(M);
    const int raw = kWBytes + a_slot + gps * kBN * 2 + (zp ? gps * 16 * 4 : 0);
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
// K is split over up to 8 CTAs until there are about three CTAs per SM.  Each
// ring stage holds one 256-wide K box.
bool plan_decode(int64_t M, int64_t N, int64_t K, int64_t g_eff, int64_t ng, bool zp,
                 int num_sms, int* ks_out, int* stages_out, size_t* smem_out, int* nt_out) {
    using namespace decode;
    if (M < 1 || M > kDecodeMaxM) return false;
    const int nt = M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8;
    const int64_t row_tiles = (N + kBN - 1) / kBN;
    const int64_t nboxes = (K + kBoxK - 1) / kBoxK;
    const int64_t target = 3LL * num_sms;
    int ks = 1;
    while (ks < 8 && row_tiles * ks < target && 2 * ks <= nboxes) ks *= 2;
    const int64_t boxes_per = (nboxes + ks - 1) / ks;
    const int sb = stage_bytes_for(M, decode_scale_box_rows(g_eff, ng), zp);
    const size_t red = ks > 1 ? size_t(kBN) * 8 * nt * 4 : 0;
    auto smem_for = [&](int s) { return size_t(s) * sb + 128 + red + 1024; };
    const size_t sm_bytes = 228 * 1024;
    const int max_ctas = nt == 1 ? 4 : nt == 2 ? 3 : 1;   // register limit of the instantiations
    // Pick the depth: at least ~96 KB of weight boxes in flight per SM (enough to
    // cover HBM latency at full bandwidth), then as many resident CTAs (consumer
    // warps) as possible, then the shallowest ring.
    int best = 1;
    long best_ctas = -1, best_inflight = -1;
    bool best_ok = false;
    for (int s = 1; s <= kMaxStages && s <= boxes_per; ++s) {
        const size_t sm = smem_for(s);
        if (sm > 227 * 1024) break;
        long ctas = long(sm_bytes / (sm + 1024));
        if (ctas > max_ctas) ctas = max_ctas;
        const long ahead = s == boxes_per ? s : s - 1;
        const long inflight = ctas * ahead * kWBytes;
        const bool ok = inflight >= 96 * 1024;
        const bool better = ok ? (!best_ok || ctas > best_ctas) : (!best_ok && inflight > best_inflight);
        if (better) {
            best = s;
            best_ctas = ctas;
            best_inflight = inflight;
            best_ok = ok;
        }
    }
    for (int stages = best; stages >= 1; --stages) {
        const size_t smem = smem_for(stages);
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
    if (!plan_decode(s.M, s.N, s.K, s.g_eff, s.ng, s.zp, num_sms, &ks, &stages, &smem, &nt))
        return cudaErrorInvalidValue;
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
    p.a_slot = a_slot_for(s.M);
    p.stage_bytes = stage_bytes_for(s.M, p.gps, s.zp);
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
