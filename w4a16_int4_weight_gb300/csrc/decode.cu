// Host side of the small-M kernel: launch planning (cluster split of K, ring
// depth, shared memory), dispatch to the per-dtype instantiations, and the
// module's device status word.  The kernel itself is in decode_kernel.cuh.
#include <algorithm>
#include <mutex>

#include "decode_kernel.cuh"

namespace w4a16 {

namespace {

__device__ int g_status;

// Token tiles of 8 of the kernel instantiation that serves M tokens.
int nt_for(int64_t M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// Activation box slot: one token tile: M rows of 256 values (512 bytes each), in
// 1024-byte units so that the scales behind it stay 128-byte aligned for TMA;
// more: four 64-value sub-boxes of the kernel's 8 NT rows x 128 bytes, each
// 1024-byte aligned for the 128-byte swizzle.
int a_slot_for(int64_t M) { return M <= 8 ? int((M * 512 + 1023) / 1024 * 1024) : 4096 * nt_for(M); }

// Columns of the split-K reduction buffer: partials travel as pairs of MMA
// columns.  One token tile: tokens 2t, 2t + 1, so M rounded up to even; more:
// tokens 8j + t and 8j + t + 4 (t < 4), one pair for each t with 8j + t < M.
int red_cols_for(int64_t M) {
    return M <= 8 ? int((M + 1) / 2 * 2) : int(2 * (4 * (M / 8) + std::min<int64_t>(4, M % 8)));
}

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

// Host-side plan for a shape: cluster size ks (K split) and ring depth, from a
// cost model fitted to a grid of GB300 timings (N 4096..28672, K 2048..14336,
// M 1 and 16, every ks and depth; the model's choice is within 3% of the best
// measured plan on average, 10% at worst):
//   work      boxes on the busiest SM: ceil(CTAs / SMs) * boxes per CTA;
//   waves     CTAs beyond what fits on the GPU at once (20% per extra wave);
//   in flight weight bytes requested ahead per SM (up to 10% below 64 KB);
//   room      small layers run best when the next kernel's CTAs fit beside
//             this one's, so that their weight prefetch (PDL) overlaps it
//             (60% when they do not fit, for <= 12 boxes per SM); with
//             32-wide groups (eight rescales per box) only when the SMs hold
//             more than 2.5 CTAs on average (measured, M = 8 with zero points:
//             11008 x 4096 four-way split 10.6 us against two-way 13.1 us,
//             14336 x 4096 four-way 14.6 us against two-way 13.4 us);
//   one CTA   a lone CTA per SM hides latency worse (20%);
//   split     each doubling of ks costs 3% (reduction).
bool plan_decode(int64_t M, int64_t N, int64_t K, int64_t g_eff, int64_t ng, bool zp,
                 int num_sms, int* ks_out, int* stages_out, size_t* smem_out, int* nt_out) {
    using namespace decode;
    if (M < 1 || M > kDecodeMaxM || num_sms < 1) return false;
    const int nt = nt_for(M);
    const int64_t row_tiles = (N + kBN - 1) / kBN;
    const int64_t nboxes = (K + kBoxK - 1) / kBoxK;
    const int gps = decode_scale_box_rows(g_eff, ng);
    const int sb = stage_bytes_for(M, gps, zp);
    const int max_ctas = nt == 1 ? 4 : nt == 2 ? 3 : 1;   // register limit of the instantiations
    constexpr int kMaxPlanStages = 5;                       // the range the model was fitted on
    double best_cost = 0.0;
    int best_ks = 0, best_st = 0;
    size_t best_smem = 0;
    for (int ks = 1; ks <= 8 && ks <= nboxes; ks *= 2) {
        const int64_t ctas = row_tiles * ks;
        const int64_t per = (ctas + num_sms - 1) / num_sms;
        const int64_t bp = (nboxes + ks - 1) / ks;
        const size_t red = ks > 1 ? size_t(kBN) * red_cols_for(M) * 4 : 0;
        for (int st = 1; st <= kMaxPlanStages; ++st) {
            if (st > bp && st > 1) break;
            const size_t smem = size_t(st) * sb + kBarBytes + red + 1024;
            if (smem > 227 * 1024) break;
            int64_t r = int64_t(228 * 1024) / int64_t(smem + 1024);
            if (r > max_ctas) r = max_ctas;
            if (r < 1) break;
            const int64_t waves = (per + r - 1) / r;
            const int64_t ahead = st == 1 ? 1 : (st < bp ? st - 1 : bp);
            const double inflight_kb = double(per < r ? per : r) * double(ahead) * 16.0;
            const double work = double(per * bp);
            double cost = work * (1.0 + 0.2 * double(waves - 1));
            if (inflight_kb < 64.0) cost *= 1.0 + 0.1 * (64.0 - inflight_kb) / 64.0;
            if (work <= 12.0 && r - per < per && (gps < 8 || 2 * ctas > 5 * int64_t(num_sms))) cost *= 1.6;
            if (per == 1) cost *= 1.2;
            int lg = 0;
            for (int k = ks; k > 1; k >>= 1) ++lg;
            cost *= 1.0 + 0.03 * lg;
            // ties: smaller split, then deeper ring
            if (best_ks == 0 || cost < best_cost - 1e-9) {
                best_cost = cost;
                best_ks = ks;
                best_st = st;
                best_smem = smem;
            } else if (cost <= best_cost + 1e-9 && ks == best_ks && st > best_st) {
                best_st = st;
                best_smem = smem;
            }
        }
    }
    if (best_ks == 0) return false;
    *ks_out = best_ks;
    *stages_out = best_st;
    *smem_out = best_smem;
    *nt_out = nt;
    return true;
}

bool decode_plan_exists(int64_t M, int64_t N, int64_t K, int64_t g_eff, int64_t ng, bool zp) {
    int ks, stages, nt;
    size_t smem;
    return plan_decode(M, N, K, g_eff, ng, zp, 1, &ks, &stages, &smem, &nt);
}

cudaError_t launch_decode(const CUtensorMap* maps, void* C, const void* bias, const LayerShape& s,
                          int num_sms, bool prefetch_weights, cudaStream_t stream) {
    using namespace decode;
    int ks, stages, nt;
    size_t smem;
    if (!plan_decode(s.M, s.N, s.K, s.g_eff, s.ng, s.zp, num_sms, &ks, &stages, &smem, &nt))
        return cudaErrorInvalidValue;
    Params p;
    p.C = static_cast<uint16_t*>(C);
    p.bias = static_cast<const uint16_t*>(bias);
    p.ldc = s.ldc;
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
    if (nt >= 2 && p.a_slot < 4 * 1024 * nt) return cudaErrorInvalidValue;   // sub-boxes must fit (never expected)
    p.mpr = red_cols_for(s.M);
    p.stage_bytes = stage_bytes_for(s.M, p.gps, s.zp);
    p.red_off = stages * p.stage_bytes + kBarBytes;
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
