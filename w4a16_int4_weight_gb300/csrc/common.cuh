// Device helpers shared by the libw4a16 kernels: inline PTX for mbarriers, TMA,
// tcgen05 (TMEM + UMMA), legacy warp MMA, bounded waits and the int4 unpack.
// sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace w4a16 {

// ---------------------------------------------------------------------------
// Bounded waits.  Every spin on a barrier gives up after kWaitLimitNs of
// global time, records a status code and lets the kernel return.
// ---------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters: split barrier and stores into a peer CTA's shared memory
// that complete on the peer's mbarrier (no cluster-scope release fence).
// ---------------------------------------------------------------------------
// Every thread of every CTA of the cluster arrives; relaxed: orders nothing by
// itself (mbarrier initialisation is published by fence_mbar_init before it).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

// Arrive with release semantics: this thread's earlier memory accesses (and what
// it has observed) are ordered before the cluster peers' accesses after their wait.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait;" ::: "memory");
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
    return r;
}

// 8-byte store into a (possibly remote) CTA's shared memory; its completion is
// counted as 8 transaction bytes on that CTA's mbarrier `remote_bar`.
__device__ __forceinline__ void st_async_f32x2(uint32_t remote_addr, float a, float b, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
                 ::"r"(remote_addr), "f"(a), "f"(b), "r"(remote_bar)
                 : "memory");
}

// 16-byte form of st_async_f32x2 (16-byte aligned address).
__device__ __forceinline__ void st_async_f32x4(uint32_t remote_addr, float a, float b, float c, float d,
                                               uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(remote_addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
                 : "memory");
}

// Barrier `id` (1..15; 0 is __syncthreads) over `threads` threads, a multiple of 32.
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// The same barrier, returning whether `pred` was true in any participating thread.
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(pred)), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete.  Returns false (after writing
// `site` into *status) if it did not within `limit_ns` of global time.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, uint32_t parity, int* status, int site,
                                                uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
            atomicCAS(status, 0, site);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, int site) {
    return mbar_wait_limit(bar, parity, status, site, kWaitLimitNs);
}

// The same wait with a long suspend-time hint on each try: a waiting thread
// sleeps until the phase completes instead of re-polling, so waiting warps
// leave their issue slots to the others (the limit stays bounded).
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, int* status, int site,
                                                uint64_t limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_u32(bar);
    auto try_wait = [&]() {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 2000000;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        return ok != 0;
    };
    if (try_wait()) return true;
    const uint64_t t0 = global_timer_ns();
    while (!try_wait()) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicCAS(status, 0, site);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), completion through an mbarrier transaction count
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// L2 policy for data read once: evicted first, so that it does not push out
// what is reused (activations, outputs, the next layer's early weight fetches).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// tma_load_2d with an L2 cache policy (l2_evict_first_policy) on the reads.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                 int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// TMA tensor store of a shared-memory tile to the tensor map's box at (x, y),
// completed through the bulk-group mechanism; elements outside the tensor are
// not written.  Callers make their shared-memory writes visible to the async
// proxy first (fence_proxy_async_smem + a barrier).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's committed bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA / tensor core) before it signals a consumer.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA (cta_group::1)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::f16 (fp16/bf16 in, fp32 acc).
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row groups 1024 bytes apart; the
// layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (16-29, unused for this layout),
// stride byte offset >> 4 (32-45), descriptor version 1 (46-47), base offset 0
// (49-51), swizzle mode 2 = 128B (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* tile) {
    const uint64_t addr = smem_u32(tile);
    return ((addr >> 4) & 0x3FFFull) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor for kind::f16 with fp32 accumulation, both operands
// K-major: D format (bits 4-5) = 1 (f32); A and B formats (7-9, 10-12) = 0 fp16
// or 1 bf16; N >> 3 in bits 17-22; M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, int m, int n) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// columns [col, col+32) of TMEM lane (warp's lane quarter base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Warp-level MMA m16n8k16, fp32 accumulate (used by the small-M kernel, where
// the weight stream, not the tensor pipe, sets the speed).
// ---------------------------------------------------------------------------
// d = a . b + c (ZERO_C: c = 0, so d is overwritten without reading it).
template <bool BF16, bool ZERO_C = false>
__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], const uint32_t (&a)[4],
                                             uint32_t b0, uint32_t b1) {
    if constexpr (ZERO_C) {
        if constexpr (BF16) {
            asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
                : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
        } else {
            asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
                : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
        }
    } else {
        if constexpr (BF16) {
            asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
        } else {
            asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
        }
    }
}

// ---------------------------------------------------------------------------
// int4 -> 16-bit float pairs by OR-ing nibbles into the mantissa of a "magic"
// constant (the fp16 form, 0x6400 = 1024 with ulp 1, is the pages'
// _int4_pair_to_fp16x2; bf16 uses 0x4300 = 128, whose ulp is also 1).
// (a & b) | c in one LOP3.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ uint32_t as_u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t v) { return *reinterpret_cast<__nv_bfloat162*>(&v); }
__device__ __forceinline__ __half2 as_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// Packed word -> the four (even, odd) K-value pairs as exact integers (q - z)
// in 16-bit float lanes.  Pair p holds values (2p, 2p+1) of the word: low lane
// value 2p (bits 4p..4p+3), high lane value 2p+1 (bits 16+4p..).
// bf16: (w >> 4p) & 0x000F000F | 0x43004300 -> 128 + v; subtract (128 + z).
// fp16: pairs 0 and 2 as 1024 + v; pairs 1 and 3 are taken unshifted with mask
// 0x00F000F0 as 1024 + 16 v and brought back by (x * 1/16) - (64 + z), exact.
struct ZeroConst {
    uint32_t lo;   // 16-bit float pair to subtract from (magic + v)
    uint32_t hi;   // fp16 only: pair added after the 1/16 scaling, -(64 + z)
};

// Bit patterns built with integer operations (z in 0..15, all values exact):
//   bf16 128 + z     = 0x4300 + z        (ulp 1 in [128, 256))
//   fp16 1024 + z    = 0x6400 + z        (ulp 1 in [1024, 2048))
//   fp16 -(64 + z)   = 0xD400 + 16 z     (ulp 1/16 in [64, 128))
template <bool BF16>
__device__ __forceinline__ ZeroConst make_zero_const(int z) {
    ZeroConst c;
    const uint32_t u = uint32_t(z) & 0xFu;
    if constexpr (BF16) {
        c.lo = (0x4300u | u) * 0x00010001u;
        c.hi = 0;
    } else {
        c.lo = (0x6400u | u) * 0x00010001u;
        c.hi = (0xD400u | (u << 4)) * 0x00010001u;
    }
    return c;
}

template <bool BF16>
__device__ __forceinline__ void unpack_word(uint32_t w, const ZeroConst& zc, uint32_t (&p)[4]) {
    if constexpr (BF16) {
        const uint32_t m = 0x000F000Fu, magic = 0x43004300u;
        const __nv_bfloat162 z2 = as_bf2(zc.lo);
        p[0] = as_u32(__hsub2(as_bf2(lop3_and_or(w, m, magic)), z2));
        p[1] = as_u32(__hsub2(as_bf2(lop3_and_or(w >> 4, m, magic)), z2));
        p[2] = as_u32(__hsub2(as_bf2(lop3_and_or(w >> 8, m, magic)), z2));
        p[3] = as_u32(__hsub2(as_bf2(lop3_and_or(w >> 12, m, magic)), z2));
    } else {
        const uint32_t magic = 0x64006400u;
        const __half2 z2 = as_h2(zc.lo);
        const __half2 zh = as_h2(zc.hi);
        const __half2 sixteenth = __half2(__float2half_rn(0.0625f), __float2half_rn(0.0625f));
        const uint32_t w8 = w >> 8;
        p[0] = as_u32(__hsub2(as_h2(lop3_and_or(w, 0x000F000Fu, magic)), z2));
        p[1] = as_u32(__hfma2(as_h2(lop3_and_or(w, 0x00F000F0u, magic)), sixteenth, zh));
        p[2] = as_u32(__hsub2(as_h2(lop3_and_or(w8, 0x000F000Fu, magic)), z2));
        p[3] = as_u32(__hfma2(as_h2(lop3_and_or(w8, 0x00F000F0u, magic)), sixteenth, zh));
    }
}

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t bits) {
    if constexpr (BF16) {
        return __uint_as_float(uint32_t(bits) << 16);
    } else {
        return __half2float(__ushort_as_half(bits));
    }
}

// Quiet NaN of the dtype: the value of outputs that a failed (timed-out) wait
// left incomplete.
template <bool BF16>
__device__ __forceinline__ uint16_t nan_bits() {
    return BF16 ? uint16_t(0x7FC0) : uint16_t(0x7E00);
}

template <bool BF16>
__device__ __forceinline__ uint16_t from_f32(float v) {
    if constexpr (BF16) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else {
        return __half_as_ushort(__float2half_rn(v));
    }
}

// Multiply a pair of exact integers (q - z) by the scale pair and round once.
template <bool BF16>
__device__ __forceinline__ uint32_t scale_pair(uint32_t qz, uint32_t s2) {
    if constexpr (BF16) {
        return as_u32(__hmul2(as_bf2(qz), as_bf2(s2)));
    } else {
        return as_u32(__hmul2(as_h2(qz), as_h2(s2)));
    }
}

}  // namespace w4a16
