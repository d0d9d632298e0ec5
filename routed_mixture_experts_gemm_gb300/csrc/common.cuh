// Device-side helpers shared by the gbmoe kernels (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gbmoe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "gbmoe kernels target sm_103a (Blackwell tcgen05); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace gbmoe {

// ---------------------------------------------------------------- status
// First device-side error wins; the host reads and clears it.
__device__ __forceinline__ void record_error(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

// ------------------------------------------------------------- misc PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

// -------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
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

// Wait for the phase with the given parity to complete, giving up after
// `limit_ns` of wall time or as soon as *abort is raised by another role.
// Returns false on give-up (and raises *abort, records GBMOE_ERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, int* status,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1;
                record_error(status, GBMOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Plain bounded wait (no abort flag): used to drain in-flight work on the
// error path.  Returns false if the phase did not complete within limit_ns.
__device__ __forceinline__ bool mbar_wait_timeout(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------- clusters (CTA pairs)
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address in the shared::cluster window of the same variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Arrive on an mbarrier of another CTA of the cluster (release at cluster
// scope: this thread's earlier memory accesses are visible to a thread that
// observes the phase with an acquire at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// The same arrival with relaxed semantics (no fence: a release at cluster
// scope would wait for this thread's copies still in flight).  Used where
// the data the arrival announces has already landed and been fenced for the
// tensor cores.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// mbar_wait_bounded for a barrier that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint64_t* bar, uint32_t parity,
                                                          volatile int* abort, int* status,
                                                          uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1;
                record_error(status, GBMOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
// Every thread of every CTA of the cluster (all threads must call it).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// -------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load of box {x: inner (K) coordinate, y: row coordinate} into smem,
// completing `bytes` on the mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
// As tma_load_2d, for the odd CTA of a pair: the copy lands in this CTA's
// shared memory and completes on an mbarrier of the pair's even CTA
// (shared::cluster address `bar_cluster`), which counts both CTAs' bytes.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* map, uint32_t bar_cluster,
                                                 int x, int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// --------------------------------------------------------------- tcgen05
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
// CTA-pair forms (cta_group::2): one warp of EACH CTA of the pair executes
// alloc / relinquish / dealloc; the pair's allocation has the same column
// address in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[tmem] (+)= A . B^T on a CTA pair (M = 256, issued by the even CTA): A rows
// 0-127 come from this CTA's shared memory at a_desc and rows 128-255 from
// the odd CTA's at the same offset; B's first N/2 rows from this CTA and the
// last N/2 from the odd CTA; D rows 0-127 land in this CTA's tensor memory,
// rows 128-255 in the odd CTA's, each with all N columns.  bf16, fp32 accumulate.
// CTA-pair form of the block-scaled MMA (issued by the even CTA; each CTA's
// tensor memory holds the scale columns at the given addresses).
__device__ __forceinline__ void umma_mx_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}
// CTA-pair form of the shared memory -> TMEM scale copy: each CTA's chunk at
// the given shared memory offset into its own tensor memory.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// umma_bf16_pair with FP8 E4M3 operands (kind::f8f6f4, 32 K-elements per
// instruction).
__device__ __forceinline__ void umma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at this offset in every CTA of `cta_mask` when
// all previously issued tcgen05 ops of this thread (pair form) complete.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T with A and B in FP8 E4M3 (kind::f8f6f4,
// 32 K-elements per instruction), fp32 accumulate.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= (A . B^T) with per-32-element block scales (kind::mxf8f6f4
// block_scale, one UE8M0 scale per 32 K-elements of every A row and B row):
// A and B in E4M3 or E2M1 (one byte per element in shared memory), 32
// K-elements per instruction, fp32 accumulate.  sfa / sfb are the TMEM
// addresses of the scale columns; the byte of each 32-bit column used by this
// instruction is selected in the instruction descriptor.
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}
// Arrive once on `bar` when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
// 32 TMEM lanes x 16 consecutive 32-bit columns; thread i of the warp gets lane (base+i).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Shared memory -> TMEM: 32 rows of 16 bytes (row r at byte 16 r of the
// source) into lanes r of all four lane quarters, 4 consecutive 32-bit
// columns.  Issued by one thread; ordered with its later tcgen05.mma.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}
// Descriptor of a contiguous, unswizzled source of 16-byte rows (8-row core
// matrices 128 bytes apart in either direction).
__device__ __forceinline__ uint64_t smem_desc_rows16(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(128 >> 4) << 16;            // leading byte offset
    d |= static_cast<uint64_t>(128 >> 4) << 32;            // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (tcgen05)
    return d;                                              // swizzle mode 0: none
}

// Shared-memory matrix descriptor for a K-major bf16 tile stored as rows of
// BK elements with the matching swizzle: BK = 64 -> 128-byte rows, 128B
// swizzle, 8-row atoms of 1024 B; BK = 32 -> 64-byte rows, 64B swizzle,
// 8-row atoms of 512 B (atoms contiguous, tiles atom-aligned).
template <int BK>
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t saddr) {
    static_assert(BK == 64 || BK == 32, "128- or 64-byte rows");
    constexpr uint64_t atom = BK == 64 ? 1024 : 512;
    constexpr uint64_t layout = BK == 64 ? 2 : 4;          // 128B / 64B swizzle
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
    d |= (atom >> 4) << 32;                                // stride byte offset: 8-row atom
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (tcgen05)
    d |= layout << 61;                                     // swizzle mode
    return d;
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
// Instruction descriptor, kind::f8f6f4: D fp32, A and B E4M3 (type code 0),
// both K-major.
__device__ __forceinline__ uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// two fp32 values -> two OCP FP8 E4M3 codes (round to nearest even,
// saturating to +-448), the first in the low byte
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}
// MX element formats (argument values of the C ABI)
constexpr int kMxE4M3 = 0, kMxE2M1 = 1;
// Shared exponent of an MX block with largest magnitude amax >= 0:
// floor(log2(amax)) - emax clamped to [-127, 127] (0 for an all-zero block),
// floor(log2) read from the fp32 bits (subnormals by their leading one).
__device__ __forceinline__ int mx_block_exp(float amax, int emax) {
    const uint32_t b = __float_as_uint(amax);
    if (b == 0u) return 0;
    const int be = static_cast<int>(b >> 23);
    const int l = be ? be - 127 : (31 - __clz(static_cast<int>(b))) - 149;
    return min(127, max(-127, l - emax));
}
// Instruction descriptor, kind::mxf8f6f4 with block scales: A type a_fmt, B
// type b_fmt (0 = E4M3, 5 = E2M1), both K-major, UE8M0 scales (bit 23);
// bits 4-5 and 29-30 select the byte of the B and A scale columns (the
// 32-element K block within a group of four).
__device__ __forceinline__ uint32_t idesc_mx(int M, int N, uint32_t a_fmt, uint32_t b_fmt,
                                             uint32_t sf_byte) {
    return (sf_byte << 4) | (a_fmt << 7) | (b_fmt << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(M >> 4) << 24) | (sf_byte << 29);
}

}  // namespace gbmoe
