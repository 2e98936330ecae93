// ptx.cuh -- hand-written inline PTX for sm_103a: mbarriers, TMA, tcgen05.
//
// Every helper is one instruction (or a short fixed sequence) from the public
// PTX ISA; nothing here is generated. Shared-memory operands are 32-bit
// shared-window addresses (see smem_u32).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fp4 {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// One probe of the phase with the given parity; true once that phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---- acquire / release ---------------------------------------------------------

// try_wait with acquire semantics at cluster scope (for barriers that threads
// of the peer CTA arrive on).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of four mbarrier phases at once (acquire, cluster scope):
// bit i of the result is set when the phase of parity p[i] of barrier b[i] has
// completed. The four tests issue back to back, so their shared-memory latency
// is paid once.
__device__ __forceinline__ uint32_t mbar_test4_cluster(const uint32_t (&b)[4], const uint32_t (&p)[4])
{
    uint32_t r0, r1, r2, r3;
    asm volatile(
        "{\n\t.reg .pred q0, q1, q2, q3;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q0, [%4], %8;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q1, [%5], %9;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q2, [%6], %10;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 q3, [%7], %11;\n\t"
        "selp.u32 %0, 1, 0, q0;\n\t"
        "selp.u32 %1, 2, 0, q1;\n\t"
        "selp.u32 %2, 4, 0, q2;\n\t"
        "selp.u32 %3, 8, 0, q3;\n\t}"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3])
        : "memory");
    return r0 | r1 | r2 | r3;
}

__device__ __forceinline__ uint32_t ld_acquire_shared(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_shared(uint32_t addr, uint32_t v)
{
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---- TMA / bulk copies ---------------------------------------------------------

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA store of a box from this CTA's shared memory (bulk-group
// completion), with an L2 cache policy. The caller's generic writes to the box
// must be fenced to the async proxy first (fence_proxy_async_shared).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t x, int32_t y,
                                             uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(src), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// This thread's committed bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// This thread's committed bulk groups have completed (their writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic shared-memory writes before later async-proxy
// (TMA, tensor core) reads of them.
__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA load into this CTA's shared memory, completing its bytes on the
// mbarrier. CG = 2 (tcgen05 CTA pair): the mbarrier may be the peer CTA's.
template <int CG>
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t x,
                                            int32_t y)
{
    if constexpr (CG == 2) {
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
            : "memory");
    } else {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
            "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
            : "memory");
    }
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Global stores with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void st_global_v4_hint(void *p, const uint4 &v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

// 32 bytes (a whole sector) from one thread; the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8_hint(void *p, const uint32_t (&w)[8], uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void st_global_b32_hint(void *p, uint32_t v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(policy) : "memory");
}

__device__ __forceinline__ void st_global_b16_hint(void *p, uint16_t v, uint64_t policy)
{
    asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(p), "h"(v), "l"(policy) : "memory");
}

// ---- tcgen05: tensor memory ------------------------------------------------------

// TMEM allocation. With CG = 2 one warp of each CTA of the pair issues it.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                     : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish()
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 async operation issued so far by this
// thread has completed. CG = 2: the arrive goes to the barrier at the same
// offset in each CTA of the pair named in `mask` (default both).
template <int CG>
__device__ __forceinline__ void tc_commit(uint32_t bar, uint16_t mask = 3)
{
    if constexpr (CG == 2)
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                bar),
            "h"(mask)
            : "memory");
    else
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
}

// Copy one 32-row x 16-byte shared-memory matrix into 4 TMEM columns, repeated
// in all four 32-lane sub-partitions (the block-scale factor placement). CG = 2:
// done in both CTAs of the pair, each from its own shared memory.
template <int CG>
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Block-scaled FP4 MMA, D[tmem] (+)= A[smem] x B[smem]^T with K = 64:
// MX = false: 16-element scale blocks, UE4M3 scales (scale_vec::4X);
// MX = true:  32-element scale blocks, UE8M0 scales (scale_vec::2X).
template <int CG, bool MX>
__device__ __forceinline__ void tc_mma_fp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
#define FP4_MMA_ASM(GROUP, VEC)                                                                                  \
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"                                            \
                 "tcgen05.mma.cta_group::" GROUP ".kind::mxf4nvf4.block_scale.scale_vec::" VEC                  \
                 " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),                                          \
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)               \
                 : "memory")
    if constexpr (CG == 2) {
        if constexpr (MX) FP4_MMA_ASM("2", "2X"); else FP4_MMA_ASM("2", "4X");
    } else {
        if constexpr (MX) FP4_MMA_ASM("1", "2X"); else FP4_MMA_ASM("1", "4X");
    }
#undef FP4_MMA_ASM
}

// 32 lanes x 8 columns of 32-bit TMEM -> 8 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

// 32 lanes x 32 columns of 32-bit TMEM -> 32 registers per thread (thread i gets lane i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 32 lanes x 16 columns of 32-bit TMEM -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// This warp's 32 lanes x 1 / 8 / 16 consecutive 32-bit TMEM columns from
// registers (thread i writes lane i). Complete once tcgen05.wait::st returns.
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r) : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint32_t *r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t *r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t *r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                 "%12, %13, %14, %15, %16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.ld destinations are undefined until tcgen05.wait::ld; the compiler
// does not know that, so after the wait every destination register is passed
// through an empty asm statement (ordered after the wait, no instructions) and
// later uses depend on it.
template <int N>
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[N])
{
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// ---- register split between warpgroups -------------------------------------------------------

// Every warp of a warpgroup executes the same one; .inc waits until the CTA's
// pool (its launch registers) has room, so the .dec's of the other warpgroups
// must free at least what the .inc's take.
template <uint32_t N>
__device__ __forceinline__ void regs_raise()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void regs_lower()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---- clusters ------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared::cluster address of `addr` (a shared address of this CTA) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by a shared::cluster address (possibly another
// CTA's), with the default release at CTA scope. The kernels use it only to hand
// TMEM over (scale columns stored, accumulator drained), which the tcgen05 wait
// and thread-sync fences order; no generic memory passes through it. A release
// at cluster scope would also wait for the SM's outstanding memory traffic to be
// acknowledged: measured, that made each such arrive cost about 1.7k cycles
// while the operand copies were streaming.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Every thread of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same barriers for threads that reach them from different places in the
// code (the warp-role branches): the non-.aligned forms.
__device__ __forceinline__ void cluster_sync_any()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void cta_sync_any()
{
    asm volatile("barrier.sync 0;" ::: "memory");
}

// ---- descriptors ---------------------------------------------------------------------

// tcgen05 shared-memory matrix descriptor: start address, leading/stride byte
// offsets (16-byte units), fixed version bits 46..48 = 0b001, base offset 0,
// relative LBO mode, swizzle mode in bits 61..63 (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
    return d;
}

// Instruction descriptor of the block-scaled FP4 MMA (kind::mxf4nvf4), both
// operands E2M1 (format code 1), K-major, dense, no negation:
//   bits 4-5 B scale-factor byte id, 7-9 A format, 10-12 B format, 17-22 N>>3,
//   23 scale type (0 UE4M3, 1 UE8M0), 27-28 M>>7, 29-30 A scale-factor byte id.
__host__ __device__ constexpr uint32_t idesc_fp4(uint32_t m, uint32_t n, bool ue8m0,
                                                        uint32_t a_sf_id, uint32_t b_sf_id)
{
    uint32_t d = 0;
    d |= (b_sf_id & 3u) << 4;
    d |= 1u << 7;
    d |= 1u << 10;
    d |= ((n >> 3) & 0x3Fu) << 17;
    d |= (ue8m0 ? 1u : 0u) << 23;
    d |= ((m >> 7) & 3u) << 27;
    d |= (a_sf_id & 3u) << 29;
    return d;
}

}  // namespace fp4

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its writes are visible (a no-op when this grid was not
// launched as a dependent), and let the next grid start its prologue early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
