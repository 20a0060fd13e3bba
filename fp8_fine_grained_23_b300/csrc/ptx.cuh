// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarriers with bounded waits, TMA tile loads,
// and the tcgen05 (5th-generation tensor core) MMA / TMEM instructions used by the GEMMs.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace fp8bs {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint32_t ld_shared_volatile_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_volatile_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Waits until the phase with the given parity has completed. Gives up (returns false) when
// `budget` SM clock cycles have passed or when another role of the CTA has set the shared word
// at `abort_addr` (0: no abort word).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t abort_addr,
                                          long long budget)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_addr != 0 && ld_shared_volatile_u32(abort_addr) != 0) return false;
        if (clock64() - t0 > budget) return false;
    }
}

// ------------------------------------------------------------------------------------
// TMA (tensor memory accelerator) tile loads, completion counted on an mbarrier
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// TMA tile store: the box at (x, y) of `map` from shared memory at `src` (laid out as the map's
// box with its swizzle), tracked by the issuing thread's bulk async-groups. Elements outside the
// tensor are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     map),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Until at most N of this thread's bulk async-groups are still reading their shared memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Until at most N of this thread's bulk async-groups are still in flight (writes performed).
template <int N>
__device__ __forceinline__ void bulk_wait_group()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------------------------
// Thread-block clusters
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster: release own prior memory operations, then wait for
// all CTAs of the cluster and acquire theirs.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// CTA pairs (cta_group::2): two CTAs of a cluster (ranks 2k, 2k+1) share one MMA
// ------------------------------------------------------------------------------------

// Shared-memory address of the same variable in the CTA of rank `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of any CTA in the cluster (address from mapa_shared). Default semantics
// (release at CTA scope): a cluster-scope release would make every arrive wait for all of the
// thread's outstanding memory traffic, and the one ordering the pair needs (TMEM reads done
// before the peer's MMA overwrites them) is already given by tcgen05.wait::ld and
// tcgen05.fence::before_thread_sync.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Tile load into this CTA's shared memory whose completion is counted on an mbarrier that may
// live in the pair's other CTA (`bar_cluster` from mapa_shared): both CTAs of a pair feed the
// pair's MMA, which waits on the even CTA's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// Plain (untiled) bulk copy of `bytes` (a multiple of 16) from global memory into shared memory;
// both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Asynchronous 4-byte copy global -> shared; with src_bytes == 0 the destination is zero-filled
// and nothing is read.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// Arrives on `bar` (without raising its expected count) once every cp.async issued so far by
// this thread has completed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later async-proxy (TMA)
// accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads, fences
// ------------------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t holder_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     holder_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// The same three operations for a CTA pair: one warp in each CTA of the pair performs them
// together, and the allocation is made at the same TMEM address in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t holder_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     holder_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> FP32, one instruction of K = 32.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Pair MMA (issued by the even CTA of a CTA pair): D (+)= A * B^T with M = 256 rows, A rows
// 0..127 and B rows 0..N/2-1 from this CTA's shared memory, the other halves from the peer CTA's
// shared memory at the same addresses; each CTA's TMEM receives its 128 rows of D.
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on the mbarrier at offset `bar` of every CTA in `cta_mask` when the pair MMAs
// issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair_multicast(uint32_t bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"(cta_mask)
        : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.wait::ld that also names the destination registers of the load it completes, so the
// compiler cannot move any use of them above the wait.
__device__ __forceinline__ void tmem_wait_ld(uint64_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+l"(r[0]), "+l"(r[1]), "+l"(r[2]), "+l"(r[3]), "+l"(r[4]), "+l"(r[5]),
                   "+l"(r[6]), "+l"(r[7]), "+l"(r[8]), "+l"(r[9]), "+l"(r[10]), "+l"(r[11]),
                   "+l"(r[12]), "+l"(r[13]), "+l"(r[14]), "+l"(r[15])
                 :
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns, returned as 16 packed pairs: r[i] holds columns
// 2i (low half) and 2i + 1 (high half) of this thread's lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint64_t (&r)[16])
{
    asm volatile(
        "{\n .reg .b32 t<32>;\n"
        " tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15,"
        "t16,t17,t18,t19,t20,t21,t22,t23,t24,t25,t26,t27,t28,t29,t30,t31}, [%16];\n"
        " mov.b64 %0, {t0, t1};\n mov.b64 %1, {t2, t3};\n mov.b64 %2, {t4, t5};\n"
        " mov.b64 %3, {t6, t7};\n mov.b64 %4, {t8, t9};\n mov.b64 %5, {t10, t11};\n"
        " mov.b64 %6, {t12, t13};\n mov.b64 %7, {t14, t15};\n mov.b64 %8, {t16, t17};\n"
        " mov.b64 %9, {t18, t19};\n mov.b64 %10, {t20, t21};\n mov.b64 %11, {t22, t23};\n"
        " mov.b64 %12, {t24, t25};\n mov.b64 %13, {t26, t27};\n mov.b64 %14, {t28, t29};\n"
        " mov.b64 %15, {t30, t31};\n}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]),
          "=l"(r[7]), "=l"(r[8]), "=l"(r[9]), "=l"(r[10]), "=l"(r[11]), "=l"(r[12]),
          "=l"(r[13]), "=l"(r[14]), "=l"(r[15])
        : "r"(taddr)
        : "memory");
}

// tcgen05.wait::ld naming the 8 packed destination pairs of a 16-column load.
__device__ __forceinline__ void tmem_wait_ld(uint64_t (&r)[8])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+l"(r[0]), "+l"(r[1]), "+l"(r[2]), "+l"(r[3]), "+l"(r[4]), "+l"(r[5]),
                   "+l"(r[6]), "+l"(r[7])
                 :
                 : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns as 8 packed pairs (columns 2i, 2i + 1 in r[i]).
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint64_t (&r)[8])
{
    asm volatile(
        "{\n .reg .b32 t<16>;\n"
        " tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15}, [%8];\n"
        " mov.b64 %0, {t0, t1};\n mov.b64 %1, {t2, t3};\n mov.b64 %2, {t4, t5};\n"
        " mov.b64 %3, {t6, t7};\n mov.b64 %4, {t8, t9};\n mov.b64 %5, {t10, t11};\n"
        " mov.b64 %6, {t12, t13};\n mov.b64 %7, {t14, t15};\n}"
        : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]),
          "=l"(r[7])
        : "r"(taddr)
        : "memory");
}

// Two FP32 lanes packed in 64 bits: the value (s, s).
__device__ __forceinline__ uint64_t f32x2_splat(float s)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
    return r;
}

// acc = fma(p, s2, acc) on packed FP32 pairs: two IEEE round-to-nearest fused multiply-adds.
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t p, uint64_t s2)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(p), "l"(s2));
}

// Packed FP32x2 multiply, each lane rounded to nearest even.
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float f32x2_lo(uint64_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v));
}

__device__ __forceinline__ float f32x2_hi(uint64_t v)
{
    return __uint_as_float(static_cast<uint32_t>(v >> 32));
}

__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi)
{
    return static_cast<uint64_t>(__float_as_uint(lo)) |
           (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are 128 bytes long and
// laid out with the 128-byte swizzle (what a TMA load with CU_TENSOR_MAP_SWIZZLE_128B and a
// 128-byte inner box writes): 8-row groups 1024 bytes apart. The tile must be 1024-aligned;
// stepping K inside the 128-byte row is done by advancing the start address.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address, 16-byte units
    d |= static_cast<uint64_t>(16u >> 4) << 16;                // leading-dim offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;              // stride between 8-row groups
    d |= static_cast<uint64_t>(1) << 46;                       // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;                       // swizzle mode: 128 bytes
    return d;
}

// Instruction descriptor of kind::f8f6f4 with A = B = E4M3, both K-major, D = FP32.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n)
{
    return (1u << 4)                                   // D format: FP32
           | (0u << 7)                                 // A format: E4M3
           | (0u << 10)                                // B format: E4M3
           | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

}  // namespace fp8bs
