// ptx.cuh -- thin inline-PTX wrappers for sm_103a: cluster, mbarrier, TMA
// (tiled and gather4), tcgen05 (TMEM alloc, MMA, commit, ld; one CTA or a CTA
// pair) and a bounded wait.
//
// Every wait in this library is bounded: a wait that has not completed after
// kWaitLimitNs of %globaltimer time records MOE_DEV_ERR_TIMEOUT in the
// device error word, raises the CTA's abort flag and returns false, so the
// kernel can drain what it issued and exit instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Device error codes (bit flags OR-ed into the workspace error word).
enum : uint32_t {
    MOE_DEV_ERR_BAD_EXPERT = 1u << 0,   // an expert id outside [0, E)
    MOE_DEV_ERR_TIMEOUT = 1u << 1,      // a bounded wait ran out
    MOE_DEV_ERR_BOUNDS = 1u << 2,       // an index outside its buffer (skipped)
};

constexpr unsigned long long kWaitLimitNs = 4000000000ull;   // 4 s

__device__ __forceinline__ void report_error(uint32_t* err, uint32_t code)
{
    if (err) atomicOr(err, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t elect_one_sync()
{
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.b32 %0, 1, 0, P;\n\t}\n"
        : "=r"(pred));
    return pred;
}

// -------------------------------------------------------------- cluster --

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the variable at shared::cta address `addr`
// in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Every thread of every CTA of the cluster (all threads must call it).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

// Sleeps about `ns` nanoseconds (bounded by %globaltimer).
__device__ __forceinline__ void sleep_ns(unsigned long long ns)
{
    const unsigned long long t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) __nanosleep(1000);
}

// ------------------------------------------- programmatic dependent launch --

// A kernel launched with programmatic stream serialization may start while
// the kernel before it in the stream is still running. pdl_wait() blocks the
// calling thread until that grid has completed and its memory operations are
// visible; every thread calls it before its first global memory access. (A
// no-op for a kernel launched without the attribute.)
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream be scheduled before this one exits (it
// still waits in its own pdl_wait() for this grid to complete).
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}\n" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}\n" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

// Arrive on a barrier of another CTA of the cluster (`bar` from mapa_shared),
// releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// CLUSTER: acquire at cluster scope (the phase was completed by arrivals from
// another CTA of the cluster).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if constexpr (CLUSTER)
        asm volatile(
            "{\n\t.reg .pred P;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 P, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, P;\n\t}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred P;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, P;\n\t}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with parity `parity`. Returns false (after
// recording a timeout and raising *abort) if it does not complete within
// kWaitLimitNs, or if another role of the CTA has already raised *abort.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* err)
{
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                report_error(err, MOE_DEV_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait used only while draining after an abort: no abort check.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity)
{
    unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Waits until *ctr >= target (acquire, GPU scope). Returns false (after
// recording a timeout and raising *abort) if that takes longer than limit_ns
// of %globaltimer time or another role has aborted.
__device__ __forceinline__ bool wait_count(const int32_t* ctr, int32_t target, volatile int* abort,
                                           uint32_t* err, unsigned long long limit_ns = kWaitLimitNs)
{
    auto load = [&]() {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        return v;
    };
    if (load() >= target) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(128);
        if (load() >= target) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort = 1;
                report_error(err, MOE_DEV_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ TMA --

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// 2D tiled load of one box at (c0 = inner coordinate, c1 = outer).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Contiguous copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global memory into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// The same load issued by either CTA of a CTA pair: the box lands in this
// CTA's shared memory and its bytes complete on `bar`, a shared::cluster
// address that may be the pair's leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                                 uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Gather of four rows r0..r3 (box one row high) starting at column c0; the
// rows land one after another at dst.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap, int32_t c0, int32_t r0,
                                            int32_t r1, int32_t r2, int32_t r3, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}

// -------------------------------------------------------------- tcgen05 --

// CG = 1: this CTA's tensor core and TMEM. CG = 2: a CTA pair (cluster ranks
// 0 and 1); every tcgen05 instruction of a kernel uses one CG, and a pair's
// alloc / relinquish / dealloc are issued by one warp in each of the two CTAs.
template <int CG = 1>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
}

template <int CG = 1>
__device__ __forceinline__ void tmem_relinquish()
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int CG = 1>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
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

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, f32 out).
// CG = 2 (issued by the pair's rank-0 CTA): A is 2 x 128 rows, one half in
// each CTA's shared memory at the same address; B's N columns are split the
// same way (rank 0 holds the first N/2); each CTA's TMEM receives its 128 rows.
template <int CG = 1>
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate)
{
    if constexpr (CG == 2)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is
// done. CG = 2: on the barrier at the same address in both CTAs of the pair.
template <int CG = 1>
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    if constexpr (CG == 2) {
        const uint16_t both = 3;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
            " [%0], %1;" ::"r"(bar),
            "h"(both)
            : "memory");
    } else {
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
            : "memory");
    }
}

// CG = 2 form of a commit that arrives on this CTA's barrier only.
__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM cells: thread i gets lane (base + i),
// columns col .. col+31 in v[0..31].
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

// 32-byte store of 8 words (a whole L2 sector). The address must be 32-byte
// aligned.
__device__ __forceinline__ void st_global_v8(void* ptr, uint32_t w0, uint32_t w1, uint32_t w2,
                                             uint32_t w3, uint32_t w4, uint32_t w5, uint32_t w6,
                                             uint32_t w7)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w0),
                 "r"(w1), "r"(w2), "r"(w3), "r"(w4), "r"(w5), "r"(w6), "r"(w7)
                 : "memory");
}

// ------------------------------------------------------- UMMA descriptors --

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1 on sm_100 family)
//   bits 49-51 base offset (0: tiles are 1024-byte aligned)
//   bits 61-63 layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// The same for a K-major operand in 64-byte-swizzled rows (layout type 4):
// 8-row groups sbo bytes apart (512 for dense 64-byte rows).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)4 << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A and B, f32 accumulator.
//   bits 4-5 D format (1 = f32); 7-9 A format (1 = bf16); 10-12 B format
//   (1 = bf16); 15 A major (0 = K); 16 B major (1 = MN); 17-22 N >> 3;
//   24-28 M >> 4 (M = 256: a CTA pair, 128 rows in each CTA's TMEM).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn_major,
                                                      bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace moe
