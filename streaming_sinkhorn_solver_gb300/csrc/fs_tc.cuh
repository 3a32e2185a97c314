// sm_103a building blocks for the tensor-core path: mbarriers with
// time-bounded waits, 1-D bulk copies (cp.async.bulk), TMEM allocation and
// loads, UMMA shared-memory / instruction descriptors and tcgen05.mma.
//
// Operand tiles are stored in global memory already in the exact byte order
// the tensor core reads from shared memory (K-major, 128-byte swizzle), so a
// whole 16 KB chunk moves with one cp.async.bulk and needs no tensor map.
#pragma once

#include "fs_internal.cuh"
#include "fs_tc_kernels.cuh"

namespace fs {
namespace tc {

constexpr uint64_t kTimeoutNs = 2000000000ull;   // any single wait: 2 s
// Suspend-time hint of every try_wait: a waiting thread sleeps until the phase
// completes (or this long) instead of returning at once and spinning, which
// took issue slots from the producer and MMA threads on the same SM
// sub-partition (measured on sm_103a).
constexpr uint32_t kSuspendHintNs = 1000000u;

// byte offset of element (r, e) of a 128 x 64 chunk in the K-major
// 128-byte-swizzled layout: row r occupies bytes [128 r, 128 r + 128); its
// 16-byte unit u = e / 8 is stored at unit u ^ (r mod 8).
__host__ __device__ __forceinline__ uint32_t swz_offset(int r, int e) {
    const int u = e >> 3;
    return (uint32_t)(r * 128 + (((u ^ (r & 7)) << 4)) + ((e & 7) << 1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// --- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
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

// Wait for the phase of parity `parity` to complete.  Gives up after
// kTimeoutNs, ORs `code` into the device error word and returns false.
//
// The whole spin (try_wait, then %globaltimer against the deadline) is one
// inline-PTX block with brace-scoped labels: with the retry loop written in
// C++ instead, the thread issuing tcgen05.mma ran its MMA stream at about a
// quarter of the tensor rate (measured on sm_103a), with the loop in PTX it
// runs at full rate.
#define FS_MBAR_WAIT_PTX(SEM)                                                     \
    "{\n\t.reg .pred p;\n\t.reg .u64 t0, t;\n\t"                                  \
    "mbarrier.try_wait.parity" SEM ".shared::cta.b64 p, [%1], %2, %4;\n\t"        \
    "@p bra.uni LAB_DONE;\n\t"                                                    \
    "mov.u64 t0, %%globaltimer;\n"                                                \
    "LAB_WAIT:\n\t"                                                               \
    "mbarrier.try_wait.parity" SEM ".shared::cta.b64 p, [%1], %2, %4;\n\t"        \
    "@p bra.uni LAB_DONE;\n\t"                                                    \
    "mov.u64 t, %%globaltimer;\n\t"                                               \
    "sub.u64 t, t, t0;\n\t"                                                       \
    "setp.lt.u64 p, t, %3;\n\t"                                                   \
    "@p bra.uni LAB_WAIT;\n\t"                                                    \
    "selp.u32 %0, 0, 0, p;\n\t"                                                   \
    "bra.uni LAB_END;\n"                                                          \
    "LAB_DONE:\n\t"                                                               \
    "mov.u32 %0, 1;\n"                                                            \
    "LAB_END:\n\t}"

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                          uint32_t code) {
    uint32_t ok;
    asm volatile(FS_MBAR_WAIT_PTX("")
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity), "l"(kTimeoutNs), "r"(kSuspendHintNs)
                 : "memory");
    if (!ok) atomicOr(err, code);
    return ok != 0;
}

// --- bulk copy global -> shared (async proxy, completes on an mbarrier) -------

__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// --- tcgen05 ----------------------------------------------------------------

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// whole warp: allocate `ncols` TMEM columns, address written to *slot
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major; one elected thread issues.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive once on `bar` when every tcgen05.mma issued so far by this thread completes
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive columns of 32-bit data: thread t gets lane t
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]),
          "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),
          "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]),
          "=f"(v[31])
        : "r"(taddr));
}

// 16 lanes x 32 columns (16x256b shape, 4 repetitions): thread t gets, for
// repetition i, columns 8i + 2(t%4) + {0, 1} of lane t/4 (v[4i], v[4i+1]) and
// of lane t/4 + 8 (v[4i+2], v[4i+3]); the lane offset comes with taddr
__device__ __forceinline__ void tmem_ld16x32(uint32_t taddr, float (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
        : "r"(taddr));
}

// 16 lanes x 128 columns (16x256b shape, 16 repetitions): the layout of
// tmem_ld16x32 with i = 0..15
__device__ __forceinline__ void tmem_ld16x128(uint32_t taddr, float* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),
          "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),
          "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]),
          "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),
          "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]),
          "=f"(v[31]), "=f"(v[32]), "=f"(v[33]), "=f"(v[34]), "=f"(v[35]), "=f"(v[36]),
          "=f"(v[37]), "=f"(v[38]), "=f"(v[39]), "=f"(v[40]), "=f"(v[41]), "=f"(v[42]),
          "=f"(v[43]), "=f"(v[44]), "=f"(v[45]), "=f"(v[46]), "=f"(v[47]), "=f"(v[48]),
          "=f"(v[49]), "=f"(v[50]), "=f"(v[51]), "=f"(v[52]), "=f"(v[53]), "=f"(v[54]),
          "=f"(v[55]), "=f"(v[56]), "=f"(v[57]), "=f"(v[58]), "=f"(v[59]), "=f"(v[60]),
          "=f"(v[61]), "=f"(v[62]), "=f"(v[63])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Order later uses of v after a tcgen05.wait::ld: the empty asm statements
// (volatile, so they stay after the wait) redefine every register of v.
template <int N>
__device__ __forceinline__ void tmem_reg_fence(float (&v)[N]) {
    static_assert(N % 8 == 0, "multiples of 8 registers");
#pragma unroll
    for (int i = 0; i < N; i += 8)
        asm volatile("" : "+f"(v[i]), "+f"(v[i + 1]), "+f"(v[i + 2]), "+f"(v[i + 3]), "+f"(v[i + 4]),
                     "+f"(v[i + 5]), "+f"(v[i + 6]), "+f"(v[i + 7]));
}

// warp: the same value x into 8 consecutive columns of the warp's 32 lanes
// (a store names one source register per column, so the 32-column form keeps
// 32 registers live where this one keeps 8)
__device__ __forceinline__ void tmem_fill8(uint32_t taddr, float x) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"r"(
                     taddr),
                 "f"(x)
                 : "memory");
}
// warp: 8 registers into 8 consecutive columns of the warp's 32 lanes
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                     taddr),
                 "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
                 "f"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// --- CTA pairs (cluster of 2, tcgen05 cta_group::2) ---------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// address of the same shared-memory object in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
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

// bounded wait on a barrier that also receives arrivals from the peer CTA
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* err,
                                                  uint32_t code) {
    uint32_t ok;
    asm volatile(FS_MBAR_WAIT_PTX(".acquire.cluster")
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity), "l"(kTimeoutNs), "r"(kSuspendHintNs)
                 : "memory");
    if (!ok) atomicOr(err, code);
    return ok != 0;
}

// all threads of both CTAs
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// TMA copy of one 128 x 64 fp16 chunk (a 2-D box {64, 128} at x = 0, y = row)
// into this CTA's shared memory, completing its bytes on an mbarrier of
// either CTA of the pair (`bar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_chunk_pair(void* dst_smem, const void* tmap, uint32_t row,
                                               uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst_smem)),
        "l"(tmap), "r"(0), "r"(row), "r"(bar_cluster)
        : "memory");
}

// L2 eviction-priority policies for the bulk tensor copies' cache hints
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// tma_chunk_pair with an L2 cache policy
__device__ __forceinline__ void tma_chunk_pair_hint(void* dst_smem, const void* tmap, uint32_t row,
                                                    uint32_t bar_cluster, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst_smem)),
        "l"(tmap), "r"(0), "r"(row), "r"(bar_cluster), "l"(policy)
        : "memory");
}

// one warp in each CTA of the pair, collectively
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D (M = 256 over the pair) (+)= A * B^T; issued by one thread of the even CTA.
// Each CTA supplies its 128 rows of A and half of B's N rows, at the same
// shared-memory offsets; each CTA's TMEM receives its 128 rows of D.
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive once on `bar` (same offset) in every CTA of `mask` when all MMAs
// issued so far by this thread complete
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core
// groups 1024 bytes apart (SBO), descriptor version 1, base offset 0 (tiles
// are 1024-byte aligned).  The start address may be advanced in 16-byte
// units inside a swizzled row to step through K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)1 << 16;                     // leading byte offset (unused here), 16 B
    d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset
    d |= (uint64_t)1 << 46;                     // version
    d |= (uint64_t)2 << 61;                     // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: A and B fp16, D fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4)                      // D format: f32
           | (0u << 7)                    // A format: f16
           | (0u << 10)                   // B format: f16
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

}  // namespace tc
}  // namespace fs
