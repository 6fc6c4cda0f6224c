// vp_umma.cuh -- tcgen05 (5th-generation tensor core) and tensor-TMA primitives
// for sm_103a, in inline PTX: TMEM allocation, shared-memory matrix and
// instruction descriptors, MMA issue and commit, TMEM loads, 2-D tiled TMA.
//
// Operand layouts: K-major bf16 tiles of 64 K-elements (128 bytes) per row, or
// MN-major tiles of 64 MN-elements per K-row, both written by TMA with the
// 128-byte swizzle in 8-row atoms of 1024 bytes.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "vp_tma.cuh"

namespace vp {

// --- TMEM -----------------------------------------------------------------
// Executed by one whole warp; the column base is written to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// --- descriptors ----------------------------------------------------------
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 1024-byte
// stride between 8-row groups (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t umma_desc_sw128(const void *smem) {
    const uint64_t addr = smem_u32(smem);
    uint64_t d = 0;
    d |= (addr >> 4) & 0x3FFFull;            // start address       [0, 14)
    d |= (uint64_t)1 << 16;                  // leading byte offset [16, 30) (unused when swizzled)
    d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset  [32, 46)
    d |= (uint64_t)1 << 46;                  // version             [46, 48)
    d |= (uint64_t)2 << 61;                  // layout: 128-byte swizzle [61, 64)
    return d;
}

// Shared-memory matrix descriptor of an MN-major operand, 128-byte swizzle:
// each atom is 8 K-rows of 64 consecutive MN elements (128 bytes per row,
// 1024 bytes per atom); atoms along MN are `mn_stride` bytes apart (LBO) and
// groups of 8 K-rows are 1024 bytes apart (SBO). A 16-deep K step advances the
// start address by 2048 bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128_mn(const void *smem, uint32_t mn_stride) {
    const uint64_t addr = smem_u32(smem);
    uint64_t d = 0;
    d |= (addr >> 4) & 0x3FFFull;                  // start address              [0, 14)
    d |= (uint64_t)((mn_stride >> 4) & 0x3FFF) << 16;   // leading byte offset: MN atoms [16, 30)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: K groups    [32, 46)
    d |= (uint64_t)1 << 46;                        // version                    [46, 48)
    d |= (uint64_t)2 << 61;                        // layout: 128-byte swizzle   [61, 64)
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator,
// shape M x N; each operand K-major unless its MN-major flag is set.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn = false, bool b_mn = false) {
    return (1u << 4)                        // accumulator format: f32   [4, 6)
           | (1u << 7)                      // A format: bf16            [7, 10)
           | (1u << 10)                     // B format: bf16            [10, 13)
           | ((a_mn ? 1u : 0u) << 15)       // A MN-major                [15]
           | ((b_mn ? 1u : 0u) << 16)       // B MN-major                [16]
           | ((uint32_t)(N >> 3) << 17)     // N / 8                     [17, 23)
           | ((uint32_t)(M >> 4) << 24);    // M / 16                    [24, 29)
}

// D[tmem] (+)= A[smem] * B[smem]^T, one M x N x 16 step, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Issue a load of 32 consecutive fp32 columns of this thread's TMEM lane (warp
// w reads lanes 32 (w % 4) .. 32 (w % 4) + 31); the registers hold the values
// only after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    tmem_ld32_issue(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive fp32 columns of this thread's TMEM lane, four loads behind one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
    uint32_t r[4][32];
#pragma unroll
    for (int k = 0; k < 4; ++k) tmem_ld32_issue(taddr + 32 * k, r[k]);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * k + i] = __uint_as_float(r[k][i]);
}

// --- 2-D tiled TMA --------------------------------------------------------
// Box at element coordinates (x = inner, y = row) into shared memory; the inner
// coordinate times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// The same load with an L2 eviction-priority policy (createpolicy) for the tile.
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy(int kind) {   // 1: evict_first, 2: evict_last, else evict_normal
    uint64_t p;
    if (kind == 1) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    else if (kind == 2) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    else asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// --- CTA pairs (clusters of two CTAs on two SMs, tcgen05 cta_group::2) ------
// (cluster rank, DSMEM addresses, cluster barriers and remote mbarrier
// arrivals are in vp_tma.cuh)
// TMA box into this CTA's shared memory, completing on the mbarrier at
// shared::cluster address `cluster_bar` (this CTA's or the pair's leader's).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t cluster_bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar), "l"(policy)
        : "memory");
}

// TMEM of a CTA pair: one warp of each CTA executes these together; the same
// columns are allocated in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// One 256 x N x 16 step of a CTA pair, issued by one thread of the leader CTA:
// rows 0-127 of A and D in the leader, rows 128-255 in the peer; each CTA holds
// N/2 rows of B; the descriptors name the same shared-memory offsets in both.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at this offset in both CTAs of the pair when the
// pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace vp
