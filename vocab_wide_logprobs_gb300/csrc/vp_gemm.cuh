// vp_gemm.cuh -- the persistent tcgen05 GEMM shared by the fused linear ops
// (linear logp, entropy, KL and JSD): single-CTA and CTA-pair kernels, the
// two-model dual form, their operand tensor maps, tile order and L2 hints, and
// the gradient GEMMs of the chunked backward.
//
// Each translation unit that includes this header gets its own copy of the
// kernels' fault word (g_linear_fault); read_linear_fault reads every copy.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "vp_device.cuh"
#include "vp_launch.h"
#include "vp_umma.cuh"

namespace vp {

constexpr int kLBM = 128, kLBN = 256, kLBK = 64;
constexpr int kLStages = 4;
constexpr int kLAStage = kLBM * kLBK * 2;          // 16 KB
constexpr int kLBStage = kLBN * kLBK * 2;          // 32 KB
constexpr int kLStageBytes = kLAStage + kLBStage;  // 48 KB
constexpr int kLSmemBytes = kLStages * kLStageBytes + 1024;  // + alignment slack
constexpr int kLThreads = 192;                     // TMA warp, MMA warp, 4 epilogue warps
// Columns per epilogue thread in the dual form (one half of a 256-column tile).
constexpr int kDualEpiCols = 128;
constexpr uint32_t kLTmemCols = 2 * kLBN;          // two accumulators

// Set when a bounded wait of the linear kernels gave up.
static __device__ uint32_t g_linear_fault;   // one per translation unit

struct LinearBars {
    uint64_t full[kLStages], empty[kLStages], acc_full[2], acc_empty[2];
    uint32_t tmem_base;
};

// ---------------------------------------------------------------------------
// Persistent tcgen05 GEMM C[M, Nn] = A[M, K] . B[Nn, K]^T (bf16 operands through
// 2-D tensor maps, fp32 accumulation in TMEM) with a pluggable epilogue.
// Operand layouts: K-major (kAMn / kBMn false: a row of the operand's tensor map
// holds K-consecutive elements; one box of 64 x rows per stage) or MN-major
// (true: the map's rows run along K and hold MN-consecutive elements; 64 x 64
// boxes, 8 KB apart in shared memory), so that a transposed operand is read in
// place. Tiles run in m-groups (tile_coords) with L2 eviction hints per operand.
// The epilogue functor is called by each epilogue thread for its accumulator
// row: epi(row, col0, ncol, taddr), taddr = the TMEM address of the row's 256
// columns. TMEM loads (tmem_ld32) are warp-collective, so every lane runs every
// load (rows past M included) and only the global accesses are guarded.
// ---------------------------------------------------------------------------
constexpr uint32_t kLMnAtomBytes = 64 * kLBK * 2;   // one 64 (MN) x 64 (K) box: 8 KB

// Tile order: groups of group_m m-blocks; within a group, m-blocks vary fastest,
// then n-blocks. group_m >= n_mb is plain N-major order (consecutive CTAs share
// one B tile, and all of A stays in L2: right when A is small); a small group_m
// keeps the concurrent tiles on a few A and B tiles each (right when both
// operands are large and stream along a long K).
__device__ __forceinline__ void tile_coords(int64_t tile, int n_mb, int n_nb, int group_m, int &mb, int &nb) {
    const int64_t per_group = (int64_t)group_m * n_nb;
    const int g = (int)(tile / per_group);
    const int first = g * group_m;
    const int gm = min(group_m, n_mb - first);
    const int w = (int)(tile - (int64_t)g * per_group);
    mb = first + w % gm;
    nb = w / gm;
}

template <class Epi, bool kAMn = false, bool kBMn = false, bool kChain = false>
__global__ void __launch_bounds__(kLThreads, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_a2, const __grid_constant__ CUtensorMap tm_b2, int M, int Nn,
                 int K, int group_m, int l2hints, const Epi epi) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ LinearBars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_mb = (M + kLBM - 1) / kLBM, n_nb = (Nn + kLBN - 1) / kLBN;
    const int64_t n_tiles = (int64_t)n_mb * n_nb;
    const int n_k = (K + kLBK - 1) / kLBK;
    const int n_kt = kChain ? 2 * n_k : n_k;   // a chained second product (A2 . B2^T, K deep) follows

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.acc_full[b], 1);
            mbar_init(&bars.acc_empty[b], kLThreads - 64);   // every epilogue thread
        }
        fence_mbar_init();
        prefetch_tensormap(&tm_a);
        prefetch_tensormap(&tm_b);
    }
    if (warp == 1) tmem_alloc(&bars.tmem_base, kLTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            // L2 eviction priority of the A and B tiles (bits 0-1 and 2-3 of l2hints)
            const uint64_t pol_a = l2_policy(l2hints & 3), pol_b = l2_policy((l2hints >> 2) & 3);
            uint32_t it = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                int mb, nb;
                tile_coords(tile, n_mb, n_nb, group_m, mb, nb);
                for (int kb = 0; kb < n_kt; ++kb, ++it) {
                    const uint32_t st = it % kLStages, use = it / kLStages;
                    if (use > 0 && !mbar_wait(&bars.empty[st], (use - 1) & 1)) { ok = false; break; }
                    uint8_t *a = smem + st * kLStageBytes;
                    mbar_arrive_expect_tx(&bars.full[st], kLStageBytes);
                    const bool second = kChain && kb >= n_k;
                    const CUtensorMap *ma = second ? &tm_a2 : &tm_a, *mbm = second ? &tm_b2 : &tm_b;
                    const int kc = (second ? kb - n_k : kb) * kLBK;
                    if (kAMn) {
#pragma unroll
                        for (int i = 0; i < kLBM / 64; ++i)
                            tma_load_2d_hint(a + i * kLMnAtomBytes, ma, mb * kLBM + 64 * i, kc, &bars.full[st],
                                             pol_a);
                    } else {
                        tma_load_2d_hint(a, ma, kc, mb * kLBM, &bars.full[st], pol_a);
                    }
                    if (kBMn) {
#pragma unroll
                        for (int i = 0; i < kLBN / 64; ++i)
                            tma_load_2d_hint(a + kLAStage + i * kLMnAtomBytes, mbm, nb * kLBN + 64 * i, kc,
                                             &bars.full[st], pol_b);
                    } else {
                        tma_load_2d_hint(a + kLAStage, mbm, kc, nb * kLBN, &bars.full[st], pol_b);
                    }
                }
            }
            if (!ok) atomicOr(&g_linear_fault, 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(kLBM, kLBN, kAMn, kBMn);
            uint32_t it = 0, j = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++j) {
                const uint32_t buf = j & 1, use_b = j >> 1;
                if (use_b > 0 && !mbar_wait(&bars.acc_empty[buf], (use_b - 1) & 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + buf * kLBN;
                for (int kb = 0; kb < n_kt; ++kb, ++it) {
                    const uint32_t st = it % kLStages;
                    if (!mbar_wait(&bars.full[st], (it / kLStages) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint8_t *a = smem + st * kLStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kLBK / 16; ++kk) {
                        // a 16-deep K step: 32 bytes along a K-major row, two 8-row groups MN-major
                        const uint64_t da = kAMn ? umma_desc_sw128_mn(a + kk * 2048, kLMnAtomBytes)
                                                 : umma_desc_sw128(a + kk * 32);
                        const uint64_t db = kBMn ? umma_desc_sw128_mn(a + kLAStage + kk * 2048, kLMnAtomBytes)
                                                 : umma_desc_sw128(a + kLAStage + kk * 32);
                        umma_bf16(d, da, db, idesc, (kb | kk) != 0);
                    }
                    umma_commit(&bars.empty[st]);       // frees the stage once these MMAs are done
                }
                umma_commit(&bars.acc_full[buf]);       // the accumulator is complete
            }
            if (!ok) atomicOr(&g_linear_fault, 2u);
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const int r_in = q * 32 + lane;
        uint32_t j = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++j) {
            int mb, nb;
            tile_coords(tile, n_mb, n_nb, group_m, mb, nb);
            const uint32_t buf = j & 1;
            if (ok && !mbar_wait(&bars.acc_full[buf], (j >> 1) & 1)) {
                ok = false;
                atomicOr(&g_linear_fault, 4u);
            }
            tc_fence_after();
            // tcgen05.ld is warp-collective: the whole warp calls the epilogue or
            // none of it does, and epilogues guard only their global accesses
            if (__all_sync(0xffffffffu, ok))
                epi(mb * kLBM + r_in, nb * kLBN, min(kLBN, Nn - nb * kLBN),
                    tmem + buf * kLBN + ((uint32_t)(q * 32) << 16));
            tc_fence_before();
            mbar_arrive(&bars.acc_empty[buf]);           // the MMA warp may reuse the accumulator
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kLTmemCols);
}

// ---------------------------------------------------------------------------
// The same GEMM on CTA pairs (clusters of two CTAs on two SMs, tcgen05
// cta_group::2): each pair computes a 256 x 256 tile. CTA r of the pair holds
// rows 128 r .. 128 r + 127 of the A tile and of the accumulator, and rows
// 128 r .. 128 r + 127 of the B tile, so a stage is 32 KB per CTA instead of
// 48 KB and six stages fit (twice the bytes in flight per FLOP of the
// single-CTA form). The leader's (rank 0) TMA thread posts the stage's byte
// count and both CTAs' TMA loads complete on the leader's "full" barrier; one
// thread of the leader issues the pair MMAs and commits each stage to the
// "empty" barriers and each tile to the "acc_full" barriers of both CTAs; the
// epilogue warps of both CTAs read their own TMEM rows and arrive on the
// leader's "acc_empty" barrier. Every wait is bounded; every thread of both
// CTAs reaches the final cluster barrier.
// Dual form (kDual, K-major operands only): each tile also computes a second
// product C2 = A2 . B2^T (K2 deep) of the same shape into the other 256 TMEM
// columns, so that an epilogue sees the same logits tile of two models at
// once. The two products fill TMEM, so instead of two accumulator sets each
// product has its own barriers (acc_full[p], acc_empty[p]): the epilogue
// copies its columns of the first product into registers as soon as that
// product is done and frees them, so the next tile's first product queues
// behind this tile's second and the tensor pipe does not drain between tiles;
// the epilogue then works through the second product while the next first
// product runs. The epilogue functor is called as epi(row, col0, ncol, x, tb),
// x the row's 128 columns (one half of the tile) of the first product and tb
// the TMEM address of the same columns of the second. The dual kernel has 12
// warps: warp 0 TMA, warp 1 MMA, warps 2-3 idle, warps 4-11 the epilogue (two
// per TMEM lane quarter, one 128-column half each). An epilogue thread holds
// 128 fp32 values, so the epilogue warpgroups take registers from the first:
// of the 168 a thread is launched with, setmaxnreg leaves 56 to warpgroup 0
// and gives 224 to warpgroups 1-2 (4 x 56 + 8 x 224 = 12 x 168); the launcher
// checks the 168 before the first launch.
// ---------------------------------------------------------------------------
constexpr int kPStages = 6;
constexpr int kPBHalf = kLBN / 2;                       // rows of the B tile per CTA
constexpr int kPAStage = kLBM * kLBK * 2;               // 16 KB
constexpr int kPBStage = kPBHalf * kLBK * 2;            // 16 KB
constexpr int kPStageBytes = kPAStage + kPBStage;       // 32 KB
constexpr int kPSmemBytes = kPStages * kPStageBytes + 1024;

struct PairBars {
    uint64_t full[kPStages], empty[kPStages], acc_full[2], acc_empty[2];
    uint32_t tmem_base;
};

constexpr int kPairDualRegsLaunch = 168, kPairDualRegsLow = 56, kPairDualRegsHigh = 224;
static_assert(4 * kPairDualRegsLow + 8 * kPairDualRegsHigh == 12 * kPairDualRegsLaunch,
              "the epilogue warpgroups take exactly what warpgroup 0 gives up");
__host__ __device__ constexpr int pair_threads(bool dual) { return dual ? 12 * 32 : kLThreads; }
__host__ __device__ constexpr int pair_epi_first_warp(bool dual) { return dual ? 4 : 2; }

template <class Epi, bool kAMn = false, bool kBMn = false, bool kDual = false, bool kChain = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(kDual), 1)
umma_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_a2, const __grid_constant__ CUtensorMap tm_b2, int M,
                      int Nn, int K, int K2, int group_m, int l2hints, const Epi epi) {
    static_assert(!kDual || (!kAMn && !kBMn), "the dual form takes K-major operands");
    static_assert(!(kDual && kChain), "one second product at a time");
    extern __shared__ uint8_t smem_raw[];
    __shared__ PairBars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int n_mp = (M + 2 * kLBM - 1) / (2 * kLBM), n_nb = (Nn + kLBN - 1) / kLBN;
    const int64_t n_tiles = (int64_t)n_mp * n_nb;
    const int n_k = (K + kLBK - 1) / kLBK;
    const int n_k2 = (kDual || kChain) ? (K2 + kLBK - 1) / kLBK : 0;   // k-blocks of the second product
    const int64_t pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
    constexpr int kEpiThreads = pair_threads(kDual) - 32 * pair_epi_first_warp(kDual);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.acc_full[b], 1);
            mbar_init(&bars.acc_empty[b], 2 * kEpiThreads);   // the epilogue threads of both CTAs
        }
        fence_mbar_init();
        prefetch_tensormap(&tm_a);
        prefetch_tensormap(&tm_b);
        if (kDual) {
            prefetch_tensormap(&tm_a2);
            prefetch_tensormap(&tm_b2);
        }
    }
    if (warp == 1) tmem_alloc_pair(&bars.tmem_base, kLTmemCols);
    tc_fence_before();
    cluster_sync();                                      // barriers and TMEM ready in both CTAs
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp < pair_epi_first_warp(kDual)) {
    // warpgroup 0 in the dual form (TMA, MMA and two idle warps)
    if constexpr (kDual) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPairDualRegsLow));
    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0) {
            const uint64_t pol_a = l2_policy(l2hints & 3), pol_b = l2_policy((l2hints >> 2) & 3);
            uint32_t it = 0;
            bool ok = true;
            for (int64_t tile = pair; tile < n_tiles && ok; tile += n_pairs) {
                int mp, nb;
                tile_coords(tile, n_mp, n_nb, group_m, mp, nb);
                const int mb = 2 * mp + (int)rank;
                const int nrow = nb * kLBN + (int)rank * kPBHalf;
                for (int kb = 0; kb < n_k + n_k2; ++kb, ++it) {
                    const uint32_t st = it % kPStages, use = it / kPStages;
                    if (use > 0 && !mbar_wait_cluster(&bars.empty[st], (use - 1) & 1)) { ok = false; break; }
                    uint8_t *a = smem + st * kPStageBytes;
                    const uint32_t fb = cluster_addr(&bars.full[st], 0);
                    if (rank == 0) mbar_arrive_expect_tx(&bars.full[st], 2 * kPStageBytes);
                    // k-blocks past n_k belong to the second product (its own maps)
                    const bool second = (kDual || kChain) && kb >= n_k;
                    const CUtensorMap *ma = second ? &tm_a2 : &tm_a, *mbm = second ? &tm_b2 : &tm_b;
                    const int kc = (second ? kb - n_k : kb) * kLBK;
                    if (kAMn) {
#pragma unroll
                        for (int i = 0; i < kLBM / 64; ++i)
                            tma_load_2d_pair(a + i * kLMnAtomBytes, ma, mb * kLBM + 64 * i, kc, fb, pol_a);
                    } else {
                        tma_load_2d_pair(a, ma, kc, mb * kLBM, fb, pol_a);
                    }
                    if (kBMn) {
#pragma unroll
                        for (int i = 0; i < kPBHalf / 64; ++i)
                            tma_load_2d_pair(a + kPAStage + i * kLMnAtomBytes, mbm, nrow + 64 * i, kc, fb, pol_b);
                    } else {
                        tma_load_2d_pair(a + kPAStage, mbm, kc, nrow, fb, pol_b);
                    }
                }
            }
            if (!ok) atomicOr(&g_linear_fault, 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader only) ----------------
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(2 * kLBM, kLBN, kAMn, kBMn);
            uint32_t it = 0, j = 0;
            bool ok = true;
            for (int64_t tile = pair; tile < n_tiles && ok; tile += n_pairs, ++j) {
                // product p of the dual form: accumulator columns p * 256 and
                // barriers acc_full[p] / acc_empty[p]; otherwise buffer j & 1
                for (int p = 0; p < (kDual ? 2 : 1) && ok; ++p) {
                    const uint32_t buf = kDual ? p : j & 1, use_b = kDual ? j : j >> 1;
                    if (use_b > 0 && !mbar_wait_cluster(&bars.acc_empty[buf], (use_b - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d = tmem + buf * kLBN;
                    // a chained second product accumulates into the same accumulator
                    const int nkb = kChain ? n_k + n_k2 : p ? n_k2 : n_k;
                    for (int kb = 0; kb < nkb; ++kb, ++it) {
                        const uint32_t st = it % kPStages;
                        if (!mbar_wait(&bars.full[st], (it / kPStages) & 1)) { ok = false; break; }
                        tc_fence_after();
                        const uint8_t *a = smem + st * kPStageBytes;
#pragma unroll
                        for (int kk = 0; kk < kLBK / 16; ++kk) {
                            const uint64_t da = kAMn ? umma_desc_sw128_mn(a + kk * 2048, kLMnAtomBytes)
                                                     : umma_desc_sw128(a + kk * 32);
                            const uint64_t db = kBMn ? umma_desc_sw128_mn(a + kPAStage + kk * 2048, kLMnAtomBytes)
                                                     : umma_desc_sw128(a + kPAStage + kk * 32);
                            umma_bf16_pair(d, da, db, idesc, (kb | kk) != 0);
                        }
                        umma_commit_pair(&bars.empty[st]);   // frees the stage in both CTAs
                    }
                    umma_commit_pair(&bars.acc_full[buf]);   // the accumulator (product) is complete
                }
            }
            if (!ok) atomicOr(&g_linear_fault, 2u);
        }
    }
    } else {
        // ---------------- epilogue (both CTAs) ----------------
        if constexpr (kDual) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPairDualRegsHigh));
        const int q = warp & 3;
        const int r_in = q * 32 + lane;
        const int half = kDual ? (warp - 4) >> 2 : 0;   // dual form: the warp's 128-column half
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        uint32_t j = 0;
        bool ok = true;
        for (int64_t tile = pair; tile < n_tiles; tile += n_pairs, ++j) {
            int mp, nb;
            tile_coords(tile, n_mp, n_nb, group_m, mp, nb);
            const int mb = 2 * mp + (int)rank;
            if constexpr (kDual) {
                const int c0 = nb * kLBN + half * kDualEpiCols;
                const int ncol = min(kDualEpiCols, Nn - c0);
                if (ok && !mbar_wait_cluster(&bars.acc_full[0], j & 1)) {
                    ok = false;
                    atomicOr(&g_linear_fault, 4u);
                }
                tc_fence_after();
                const uint32_t ta = tmem + half * kDualEpiCols + lanes;
                float x[kDualEpiCols];                   // the first product, out of TMEM
                if (__all_sync(0xffffffffu, ok) && ncol > 0) tmem_ld128(ta, x);
                tc_fence_before();
                mbar_arrive_cluster(cluster_addr(&bars.acc_empty[0], 0));   // the next first product may start
                if (ok && !mbar_wait_cluster(&bars.acc_full[1], j & 1)) {
                    ok = false;
                    atomicOr(&g_linear_fault, 4u);
                }
                tc_fence_after();
                if (__all_sync(0xffffffffu, ok) && ncol > 0) epi(mb * kLBM + r_in, c0, ncol, x, ta + kLBN);
                tc_fence_before();
                mbar_arrive_cluster(cluster_addr(&bars.acc_empty[1], 0));
            } else {
                const uint32_t buf = j & 1;
                if (ok && !mbar_wait_cluster(&bars.acc_full[buf], (j >> 1) & 1)) {
                    ok = false;
                    atomicOr(&g_linear_fault, 4u);
                }
                tc_fence_after();
                if (__all_sync(0xffffffffu, ok))
                    epi(mb * kLBM + r_in, nb * kLBN, min(kLBN, Nn - nb * kLBN), tmem + buf * kLBN + lanes);
                tc_fence_before();
                mbar_arrive_cluster(cluster_addr(&bars.acc_empty[buf], 0));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                      // no arrival or copy still targets either CTA
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kLTmemCols);
}

// dz of the backward K1 epilogues: n (a multiple of 8) consecutive values as
// bf16, rounded to nearest even, at dst (16-byte stores). With lo_off != 0 the
// remainders x - bf16(x) (exact in fp32), rounded to bf16, go to dst + lo_off,
// the dz_lo buffer of the chained gradient GEMMs.
template <int n>
__device__ __forceinline__ void store_dz(__nv_bfloat16 *dst, const float (&d)[n], int64_t lo_off) {
    static_assert(n % 8 == 0, "whole 16-byte vectors");
#pragma unroll
    for (int k = 0; k < n / 8; ++k) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x0 = d[8 * k + 2 * i], x1 = d[8 * k + 2 * i + 1];
            const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
            hi[i] = *reinterpret_cast<const uint32_t *>(&h);
            const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
            lo[i] = *reinterpret_cast<const uint32_t *>(&l);
        }
        reinterpret_cast<uint4 *>(dst)[k] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (lo_off) reinterpret_cast<uint4 *>(dst + lo_off)[k] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Backward K2 epilogue: acc[row][col] (+)= tile, fp32 (pitch ld).
// On the last chunk (out non-null) the sum is rounded to bf16 and written to
// out (same pitch) instead of acc: the dhidden output, with no separate pass.
struct AccEpi {
    int M, ld;
    bool first;
    float *acc;
    __nv_bfloat16 *out;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < M;
        const int64_t off = (int64_t)(valid ? row : 0) * ld + col0;
        float *dst = acc + off;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            if (!valid || c * 32 >= ncol) continue;
            float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
            uint32_t packed[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float4 o = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                if (!first) {
                    const float4 a = d4[k];
                    o.x += a.x; o.y += a.y; o.z += a.z; o.w += a.w;
                }
                if (out) {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
                    packed[2 * k] = *reinterpret_cast<uint32_t *>(&lo);
                    packed[2 * k + 1] = *reinterpret_cast<uint32_t *>(&hi);
                } else {
                    d4[k] = o;
                }
            }
            if (out) {
                uint4 *o4 = reinterpret_cast<uint4 *>(out + off + c * 32);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o4[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
            }
        }
    }
};

// Backward K3 epilogue: out[row0 + row][col] = bf16(tile) (pitch ld), rows < M.
struct StoreBf16Epi {
    int M, ld;
    int64_t row0;
    __nv_bfloat16 *out;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < M;
        __nv_bfloat16 *dst = out + (row0 + (valid ? row : 0)) * (int64_t)ld + col0;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            if (!valid || c * 32 >= ncol) continue;
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                packed[i] = *reinterpret_cast<uint32_t *>(&b);
            }
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                d4[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
        }
    }
};

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load();
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// Row-major bf16 matrix of `rows` rows of `cols` valid elements, `pitch`
// elements apart; boxes of box_rows x 64 with the 128-byte swizzle. Boxes past
// the extents read as zeros.
static bool make_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, int64_t pitch, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
    cuuint32_t box[2] = {(cuuint32_t)kLBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major operand map: `rows` along K, `cols` (the operand's M or N) consecutive,
// boxes of 64 x 64.
static bool make_map_mn(CUtensorMap *map, const void *ptr, int64_t rows, int64_t cols, int64_t pitch) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)kLBK};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Epi, bool kAMn = false, bool kBMn = false, bool kChain = false>
static cudaError_t launch_gemm_impl(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ta2,
                                    const CUtensorMap &tb2, int M, int Nn, int K, int group_m, int l2hints,
                                    const Epi &epi, cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(attr_done.load() & (1ull << (dev & 63)))) {
        cudaError_t e = cudaFuncSetAttribute(umma_gemm_kernel<Epi, kAMn, kBMn, kChain>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kLSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(1ull << (dev & 63));
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n_tiles = (int64_t)((M + kLBM - 1) / kLBM) * ((Nn + kLBN - 1) / kLBN);
    const unsigned grid = (unsigned)(n_tiles < sms ? n_tiles : sms);
    const int n_mb = (M + kLBM - 1) / kLBM;
    if (group_m <= 0)   // about 32 MB of A per m-group
        group_m = (int)std::max<int64_t>(1, ((int64_t)32 << 20) / ((int64_t)kLBM * K * 2));
    if (group_m > n_mb) group_m = n_mb;
    umma_gemm_kernel<Epi, kAMn, kBMn, kChain><<<grid, kLThreads, kLSmemBytes, stream>>>(ta, tb, ta2, tb2, M, Nn, K,
                                                                                        group_m, l2hints, epi);
    return cudaGetLastError();
}

// L2 eviction priorities of the operand tiles (l2hints: A in bits 0-1, B in bits 2-3;
// 1 = evict_first, 2 = evict_last, 0 = normal), measured on GB300 at hidden
// [8192, 4096] x W [75968, 4096]:
//  - logits GEMMs (forward, backward K1, the dual form): A = hidden rows,
//    reused by every vocabulary tile of the group, evict_last; with groups of
//    about 32 MB of A this cut the forward's DRAM reads from 6.3 GB (h
//    re-fetched for every few W tiles) to near one read of W, and its time by
//    16%. B = W evict_last as well: with W evict_first, the CTA pairs of a
//    group that share a W tile missed it in L2 (on one box the logp forward
//    took 2.76 ms against 2.66 ms, its backward 8.52 against 8.31 ms, and the
//    KL forward 5.79 against 5.65 ms).
//  - K2 (dz . W_c): both operands evict_last (each is re-read by the other's
//    group).
//  - K3 (dz^T . h): both evict_last, in groups of 4 m-blocks (2 on CTA pairs):
//    h (64 MB) then stays in L2 while dz streams past it; with h evict_first
//    it was re-read from DRAM for every group, and the backward took 8.5 ms
//    instead of 8.1-8.2 ms.
constexpr int kHintLogits = 2 | (2 << 2);
constexpr int kHintK2 = 2 | (2 << 2);
constexpr int kHintK3 = 2 | (2 << 2);

// group_m <= 0: about 32 MB of A per m-group (see tile_coords and launch_gemm_impl)
template <class Epi, bool kAMn = false, bool kBMn = false>
static cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, int M, int Nn, int K, const Epi &epi,
                               cudaStream_t stream, int group_m = 0, int l2hints = kHintLogits) {
    return launch_gemm_impl<Epi, kAMn, kBMn>(ta, tb, ta, tb, M, Nn, K, group_m, l2hints, epi, stream);
}

// CTA-pair form (umma_gemm_pair_kernel): K-major B maps need boxes of 128 rows
// (kPBHalf); MN-major maps are the same 64 x 64 boxes as for one CTA. group_m
// counts 256-row pair blocks; <= 0 picks about 32 MB of A per group.
template <class Epi, bool kAMn, bool kBMn, bool kDual, bool kChain = false>
static cudaError_t launch_gemm_pair_impl(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ta2,
                                        const CUtensorMap &tb2, int M, int Nn, int K, int K2, const Epi &epi,
                                        cudaStream_t stream, int group_m, int l2hints) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(attr_done.load() & (1ull << (dev & 63)))) {
        cudaError_t e = cudaFuncSetAttribute(umma_gemm_pair_kernel<Epi, kAMn, kBMn, kDual, kChain>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmemBytes);
        if (e != cudaSuccess) return e;
        if (kDual) {
            // the register split assumes the kernel is launched with exactly
            // kPairDualRegsLaunch registers a thread; with fewer, setmaxnreg.inc
            // would wait for registers that do not exist, so refuse instead
            cudaFuncAttributes fa;
            if ((e = cudaFuncGetAttributes(&fa, umma_gemm_pair_kernel<Epi, kAMn, kBMn, kDual, kChain>)) != cudaSuccess)
                return e;
            if (fa.numRegs != kPairDualRegsLaunch) return cudaErrorInvalidConfiguration;
        }
        attr_done.fetch_or(1ull << (dev & 63));
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int n_mp = (M + 2 * kLBM - 1) / (2 * kLBM);
    const int64_t n_tiles = (int64_t)n_mp * ((Nn + kLBN - 1) / kLBN);
    const int64_t pairs = std::max(1, sms / 2);
    const unsigned grid = (unsigned)(2 * (n_tiles < pairs ? n_tiles : pairs));
    if (group_m <= 0)   // about 32 MB of A (both products' A tiles in the dual form) per m-group
        group_m = (int)std::max<int64_t>(1, ((int64_t)32 << 20) / ((int64_t)2 * kLBM * (K + (kDual ? K2 : 0)) * 2));
    if (group_m > n_mp) group_m = n_mp;
    umma_gemm_pair_kernel<Epi, kAMn, kBMn, kDual, kChain><<<grid, pair_threads(kDual), kPSmemBytes, stream>>>(
        ta, tb, ta2, tb2, M, Nn, K, K2, group_m, l2hints, epi);
    return cudaGetLastError();
}
template <class Epi, bool kAMn = false, bool kBMn = false>
static cudaError_t launch_gemm_pair(const CUtensorMap &ta, const CUtensorMap &tb, int M, int Nn, int K,
                                   const Epi &epi, cudaStream_t stream, int group_m, int l2hints) {
    return launch_gemm_pair_impl<Epi, kAMn, kBMn, false>(ta, tb, ta, tb, M, Nn, K, 0, epi, stream, group_m, l2hints);
}

#ifndef VP_GEMM_PAIRS
#define VP_GEMM_PAIRS 1
#endif
#ifndef VP_GEMM_FWD_PAIRS
#define VP_GEMM_FWD_PAIRS 1
#endif
constexpr bool kGemmPairs = VP_GEMM_PAIRS != 0;        // backward GEMMs on CTA pairs
constexpr bool kFwdPairs = VP_GEMM_FWD_PAIRS != 0;     // forward logits GEMMs on CTA pairs

// A logits GEMM: A = hidden rows [M, K], B = rows of W [Nn, K], both bf16
// row-major (K-major), on CTA pairs or single CTAs; builds its tensor maps.
template <class Epi>
static cudaError_t launch_logits_gemm(const void *A, const void *B, int M, int Nn, int K, const Epi &epi,
                                      cudaStream_t stream, bool pairs) {
    CUtensorMap ta, tb;
    if (!make_map(&ta, A, M, K, K, kLBM) || !make_map(&tb, B, Nn, K, K, pairs ? kPBHalf : kLBN))
        return cudaErrorInvalidValue;
    return pairs ? launch_gemm_pair<Epi>(ta, tb, M, Nn, K, epi, stream, 0, kHintLogits)
                 : launch_gemm(ta, tb, M, Nn, K, epi, stream);
}

// Both products of the dual form, on CTA pairs: C = A . B^T (K deep) and
// C2 = A2 . B2^T (K2 deep); the B maps have kPBHalf-row boxes.
template <class Epi>
static cudaError_t launch_gemm_dual(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ta2,
                                    const CUtensorMap &tb2, int M, int Nn, int K, int K2, const Epi &epi,
                                    cudaStream_t stream) {
    return launch_gemm_pair_impl<Epi, false, false, true>(ta, tb, ta2, tb2, M, Nn, K, K2, epi, stream, 0, kHintLogits);
}

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// Backward vocabulary chunk: vc rows of W at a time (32768 for up to 8192
// hidden rows, fewer for more rows, so that dz of a chunk stays near 0.5 GB;
// larger chunks mean fewer launches and fewer read-modify-write passes over
// dhidden).
static int64_t chunk_cols(int64_t N, int64_t V) {
    const int64_t vc = N <= 8192 ? 32768 : N <= 16384 ? 16384 : 8192;
    return V < vc ? ((V + 255) / 256) * 256 : vc;
}

// The two gradient GEMMs of one vocabulary chunk [v0, v0 + nv) for one model
// (hidden h [N, D], head W [V, D]) given the chunk's dz (bf16 [N, nv], pitch vc):
//   K2  acc (+)= dz . W_c  (A = dz K-major, B = W_c MN-major, K = nv; the first
//       chunk stores; the last one (last = true) writes bf16(acc + tile) to
//       dhidden instead)
//   K3  dW_c = dz^T . h    (A = dz MN-major, B = h MN-major, K = N), written as bf16
// With dz_lo (the same layout) dz is the pair dz_hi + dz_lo of bf16 values
// (dz_hi = dz rounded to bf16, dz_lo = the remainder rounded to bf16, about 16
// significant bits together), and each GEMM chains a second product with
// dz_lo in place of dz into the same fp32 accumulator, at twice the work.
// acc and dW may each be null (that GEMM is skipped); dhidden is non-null when
// acc is. Both GEMMs stream two
// operands far larger than L2 along a long K, so their tiles run in small
// m-groups (tile_coords): the concurrent CTAs then share a few A and B tiles
// instead of each A tile being fetched from DRAM once per n-block.
#ifndef VP_K2_GROUP
#define VP_K2_GROUP 16
#endif
#ifndef VP_K3_GROUP
#define VP_K3_GROUP 4
#endif
constexpr int kGradGroupM = VP_K2_GROUP;   // K2: m-blocks of dz (8 MB each at vc = 32768) x the 16 n-blocks of D = 4096
constexpr int kWGroupM = VP_K3_GROUP;      // K3: m-blocks of dz^T (2 MB each at N = 8192) x the n-blocks of D

template <class Epi, bool kAMn, bool kBMn>
static cudaError_t launch_grad_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &ta2,
                                    bool chain, int M, int Nn, int K, const Epi &epi, cudaStream_t stream,
                                    int group_m, int l2hints) {
    if (kGemmPairs)
        return chain ? launch_gemm_pair_impl<Epi, kAMn, kBMn, false, true>(ta, tb, ta2, tb, M, Nn, K, K, epi, stream,
                                                                          (group_m + 1) / 2, l2hints)
                     : launch_gemm_pair_impl<Epi, kAMn, kBMn, false>(ta, tb, ta, tb, M, Nn, K, 0, epi, stream,
                                                                    (group_m + 1) / 2, l2hints);
    return chain ? launch_gemm_impl<Epi, kAMn, kBMn, true>(ta, tb, ta2, tb, M, Nn, K, group_m, l2hints, epi, stream)
                 : launch_gemm_impl<Epi, kAMn, kBMn>(ta, tb, ta, tb, M, Nn, K, group_m, l2hints, epi, stream);
}

static cudaError_t chunk_gradient_gemms(const CUtensorMap &tm_h_mn, const __nv_bfloat16 *W, int N, int D, int64_t v0,
                                        int nv, int64_t vc, const __nv_bfloat16 *dz, const __nv_bfloat16 *dz_lo,
                                        float *acc, __nv_bfloat16 *dhidden, __nv_bfloat16 *dW, bool last,
                                        cudaStream_t stream) {
    cudaError_t e;
    const bool chain = dz_lo != nullptr;
    if (acc) {
        CUtensorMap tm_dz, tm_dz_lo, tm_wc_mn;
        if (!make_map(&tm_dz, dz, N, nv, vc, kLBM) || !make_map_mn(&tm_wc_mn, W + v0 * D, nv, D, D) ||
            (chain && !make_map(&tm_dz_lo, dz_lo, N, nv, vc, kLBM)))
            return cudaErrorInvalidValue;
        const AccEpi ae{N, D, v0 == 0, acc, last ? dhidden : nullptr};
        e = launch_grad_gemm<AccEpi, false, true>(tm_dz, tm_wc_mn, chain ? tm_dz_lo : tm_dz, chain, N, D, nv, ae,
                                                  stream, kGradGroupM, kHintK2);
        if (e != cudaSuccess) return e;
    }
    if (dW) {
        CUtensorMap tm_dz_mn, tm_dz_lo_mn;
        if (!make_map_mn(&tm_dz_mn, dz, N, nv, vc) || (chain && !make_map_mn(&tm_dz_lo_mn, dz_lo, N, nv, vc)))
            return cudaErrorInvalidValue;
        const StoreBf16Epi se{nv, D, v0, dW};
        e = launch_grad_gemm<StoreBf16Epi, true, true>(tm_dz_mn, tm_h_mn, chain ? tm_dz_lo_mn : tm_dz_mn, chain, nv, D,
                                                       N, se, stream, kWGroupM, kHintK3);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Reads (and optionally clears) this translation unit's fault word.
static cudaError_t read_tu_fault(uint32_t *value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_linear_fault, sizeof(uint32_t));
    if (e == cudaSuccess && clear && *value) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_linear_fault, &zero, sizeof(uint32_t));
    }
    return e;
}

}  // namespace vp
