// vp_linear.cu -- fused linear logp forward and backward on tcgen05 tensor cores.
//
// Sources:
//   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton", "Implementation":
//        the forward computes logp = h . w_t - LSE_j(h . w_j) over a vocabulary
//        shard without materialising the logits and returns (logp, lse); a
//        tensor-parallel merge takes the max of the running maxima, rescales
//        and sums the running sums, and sums the target logit, which exactly
//        one shard owns.
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL",
//        second commit message (partials re-centred on the max).
//
// Kernel 1 (umma_gemm_kernel<LseEpi>), a persistent grid of one CTA per SM:
//   tiles of 128 hidden rows x 256 vocabulary rows of W, K = D in steps of 64;
//   warp 0 (one thread) streams the bf16 operand tiles with 2-D TMA into a
//   4-stage ring (48 KB per stage, 128-byte swizzle); warp 1 (one thread)
//   issues tcgen05.mma (M = 128, N = 256, K = 16 per instruction) into one of
//   two 256-column fp32 accumulators in TMEM and commits each stage back to
//   the producer; warps 2-5 read a finished accumulator with tcgen05.ld (one
//   thread per row), take the tile's per-row max m and sum-exp S in fp32,
//   pick out the target logit when the target falls in the tile, and hand the
//   accumulator back. The logits exist only in TMEM and registers.
//   Tiles run vocabulary-major, so the CTAs working at the same time share one
//   2 MB slice of W through L2 while the hidden states (here 64 MB) stay
//   resident in L2.
// Kernel 2 (linear_merge_kernel): one warp per row re-centres the row's
//   per-tile (m, S) on their max (fp32 exponentials, double-float sums), in a
//   fixed order, and writes logp and the vp_rowstat record (fp64 finish).
// Scratch: float2 partials [N][ceil(V/256)] and the target logits [N] fp32,
//   in a caller-provided workspace (see vp_linear_logp_workspace_size).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "vp_device.cuh"
#include "vp_launch.h"
#include "vp_stats.cuh"
#include "vp_umma.cuh"

namespace vp {

constexpr int kLBM = 128, kLBN = 256, kLBK = 64;
constexpr int kLStages = 4;
constexpr int kLAStage = kLBM * kLBK * 2;          // 16 KB
constexpr int kLBStage = kLBN * kLBK * 2;          // 32 KB
constexpr int kLStageBytes = kLAStage + kLBStage;  // 48 KB
constexpr int kLSmemBytes = kLStages * kLStageBytes + 1024;  // + alignment slack
constexpr int kLThreads = 192;                     // TMA warp, MMA warp, 4 epilogue warps
constexpr uint32_t kLTmemCols = 2 * kLBN;          // two accumulators

// Set when a bounded wait of the linear kernels gave up.
__device__ uint32_t g_linear_fault;

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
// place. Tiles run N-major (consecutive CTAs share one B tile through L2).
// The epilogue functor is called by each of the 128 epilogue threads for its
// accumulator row: epi(row, col0, ncol, taddr), taddr = the TMEM address of the
// row's 256 columns; it reads them with tmem_ld32, which is warp-collective, so
// every lane runs every load (rows past M included) and only the global
// accesses are guarded.
// ---------------------------------------------------------------------------
constexpr uint32_t kLMnAtomBytes = 64 * kLBK * 2;   // one 64 (MN) x 64 (K) box: 8 KB

template <class Epi, bool kAMn = false, bool kBMn = false>
__global__ void __launch_bounds__(kLThreads, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int M, int Nn,
                 int K, const Epi epi) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ LinearBars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_mb = (M + kLBM - 1) / kLBM, n_nb = (Nn + kLBN - 1) / kLBN;
    const int64_t n_tiles = (int64_t)n_mb * n_nb;
    const int n_k = (K + kLBK - 1) / kLBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.acc_full[b], 1);
            mbar_init(&bars.acc_empty[b], 4 * 32);
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
            uint32_t it = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                const int mb = (int)(tile % n_mb), nb = (int)(tile / n_mb);
                for (int kb = 0; kb < n_k; ++kb, ++it) {
                    const uint32_t st = it % kLStages, use = it / kLStages;
                    if (use > 0 && !mbar_wait(&bars.empty[st], (use - 1) & 1)) { ok = false; break; }
                    uint8_t *a = smem + st * kLStageBytes;
                    mbar_arrive_expect_tx(&bars.full[st], kLStageBytes);
                    if (kAMn) {
#pragma unroll
                        for (int i = 0; i < kLBM / 64; ++i)
                            tma_load_2d(a + i * kLMnAtomBytes, &tm_a, mb * kLBM + 64 * i, kb * kLBK, &bars.full[st]);
                    } else {
                        tma_load_2d(a, &tm_a, kb * kLBK, mb * kLBM, &bars.full[st]);
                    }
                    if (kBMn) {
#pragma unroll
                        for (int i = 0; i < kLBN / 64; ++i)
                            tma_load_2d(a + kLAStage + i * kLMnAtomBytes, &tm_b, nb * kLBN + 64 * i, kb * kLBK,
                                        &bars.full[st]);
                    } else {
                        tma_load_2d(a + kLAStage, &tm_b, kb * kLBK, nb * kLBN, &bars.full[st]);
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
                for (int kb = 0; kb < n_k; ++kb, ++it) {
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
            const int mb = (int)(tile % n_mb), nb = (int)(tile / n_mb);
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

// Forward epilogue: the tile's per-row max m and sum-exp S (fp32) and the target
// logit when the row's target falls in the tile.
struct LseEpi {
    int N, V, n_vt;
    int64_t vocab_start;
    const int64_t *targets;
    float2 *partials;   // [N][n_vt]
    float *tgt_logit;   // [N]
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const int64_t tg = valid ? targets[row] : -1;
        const int64_t t = tg - vocab_start - col0;
        const int tloc = (tg >= 0 && t >= 0 && t < ncol) ? (int)t : -1;
        float m = -INFINITY, S = 0.f, zt = 0.f;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            float cm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (c * 32 + i >= ncol) v[i] = -INFINITY;   // past the vocabulary
                if (c * 32 + i == tloc) zt = v[i];
                cm = fmaxf(cm, v[i]);
            }
            if (cm > m) {
                S *= exp2f((m - cm) * kLog2e);
                m = cm;
            }
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                s0 += exp2f((v[i] - m) * kLog2e);
                s1 += exp2f((v[i + 1] - m) * kLog2e);
            }
            S += s0 + s1;
        }
        if (!valid) return;
        partials[(int64_t)row * n_vt + col0 / kLBN] = make_float2(m, S);
        if (tloc >= 0) tgt_logit[row] = zt;
    }
};

// Backward K1 epilogue: dz = g (onehot - p), p = exp((z - m) - logS), for a
// 256-column tile of a vocabulary chunk starting at shard column v0, written
// as bf16 (round to nearest even) row-major dz[row][col] (pitch ldz); the two
// gradient GEMMs read it in place, dz^T through an MN-major tensor map. Rows
// with an ignored target get 0, rows with a data error or without valid
// statistics get NaN.
struct DzEpi {
    int N, V, v0, ldz;
    int64_t vocab_start;
    const int64_t *targets;
    const RowStat *stats;
    const float *g;
    __nv_bfloat16 *dz;
    int32_t *err;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const RowStat s = load_rowstat(stats + (valid ? row : 0));
        const int64_t tg = valid ? targets[row] : -1;
        const int64_t tl = tg - vocab_start;                // target column in the shard
        int mode = 0;                                      // 0 normal, 1 zero row, 2 NaN row
        if (tg < 0) mode = 1;
        else if (tl < 0 || tl >= V) mode = 2;
        if (s.flags & (kRowNanInf | kRowEmpty)) mode = mode == 1 ? 1 : 2;
        if (valid && mode == 2 && err && col0 == 0 && v0 == 0 && tg >= 0 && (tl < 0 || tl >= V))
            atomicOr(err, VP_ERRBIT_TARGET_);
        const int64_t tcol = tl - v0 - col0;               // target column within this tile
        const float gr = valid ? g[row] : 0.f;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                float d[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = c * 32 + i + e;
                    const float p = ex2_fast(((v[i + e] - s.m) - s.logS_hi) * kLog2e);
                    float x = (col == tcol) ? gr * (1.f - p) : -gr * p;
                    if (mode == 1 || col >= ncol) x = 0.f;
                    else if (mode == 2) x = __int_as_float(0x7fc00000);
                    d[e] = x;
                }
                __nv_bfloat162 b = __floats2bfloat162_rn(d[0], d[1]);
                packed[i / 2] = *reinterpret_cast<uint32_t *>(&b);
            }
            if (!valid) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(dz + (int64_t)row * ldz + col0 + c * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dst[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
        }
    }
};

// Backward K2 epilogue: acc[row][col] (+)= tile, fp32 (pitch ld).
struct AccEpi {
    int M, ld;
    bool first;
    float *acc;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < M;
        float *dst = acc + (int64_t)(valid ? row : 0) * ld + col0;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            if (!valid || c * 32 >= ncol) continue;
            float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float4 o = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                if (!first) {
                    const float4 a = d4[k];
                    o.x += a.x; o.y += a.y; o.z += a.z; o.w += a.w;
                }
                d4[k] = o;
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

// out[i] = bf16(acc[i]) for rows x cols (pitches in elements)
__global__ void __launch_bounds__(256) to_bf16_kernel(const float *__restrict__ acc, int64_t n,
                                                      __nv_bfloat16 *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = __float2bfloat16_rn(acc[i]);
}

// One warp per row: merge of the row's per-tile (m, S) in a fixed order.
__global__ void __launch_bounds__(256)
linear_merge_kernel(int N, int V, int64_t vocab_start, const int64_t *__restrict__ targets,
                    const float2 *__restrict__ partials, const float *__restrict__ tgt_logit,
                    float *__restrict__ logp, RowStat *__restrict__ stats, int32_t *__restrict__ err) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const int n_vt = (V + kLBN - 1) / kLBN;
    const float2 *p = partials + (int64_t)row * n_vt;
    float M = -INFINITY;
    for (int i = lane; i < n_vt; i += 32) M = fmaxf(M, p[i].x);
    M = warp_max(M);
    // fp32 exponentials summed as double-floats: each term carries a few fp32
    // roundings and the positive sum adds none, so S keeps ~1e-7 relative
    // accuracy without the narrow fp64 pipe
    DF Sdf{0.f, 0.f};
    bool nan = false;
    for (int i = lane; i < n_vt; i += 32) {
        const float2 v = p[i];
        if (v.y != v.y) nan = true;
        else if (v.y > 0.f) df_add(Sdf, v.y * expf(v.x - M));
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) df_add(Sdf, shfl_xor(Sdf, m));
    nan = __any_sync(0xffffffffu, nan);
    if (lane != 0) return;
    const double S = df_value(Sdf);
    uint32_t flags = 0;
    if (nan || S != S) flags |= kRowNanInf;
    else if (S == 0.0) flags |= kRowEmpty;
    const double logS = log(S);
    store_rowstat(stats + row, M, logS, 0.0, flags);
    const int64_t t = targets[row];
    if (t < 0) { logp[row] = 0.f; return; }
    const int64_t loc = t - vocab_start;
    if (loc < 0 || loc >= V) {
        logp[row] = qnan();
        if (err) atomicOr(err, VP_ERRBIT_TARGET_);
        return;
    }
    logp[row] = flags ? qnan() : (float)(((double)tgt_logit[row] - (double)M) - logS);
}

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

template <class Epi, bool kAMn = false, bool kBMn = false>
static cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, int M, int Nn, int K, const Epi &epi,
                               cudaStream_t stream) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(attr_done.load() & (1ull << (dev & 63)))) {
        cudaError_t e = cudaFuncSetAttribute(umma_gemm_kernel<Epi, kAMn, kBMn>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kLSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(1ull << (dev & 63));
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n_tiles = (int64_t)((M + kLBM - 1) / kLBM) * ((Nn + kLBN - 1) / kLBN);
    const unsigned grid = (unsigned)(n_tiles < sms ? n_tiles : sms);
    umma_gemm_kernel<Epi, kAMn, kBMn><<<grid, kLThreads, kLSmemBytes, stream>>>(ta, tb, M, Nn, K, epi);
    return cudaGetLastError();
}

size_t linear_workspace_bytes(int64_t N, int64_t V) {
    const int64_t n_vt = (V + kLBN - 1) / kLBN;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return up((size_t)N * n_vt * sizeof(float2)) + up((size_t)N * sizeof(float));
}

cudaError_t launch_linear_logp_fwd(const LinearFwdArgs &a) {
    CUtensorMap tm_h, tm_w;
    if (!make_map(&tm_h, a.hidden, a.N, a.D, a.D, kLBM) || !make_map(&tm_w, a.weight, a.V, a.D, a.D, kLBN))
        return cudaErrorInvalidValue;
    const int64_t n_vt = (a.V + kLBN - 1) / kLBN;
    float2 *partials = static_cast<float2 *>(a.workspace);
    float *tgt = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) +
                                           (((size_t)a.N * n_vt * sizeof(float2) + 255) & ~(size_t)255));
    const LseEpi epi{(int)a.N, (int)a.V, (int)n_vt, a.vocab_start, a.targets, partials, tgt};
    cudaError_t e = launch_gemm(tm_h, tm_w, (int)a.N, (int)a.V, (int)a.D, epi, a.stream);
    if (e != cudaSuccess) return e;
    linear_merge_kernel<<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
        (int)a.N, (int)a.V, a.vocab_start, a.targets, partials, tgt, a.logp, static_cast<RowStat *>(a.stats), a.err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// No-allocation variant: the same two kernels with their scratch in a fixed
// array inside the library instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device. In host code the
// symbol's name is only a host-side stand-in, so the address is looked up once
// per device with that device current, and cached.
static cudaError_t noalloc_scratch_address(void **out) {
    static std::atomic<void *> cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void *p = cached[dev].load();
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        cached[dev].store(p);
    }
    *out = p;
    return cudaSuccess;
}

cudaError_t launch_linear_logp_fwd_noalloc(const LinearFwdArgs &a) {
    void *scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    CUtensorMap tm_h, tm_w;
    if (!make_map(&tm_h, a.hidden, a.N, a.D, a.D, kLBM) || !make_map(&tm_w, a.weight, a.V, a.D, a.D, kLBN))
        return cudaErrorInvalidValue;
    const int64_t n_vt = (a.V + kLBN - 1) / kLBN;
    // Every partial and every in-shard target logit is written by the first
    // kernel before the merge reads it, so nothing in the array needs clearing.
    float2 *partials = static_cast<float2 *>(scratch);
    float *tgt = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) +
                                           (((size_t)a.N * n_vt * sizeof(float2) + 255) & ~(size_t)255));
    const LseEpi epi{(int)a.N, (int)a.V, (int)n_vt, a.vocab_start, a.targets, partials, tgt};
    e = launch_gemm(tm_h, tm_w, (int)a.N, (int)a.V, (int)a.D, epi, a.stream);
    if (e != cudaSuccess) return e;
    linear_merge_kernel<<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
        (int)a.N, (int)a.V, a.vocab_start, a.targets, partials, tgt, a.logp, static_cast<RowStat *>(a.stats), a.err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Backward: vocabulary chunks of vc rows of W (32768 for up to 8192 hidden rows,
// fewer for more rows, so that dz of a chunk stays near 0.5 GB; larger chunks
// mean fewer launches and fewer read-modify-write passes over dhidden).
//   K1  logits tile (h . W_c^T, K = D) -> dz                   (DzEpi)
//   K2  dhidden_acc (+)= dz . W_c     (A = dz K-major, B = W_c MN-major, K = chunk)   (AccEpi)
//   K3  dW_c = dz^T . h               (A = dz MN-major, B = h MN-major, K = N)        (StoreBf16Epi)
// The transposed operands are read in place through MN-major tensor maps.
// ---------------------------------------------------------------------------
static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct BwdLayout {
    size_t dz, acc, total;
};

static int64_t chunk_cols(int64_t N, int64_t V) {
    const int64_t vc = N <= 8192 ? 32768 : N <= 16384 ? 16384 : 8192;
    return V < vc ? ((V + 255) / 256) * 256 : vc;
}

static BwdLayout bwd_layout(int64_t N, int64_t V, int64_t D) {
    const int64_t vc = chunk_cols(N, V);
    BwdLayout L;
    L.dz = 0;
    L.acc = L.dz + up256((size_t)N * vc * 2);
    L.total = L.acc + up256((size_t)N * D * 4);
    return L;
}

size_t linear_bwd_workspace_bytes(int64_t N, int64_t V, int64_t D) { return bwd_layout(N, V, D).total; }

cudaError_t launch_linear_logp_bwd(const LinearBwdArgs &a) {
    const BwdLayout L = bwd_layout(a.N, a.V, a.D);
    const int64_t vc = chunk_cols(a.N, a.V);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    __nv_bfloat16 *dz = reinterpret_cast<__nv_bfloat16 *>(ws + L.dz);
    float *acc = reinterpret_cast<float *>(ws + L.acc);
    const __nv_bfloat16 *h = static_cast<const __nv_bfloat16 *>(a.hidden);
    const __nv_bfloat16 *W = static_cast<const __nv_bfloat16 *>(a.weight);
    const int N = (int)a.N, V = (int)a.V, D = (int)a.D;
    cudaError_t e;

    CUtensorMap tm_h, tm_h_mn;
    if (!make_map(&tm_h, h, N, D, D, kLBM) || !make_map_mn(&tm_h_mn, h, N, D, D)) return cudaErrorInvalidValue;
    for (int64_t v0 = 0; v0 < V; v0 += vc) {
        const int nv = (int)(V - v0 < vc ? V - v0 : vc);
        // K1 over this chunk's rows of W (the map's rows start at v0)
        CUtensorMap tm_wc;
        if (!make_map(&tm_wc, W + v0 * D, nv, D, D, kLBN)) return cudaErrorInvalidValue;
        const DzEpi de{N, V, (int)v0, (int)vc, a.vocab_start, a.targets, static_cast<const RowStat *>(a.stats), a.g,
                       dz, a.err};
        if ((e = launch_gemm(tm_h, tm_wc, N, nv, D, de, a.stream)) != cudaSuccess) return e;
        if (a.dhidden) {
            CUtensorMap tm_dz, tm_wc_mn;
            if (!make_map(&tm_dz, dz, N, nv, vc, kLBM) || !make_map_mn(&tm_wc_mn, W + v0 * D, nv, D, D))
                return cudaErrorInvalidValue;
            const AccEpi ae{N, D, v0 == 0, acc};
            if ((e = launch_gemm<AccEpi, false, true>(tm_dz, tm_wc_mn, N, D, nv, ae, a.stream)) != cudaSuccess)
                return e;
        }
        if (a.dW) {
            CUtensorMap tm_dz_mn;
            if (!make_map_mn(&tm_dz_mn, dz, N, nv, vc)) return cudaErrorInvalidValue;
            const StoreBf16Epi se{nv, D, v0, static_cast<__nv_bfloat16 *>(a.dW)};
            if ((e = launch_gemm<StoreBf16Epi, true, true>(tm_dz_mn, tm_h_mn, nv, D, N, se, a.stream)) != cudaSuccess)
                return e;
        }
    }
    if (a.dhidden) {
        const int64_t n = (int64_t)N * D;
        to_bf16_kernel<<<(unsigned)((n + 255) / 256 < 65535 ? (n + 255) / 256 : 65535), 256, 0, a.stream>>>(
            acc, n, static_cast<__nv_bfloat16 *>(a.dhidden));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t read_linear_fault(uint32_t *value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_linear_fault, sizeof(uint32_t));
    if (e == cudaSuccess && clear && *value) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_linear_fault, &zero, sizeof(uint32_t));
    }
    return e;
}

}  // namespace vp
