// vp_linear.cu -- fused linear logp forward on tcgen05 tensor cores.
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
// Kernel 1 (linear_lse_kernel), a persistent grid of one CTA per SM:
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
//   per-tile (m, S) on their max in fp64, in a fixed order, and writes logp
//   and the vp_rowstat record.
// Scratch: float2 partials [N][ceil(V/256)] and the target logits [N] fp32,
//   in a caller-provided workspace (see vp_linear_logp_workspace_size).
#include <cuda.h>
#include <cudaTypedefs.h>

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
constexpr uint32_t kLTmemCols = 2 * kLBN;          // two accumulators

// Set when a bounded wait of the linear kernels gave up.
__device__ uint32_t g_linear_fault;

struct LinearBars {
    uint64_t full[kLStages], empty[kLStages], acc_full[2], acc_empty[2];
    uint32_t tmem_base;
};

__global__ void __launch_bounds__(kLThreads, 1)
linear_lse_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w, int N, int V,
                  int D, int64_t vocab_start, const int64_t *__restrict__ targets, float2 *__restrict__ partials,
                  float *__restrict__ tgt_logit) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ LinearBars bars;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rb = (N + kLBM - 1) / kLBM, n_vt = (V + kLBN - 1) / kLBN;
    const int64_t n_tiles = (int64_t)n_rb * n_vt;
    const int n_k = D / kLBK;

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
        prefetch_tensormap(&tm_h);
        prefetch_tensormap(&tm_w);
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
                const int rb = (int)(tile % n_rb), vt = (int)(tile / n_rb);
                for (int kb = 0; kb < n_k; ++kb, ++it) {
                    const uint32_t st = it % kLStages, use = it / kLStages;
                    if (use > 0 && !mbar_wait(&bars.empty[st], (use - 1) & 1)) { ok = false; break; }
                    uint8_t *a = smem + st * kLStageBytes;
                    mbar_arrive_expect_tx(&bars.full[st], kLStageBytes);
                    tma_load_2d(a, &tm_h, kb * kLBK, rb * kLBM, &bars.full[st]);
                    tma_load_2d(a + kLAStage, &tm_w, kb * kLBK, vt * kLBN, &bars.full[st]);
                }
            }
            if (!ok) atomicOr(&g_linear_fault, 1u);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16(kLBM, kLBN);
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
                    for (int kk = 0; kk < kLBK / 16; ++kk)
                        umma_bf16(d, umma_desc_sw128(a + kk * 32), umma_desc_sw128(a + kLAStage + kk * 32), idesc,
                                  (kb | kk) != 0);
                    umma_commit(&bars.empty[st]);       // frees the stage once these MMAs are done
                }
                umma_commit(&bars.acc_full[buf]);       // the accumulator is complete
            }
            if (!ok) atomicOr(&g_linear_fault, 2u);
        }
    } else {
        // ---------------- epilogue: per-row (m, S) of each tile ----------------
        const int q = warp & 3;                          // TMEM lane quarter of this warp
        const int r_in = q * 32 + lane;
        uint32_t j = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++j) {
            const int rb = (int)(tile % n_rb), vt = (int)(tile / n_rb);
            const uint32_t buf = j & 1;
            if (ok && !mbar_wait(&bars.acc_full[buf], (j >> 1) & 1)) {
                ok = false;
                atomicOr(&g_linear_fault, 4u);
            }
            tc_fence_after();
            const int row = rb * kLBM + r_in;
            const int ncol = min(kLBN, V - vt * kLBN);   // valid vocabulary columns of this tile
            int tloc = -1;
            if (row < N) {
                const int64_t t = targets[row] - vocab_start - (int64_t)vt * kLBN;
                if (targets[row] >= 0 && t >= 0 && t < ncol) tloc = (int)t;
            }
            float m = -INFINITY, S = 0.f, zt = 0.f;
            const uint32_t base = tmem + buf * kLBN + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < kLBN / 32; ++c) {
                float v[32];
                tmem_ld32(base + c * 32, v);
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
            tc_fence_before();
            mbar_arrive(&bars.acc_empty[buf]);           // the MMA warp may reuse the accumulator
            if (row < N && ok) {
                partials[(int64_t)row * n_vt + vt] = make_float2(m, S);
                if (tloc >= 0) tgt_logit[row] = zt;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, kLTmemCols);
}

// One warp per row: fp64 merge of the row's per-tile (m, S), in a fixed order.
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
    double S = 0.0;
    bool nan = false;
    for (int i = lane; i < n_vt; i += 32) {
        const float2 v = p[i];
        if (v.y != v.y) nan = true;
        else if (v.y > 0.f) S += (double)v.y * exp((double)v.x - (double)M);
    }
    S = warp_sum(S);
    nan = __any_sync(0xffffffffu, nan);
    if (lane != 0) return;
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

// Row-major [rows, D] bf16 matrix, boxes of box_rows x 64 with the 128-byte swizzle.
static bool make_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t D, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {(cuuint32_t)kLBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t linear_workspace_bytes(int64_t N, int64_t V) {
    const int64_t n_vt = (V + kLBN - 1) / kLBN;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return up((size_t)N * n_vt * sizeof(float2)) + up((size_t)N * sizeof(float));
}

cudaError_t launch_linear_logp_fwd(const LinearFwdArgs &a) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(attr_done.load() & (1ull << (dev & 63)))) {
        cudaError_t e = cudaFuncSetAttribute(linear_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kLSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(1ull << (dev & 63));
    }
    CUtensorMap tm_h, tm_w;
    if (!make_map(&tm_h, a.hidden, a.N, a.D, kLBM) || !make_map(&tm_w, a.weight, a.V, a.D, kLBN))
        return cudaErrorInvalidValue;
    const int64_t n_vt = (a.V + kLBN - 1) / kLBN;
    float2 *partials = static_cast<float2 *>(a.workspace);
    float *tgt = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) +
                                           (((size_t)a.N * n_vt * sizeof(float2) + 255) & ~(size_t)255));
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n_tiles = ((a.N + kLBM - 1) / kLBM) * n_vt;
    const unsigned grid = (unsigned)(n_tiles < sms ? n_tiles : sms);
    linear_lse_kernel<<<grid, kLThreads, kLSmemBytes, a.stream>>>(tm_h, tm_w, (int)a.N, (int)a.V, (int)a.D,
                                                                   a.vocab_start, a.targets, partials, tgt);
    cudaError_t e = cudaGetLastError();
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
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(attr_done.load() & (1ull << (dev & 63)))) {
        e = cudaFuncSetAttribute(linear_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(1ull << (dev & 63));
    }
    CUtensorMap tm_h, tm_w;
    if (!make_map(&tm_h, a.hidden, a.N, a.D, kLBM) || !make_map(&tm_w, a.weight, a.V, a.D, kLBN))
        return cudaErrorInvalidValue;
    const int64_t n_vt = (a.V + kLBN - 1) / kLBN;
    // Every partial and every in-shard target logit is written by the first
    // kernel before the merge reads it, so nothing in the array needs clearing.
    float2 *partials = static_cast<float2 *>(scratch);
    float *tgt = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) +
                                           (((size_t)a.N * n_vt * sizeof(float2) + 255) & ~(size_t)255));
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t n_tiles = ((a.N + kLBM - 1) / kLBM) * n_vt;
    const unsigned grid = (unsigned)(n_tiles < sms ? n_tiles : sms);
    linear_lse_kernel<<<grid, kLThreads, kLSmemBytes, a.stream>>>(tm_h, tm_w, (int)a.N, (int)a.V, (int)a.D,
                                                                   a.vocab_start, a.targets, partials, tgt);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    linear_merge_kernel<<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
        (int)a.N, (int)a.V, a.vocab_start, a.targets, partials, tgt, a.logp, static_cast<RowStat *>(a.stats), a.err);
    return cudaGetLastError();
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
