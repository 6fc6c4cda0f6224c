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
// Kernel 1 (umma_gemm_pair_kernel<LseEpi>, vp_gemm.cuh), a persistent grid of
//   CTA pairs: tiles of 256 hidden rows x 256 vocabulary rows of W, K = D in
//   steps of 64. Each CTA of a pair holds 128 rows of the hidden tile, 128 rows
//   of the W tile and its 128 rows of the accumulators; its TMA thread streams
//   the bf16 operand tiles into a 6-stage ring (32 KB per stage, 128-byte
//   swizzle); one thread of the leader issues tcgen05.mma.cta_group::2
//   (M = 256, N = 256, K = 16) into one of two 256-column fp32 accumulators in
//   TMEM. The epilogue warps read a finished accumulator with tcgen05.ld (one
//   thread per row), take the tile's per-row max m and sum-exp S in fp32, pick
//   out the target logit when the target falls in the tile, and hand the
//   accumulator back. The logits exist only in TMEM and registers. Tiles run
//   in groups of about 32 MB of hidden rows, with the hidden tiles marked
//   evict_last and the W tiles evict_first in L2, so that W is read from DRAM
//   about once per group while the group's hidden rows stay in L2.
// Kernel 2 (linear_merge_kernel): one warp per row re-centres the row's
//   per-tile (m, S) on their max (fp32 exponentials, double-float sums), in a
//   fixed order, and writes logp and the vp_rowstat record (fp64 finish).
// Scratch: float2 partials [N][ceil(V/256)] and the target logits [N] fp32,
//   in a caller-provided workspace (see vp_linear_logp_workspace_size).
#include <mutex>

#include "vp_gemm.cuh"
#include "vp_stats.cuh"

namespace vp {

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
// as bf16 (round to nearest even) row-major dz[row][col] (pitch ldz), and with
// lo_off != 0 the remainder as a second bf16 array at dz + lo_off (store_dz);
// the gradient GEMMs read both in place, dz^T through an MN-major tensor map.
// At the target 1 - p is formed as -(e^{log p} - 1) where p > e^{-1/2}, so it
// keeps its relative accuracy as p -> 1. Rows with an ignored target get 0,
// rows with a data error or without valid statistics get NaN.
struct DzEpi {
    int N, V, v0, ldz;
    int64_t vocab_start;
    const int64_t *targets;
    const RowStat *stats;
    const float *g;
    __nv_bfloat16 *dz;
    int32_t *err;
    int64_t lo_off;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const RowStat s = load_rowstat(stats + (valid ? row : 0));
        const int64_t tg = valid ? targets[row] : -1;
        const int64_t tl = tg - vocab_start;                // target column in the shard
        int mode = 0;                                      // 0 normal, 1 zero row, 2 NaN row
        // records merged from vocabulary shards (kRowSharded): a target outside
        // this shard has its onehot term in another shard; the merge flagged
        // the rows whose target no shard holds (kRowBadTarget)
        const bool sharded = (s.flags & kRowSharded) != 0;
        if (tg < 0) mode = 1;
        else if ((tl < 0 || tl >= V) && !sharded) mode = 2;
        if (s.flags & (kRowNanInf | kRowEmpty)) mode = mode == 1 ? 1 : 2;
        if (tg >= 0 && (s.flags & kRowBadTarget)) mode = 2;
        if (valid && mode == 2 && err && col0 == 0 && v0 == 0 && tg >= 0 && (tl < 0 || tl >= V) && !sharded)
            atomicOr(err, VP_ERRBIT_TARGET_);
        const int64_t tcol = tl - v0 - col0;               // target column within this tile
        const float gr = valid ? g[row] : 0.f;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int col = c * 32 + i;
                const float lp = (v[i] - s.m) - s.logS_hi;
                const float p = ex2_fast(lp * kLog2e);
                float x = -gr * p;
                if (col == tcol) {
                    const float lpt = lp - s.logS_lo;
                    x = gr * (lpt > -0.5f ? -expm1_small(lpt) : 1.f - p);
                }
                if (mode == 1 || col >= ncol) x = 0.f;
                else if (mode == 2) x = __int_as_float(0x7fc00000);
                v[i] = x;
            }
            if (valid) store_dz(dz + (int64_t)row * ldz + col0 + c * 32, v, lo_off);
        }
    }
};

// One warp per row: merge of the row's per-tile (m, S) in a fixed order.
// kPart: the row's record over this vocabulary shard (vp_partial) instead of
// logp and the row statistics; a target in another shard is not an error.
template <bool kPart>
__global__ void __launch_bounds__(256)
linear_merge_kernel(int N, int V, int64_t vocab_start, const int64_t *__restrict__ targets,
                    const float2 *__restrict__ partials, const float *__restrict__ tgt_logit,
                    float *__restrict__ logp, RowStat *__restrict__ stats, int32_t *__restrict__ err,
                    PartialRec *__restrict__ shard_parts) {
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
    if constexpr (kPart) {
        uint32_t pf = (nan || S != S) ? kPartNanInf : 0u;
        const int64_t t = targets[row];
        float zt = 0.f;
        if (t < 0) {
            pf |= kPartIgnored;
        } else if (t - vocab_start >= 0 && t - vocab_start < V) {
            pf |= kPartHasTarget;
            zt = tgt_logit[row];
        }
        shard_parts[row] = PartialRec{S > 0.0 ? M : kNegBig, 0.f, S, 0.0, 0.0, zt, pf};
        return;
    }
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

size_t linear_workspace_bytes(int64_t N, int64_t V) {
    const int64_t n_vt = (V + kLBN - 1) / kLBN;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return up((size_t)N * n_vt * sizeof(float2)) + up((size_t)N * sizeof(float));
}

cudaError_t launch_linear_logp_fwd(const LinearFwdArgs &a) {
    const int64_t n_vt = (a.V + kLBN - 1) / kLBN;
    float2 *partials = static_cast<float2 *>(a.workspace);
    float *tgt = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) +
                                           (((size_t)a.N * n_vt * sizeof(float2) + 255) & ~(size_t)255));
    const LseEpi epi{(int)a.N, (int)a.V, (int)n_vt, a.vocab_start, a.targets, partials, tgt};
    cudaError_t e = launch_logits_gemm(a.hidden, a.weight, (int)a.N, (int)a.V, (int)a.D, epi, a.stream, kFwdPairs);
    if (e != cudaSuccess) return e;
    PartialRec *parts = static_cast<PartialRec *>(a.parts);
    if (parts)
        linear_merge_kernel<true><<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
            (int)a.N, (int)a.V, a.vocab_start, a.targets, partials, tgt, nullptr, nullptr, nullptr, parts);
    else
        linear_merge_kernel<false><<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
            (int)a.N, (int)a.V, a.vocab_start, a.targets, partials, tgt, a.logp, static_cast<RowStat *>(a.stats),
            a.err, nullptr);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// No-allocation variant: the same two kernels with their scratch in a fixed
// array inside the library instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current context. In host code the
// symbol's name is only a host-side stand-in, so the address is looked up with
// the device current (cudaGetSymbolAddress) at the first call on each device,
// and cached together with the context it belongs to: a call from another
// context on that device (after cudaDeviceReset, or a context the caller made
// current) looks the address up again instead of reusing a stale one.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

static CUcontext current_context() {
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load();
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f);
    }
    CUcontext ctx = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f)(&ctx) == CUDA_SUCCESS ? ctx : nullptr;
}

static cudaError_t noalloc_scratch_address(void **out) {
    struct Entry {
        CUcontext ctx;
        void *addr;
    };
    static Entry cached[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    CUcontext ctx = current_context();
    if (!cached[dev].addr || !ctx || cached[dev].ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        cached[dev] = Entry{current_context(), p};   // the lookup makes the primary context current if none was
    }
    *out = cached[dev].addr;
    return cudaSuccess;
}

cudaError_t launch_linear_logp_fwd_noalloc(const LinearFwdArgs &a) {
    void *scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    const int64_t n_vt = (a.V + kLBN - 1) / kLBN;
    // Every partial and every in-shard target logit is written by the first
    // kernel before the merge reads it, so nothing in the array needs clearing.
    float2 *partials = static_cast<float2 *>(scratch);
    float *tgt = reinterpret_cast<float *>(static_cast<uint8_t *>(scratch) +
                                           (((size_t)a.N * n_vt * sizeof(float2) + 255) & ~(size_t)255));
    const LseEpi epi{(int)a.N, (int)a.V, (int)n_vt, a.vocab_start, a.targets, partials, tgt};
    e = launch_logits_gemm(a.hidden, a.weight, (int)a.N, (int)a.V, (int)a.D, epi, a.stream, kFwdPairs);
    if (e != cudaSuccess) return e;
    linear_merge_kernel<false><<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
        (int)a.N, (int)a.V, a.vocab_start, a.targets, partials, tgt, a.logp, static_cast<RowStat *>(a.stats), a.err,
        nullptr);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Backward, per vocabulary chunk of vc rows of W:
//   K1  logits tile (h . W_c^T, K = D) -> dz                   (DzEpi)
//   K2, K3  dhidden_acc (+)= dz . W_c and dW_c = dz^T . h      (chunk_gradient_gemms)
// The transposed operands are read in place through MN-major tensor maps.
// ---------------------------------------------------------------------------
struct BwdLayout {
    size_t dz, acc, total;
};

// dz of one chunk twice over (hi and lo halves of the exact form; the fast
// form uses the first), then the fp32 dhidden accumulator
static BwdLayout bwd_layout(int64_t N, int64_t V, int64_t D) {
    const int64_t vc = chunk_cols(N, V);
    BwdLayout L;
    L.dz = 0;
    L.acc = L.dz + up256((size_t)2 * N * vc * 2);
    L.total = L.acc + up256((size_t)N * D * 4);
    return L;
}

size_t linear_bwd_workspace_bytes(int64_t N, int64_t V, int64_t D) { return bwd_layout(N, V, D).total; }

cudaError_t launch_linear_logp_bwd(const LinearBwdArgs &a) {
    const BwdLayout L = bwd_layout(a.N, a.V, a.D);
    const int64_t vc = chunk_cols(a.N, a.V);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    __nv_bfloat16 *dz = reinterpret_cast<__nv_bfloat16 *>(ws + L.dz);
    const int64_t lo_off = a.precision == VP_GRAD_EXACT_ ? a.N * vc : 0;   // dz_lo follows dz_hi
    float *acc = a.dhidden ? reinterpret_cast<float *>(ws + L.acc) : nullptr;
    const __nv_bfloat16 *h = static_cast<const __nv_bfloat16 *>(a.hidden);
    const __nv_bfloat16 *W = static_cast<const __nv_bfloat16 *>(a.weight);
    const int N = (int)a.N, V = (int)a.V, D = (int)a.D;
    cudaError_t e;

    CUtensorMap tm_h_mn;
    if (!make_map_mn(&tm_h_mn, h, N, D, D)) return cudaErrorInvalidValue;
    for (int64_t v0 = 0; v0 < V; v0 += vc) {
        const int nv = (int)(V - v0 < vc ? V - v0 : vc);
        // K1 over this chunk's rows of W
        const DzEpi de{N, V, (int)v0, (int)vc, a.vocab_start, a.targets, static_cast<const RowStat *>(a.stats), a.g,
                       dz, a.err, lo_off};
        if ((e = launch_logits_gemm(h, W + v0 * D, N, nv, D, de, a.stream, kGemmPairs)) != cudaSuccess) return e;
        if ((e = chunk_gradient_gemms(tm_h_mn, W, N, D, v0, nv, vc, dz, lo_off ? dz + lo_off : nullptr, acc,
                                      static_cast<__nv_bfloat16 *>(a.dhidden), static_cast<__nv_bfloat16 *>(a.dW),
                                      v0 + vc >= V, a.stream)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t read_linear_logp_fault(uint32_t *value, bool clear) { return read_tu_fault(value, clear); }

}  // namespace vp
