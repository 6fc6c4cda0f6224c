// vp_linear_ent_kl.cu -- fused linear entropy, and fused linear KL between the
// next-token distributions of two models, on tcgen05 tensor cores, without
// materialising the logits.
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL":
//        second commit message and the reviewer's suggested change (one read
//        per logit: max, sum-exp and the max-centred weighted sum; partials
//        re-centred on the row max), the commit message adding
//        vocab_parallel_jsd ("Motivation": teacher-student divergences over
//        tiled LM-head projections without the full logits).
//   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton": "Implementation"
//        (logits h . W^T produced tile by tile and reduced on the fly) and the
//        review nitpick on the chunked backward (dz, then dhidden = dz . W and
//        dW = dz^T . h).
//
// Entropy of softmax(h . W^T), per row r:
//   forward   one GEMM (umma_gemm_kernel<EntEpi>): per 128 x 256 logits tile and
//             row, the tile max m, S = sum e^{z - m} and W = sum e^{z - m}(z - m)
//             (two passes over the tile in TMEM: max, then the sums); then a
//             merge per row re-centres the tiles on the row max (every term of W
//             is <= 0, so the merge has no cancellation) and writes
//             H = log S - W / S and the record (m, logS, c = W / S);
//   backward  per vocabulary chunk, the logits tile again and
//             dz = -g p ((z - m) - c) in the epilogue (DzEntEpi), then the two
//             gradient GEMMs.
// KL between model A (h_a . W_a^T) and model B (h_b . W_b^T), each model with
// its own hidden size; reverse = KL(A||B), forward = KL(B||A):
//   forward   the dual GEMM puts the same tile of both models' logits in TMEM
//             (A in columns 0-255, B in 256-511); the epilogue (KLEpi) takes the
//             tile's maxima of P and Q, S_P, S_Q and W = sum e^{P - m_P}
//             ((P - m_P) - (Q - m_Q)); the merge re-centres the tiles
//             (W_i -> alpha_i (W_i - (dP_i - dQ_i) S_P,i)) and writes
//             KL = W / S_P - log S_P + log S_Q with both records;
//   backward  the dual GEMM again, dP = g p ((P - m_P) - (Q - m_Q) - c) and
//             dQ = g (q - p) in the epilogue (DzKLEpi), then the gradient GEMMs
//             of each model whose gradients are asked for.
// The logits of a GEMM are finite for finite inputs, so there is no support
// mismatch; NaN or +inf logits make the row NaN (outputs and gradient rows).
#include "vp_gemm.cuh"
#include "vp_stats.cuh"

namespace vp {

// ---------------------------------------------------------------------------
// Forward epilogues (one thread per accumulator row; rows past N and columns
// past ncol take part in the TMEM loads but not in the results)
// ---------------------------------------------------------------------------
struct EntTile {
    float m, S, W, pad;   // tile max, sum e^{z-m}, sum e^{z-m} (z-m) (<= 0)
};

struct EntEpi {
    int N, n_vt;
    EntTile *parts;   // [N][n_vt]
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        float m = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i < ncol) m = fmaxf(m, v[i]);
        }
        float s0 = 0.f, s1 = 0.f, w0 = 0.f, w1 = 0.f;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float t0 = v[i] - m, t1 = v[i + 1] - m;
                const float e0 = c * 32 + i < ncol ? ex2_fast(t0 * kLog2e) : 0.f;
                const float e1 = c * 32 + i + 1 < ncol ? ex2_fast(t1 * kLog2e) : 0.f;
                s0 += e0;
                s1 += e1;
                w0 = e0 == 0.f ? w0 : fmaf(e0, t0, w0);   // zero-weight terms add nothing
                w1 = e1 == 0.f ? w1 : fmaf(e1, t1, w1);
            }
        }
        if (row >= N) return;
        parts[(int64_t)row * n_vt + col0 / kLBN] = EntTile{m, s0 + s1, w0 + w1, 0.f};
    }
};

struct KLTile {
    float mp, Sp, mq, Sq, W, pad0, pad1, pad2;
};

struct KLEpi {
    int N, n_vt;
    bool p_is_a;      // reverse: P = A (accumulator columns 0-255), Q = B (256-511)
    KLTile *parts;    // [N][n_vt]
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const uint32_t tp = taddr + (p_is_a ? 0u : (uint32_t)kLBN), tq = taddr + (p_is_a ? (uint32_t)kLBN : 0u);
        float mp = -INFINITY, mq = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < kDualEpiCols / 32; ++c) {
            float a[32], b[32];
            tmem_ld32(tp + c * 32, a);
            tmem_ld32(tq + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i < ncol) {
                    mp = fmaxf(mp, a[i]);
                    mq = fmaxf(mq, b[i]);
                }
        }
        float sp = 0.f, sq = 0.f, w = 0.f;
#pragma unroll 1
        for (int c = 0; c < kDualEpiCols / 32; ++c) {
            float a[32], b[32];
            tmem_ld32(tp + c * 32, a);
            tmem_ld32(tq + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const bool in = c * 32 + i < ncol;
                const float tP = a[i] - mp, tQ = b[i] - mq;
                const float ep = in ? ex2_fast(tP * kLog2e) : 0.f;
                const float eq = in ? ex2_fast(tQ * kLog2e) : 0.f;
                sp += ep;
                sq += eq;
                w = ep == 0.f ? w : fmaf(ep, tP - tQ, w);
            }
        }
        if (row >= N) return;
        parts[(int64_t)row * n_vt + col0 / kDualEpiCols] = KLTile{mp, sp, mq, sq, w, 0.f, 0.f, 0.f};
    }
};

// ---------------------------------------------------------------------------
// Merges: one warp per row, the row's tiles in a fixed order (lane-strided,
// then a fixed shuffle tree), fp32 exponentials summed as double-floats, fp64
// finish; the result depends on V only, not on N (batch invariance).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
linear_entropy_merge_kernel(int N, int n_vt, const EntTile *__restrict__ parts, float *__restrict__ H,
                            RowStat *__restrict__ stats) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const EntTile *p = parts + (int64_t)row * n_vt;
    float M = -INFINITY;
    for (int i = lane; i < n_vt; i += 32) M = fmaxf(M, p[i].m);
    M = warp_max(M);
    DF S{0.f, 0.f}, W{0.f, 0.f};
    bool nan = false;
    for (int i = lane; i < n_vt; i += 32) {
        const EntTile t = p[i];
        if (t.S != t.S || t.W != t.W || t.m == INFINITY) { nan = true; continue; }
        if (!(t.S > 0.f)) continue;                       // zero-weight tile
        const float a = expf(t.m - M);
        if (a == 0.f) continue;
        df_add(S, a * t.S);
        df_add(W, a * fmaf(-(M - t.m), t.S, t.W));        // both terms <= 0
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        df_add(S, shfl_xor(S, m));
        df_add(W, shfl_xor(W, m));
    }
    nan = __any_sync(0xffffffffu, nan);
    if (lane != 0) return;
    const double s = df_value(S), w = df_value(W);
    uint32_t flags = 0;
    if (nan || s != s || M != M) flags |= kRowNanInf;
    else if (!(s > 0.0)) flags |= kRowEmpty;
    const double logS = log(s), c = w / s;
    store_rowstat(stats + row, M, logS, c, flags);
    H[row] = flags ? qnan() : (float)(logS - c);
}

__global__ void __launch_bounds__(256)
linear_kl_merge_kernel(int N, int n_vt, const KLTile *__restrict__ parts, float *__restrict__ kl,
                       RowStat *__restrict__ stats_p, RowStat *__restrict__ stats_q) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const KLTile *p = parts + (int64_t)row * n_vt;
    float Mp = -INFINITY, Mq = -INFINITY;
    for (int i = lane; i < n_vt; i += 32) {
        Mp = fmaxf(Mp, p[i].mp);
        Mq = fmaxf(Mq, p[i].mq);
    }
    Mp = warp_max(Mp);
    Mq = warp_max(Mq);
    DF Sp{0.f, 0.f}, Sq{0.f, 0.f}, W{0.f, 0.f};
    bool nanp = false, nanq = false;
    for (int i = lane; i < n_vt; i += 32) {
        const KLTile t = p[i];
        const bool bp = t.Sp != t.Sp || t.W != t.W || t.mp == INFINITY;
        const bool bq = t.Sq != t.Sq || t.mq == INFINITY;
        nanp |= bp;
        nanq |= bq;
        if (bp || bq) continue;
        if (t.Sq > 0.f) {
            const float aq = expf(t.mq - Mq);
            if (aq != 0.f) df_add(Sq, aq * t.Sq);
        }
        if (t.Sp > 0.f) {
            const float ap = expf(t.mp - Mp);
            if (ap != 0.f) {
                df_add(Sp, ap * t.Sp);
                // W_i about the row centres: W_i - ((Mp - mp_i) - (Mq - mq_i)) S_P,i
                const float shift = (Mp - t.mp) - (Mq - t.mq);
                df_add(W, ap * t.W);
                df_add(W, -(ap * shift) * t.Sp);
            }
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        df_add(Sp, shfl_xor(Sp, m));
        df_add(Sq, shfl_xor(Sq, m));
        df_add(W, shfl_xor(W, m));
    }
    nanp = __any_sync(0xffffffffu, nanp);
    nanq = __any_sync(0xffffffffu, nanq);
    if (lane != 0) return;
    const double sp = df_value(Sp), sq = df_value(Sq), w = df_value(W);
    uint32_t fp = 0, fq = 0;
    if (nanp || sp != sp || Mp != Mp) fp |= kRowNanInf;
    else if (!(sp > 0.0)) fp |= kRowEmpty;
    if (nanq || sq != sq || Mq != Mq) fq |= kRowNanInf;
    else if (!(sq > 0.0)) fq |= kRowEmpty;
    const double logSp = log(sp), logSq = log(sq), c = w / sp;   // c = E_p[(P - m_P) - (Q - m_Q)]
    store_rowstat(stats_p + row, Mp, logSp, c, fp);
    store_rowstat(stats_q + row, Mq, logSq, 0.0, fq);
    kl[row] = (fp | fq) ? qnan() : (float)(c - logSp + logSq);
}

// ---------------------------------------------------------------------------
// Backward K1 epilogues: dz of a 256-column tile of a vocabulary chunk, bf16
// (round to nearest even), row-major [row][col] with pitch ldz; the gradient
// GEMMs read it in place. Rows without valid statistics get NaN.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store_dz32(__nv_bfloat16 *dst, const float (&d)[32]) {
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        __nv_bfloat162 b = __floats2bfloat162_rn(d[2 * i], d[2 * i + 1]);
        packed[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int k = 0; k < 4; ++k) d4[k] = make_uint4(packed[4 * k], packed[4 * k + 1], packed[4 * k + 2], packed[4 * k + 3]);
}

// Entropy: dz = -g p ((z - m) - c), c = W / S from the record (so that
// (z - m) - c = log p + H).
struct DzEntEpi {
    int N, ldz;
    const RowStat *stats;
    const float *g;
    __nv_bfloat16 *dz;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const RowStat s = load_rowstat(stats + (valid ? row : 0));
        const bool nan = (s.flags & (kRowNanInf | kRowEmpty)) != 0;
        const float gr = valid ? g[row] : 0.f;
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float t = v[i] - s.m;
                const float p = ex2_fast((t - s.logS_hi) * kLog2e);
                float x = p == 0.f ? 0.f : -gr * p * ((t - s.c_hi) - s.c_lo);
                if (c * 32 + i >= ncol) x = 0.f;
                else if (nan) x = qnan();
                v[i] = x;
            }
            if (valid) store_dz32(dz + (int64_t)row * ldz + col0 + c * 32, v);
        }
    }
};

// KL(P||Q): dP = g p ((tP - tQ) - c), dQ = g (q - p), tX = X - m_X, c from P's
// record; written to the dz of A and / or B (either may be null) by direction.
struct DzKLEpi {
    int N, ldz;
    bool p_is_a;
    const RowStat *sp, *sq;
    const float *g;
    __nv_bfloat16 *dza, *dzb;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const int r = valid ? row : 0;
        const RowStat P = load_rowstat(sp + r), Q = load_rowstat(sq + r);
        const bool nan = ((P.flags & (kRowNanInf | kRowEmpty)) | (Q.flags & kRowNanInf)) != 0;
        const float gr = valid ? g[row] : 0.f;
        const uint32_t tp = taddr + (p_is_a ? 0u : (uint32_t)kLBN), tq = taddr + (p_is_a ? (uint32_t)kLBN : 0u);
        __nv_bfloat16 *dzp = p_is_a ? dza : dzb, *dzq = p_is_a ? dzb : dza;
#pragma unroll 1
        for (int c = 0; c < kDualEpiCols / 32; ++c) {
            float a[32], b[32];
            tmem_ld32(tp + c * 32, a);
            tmem_ld32(tq + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float tP = a[i] - P.m, tQ = b[i] - Q.m;
                const float p = ex2_fast((tP - P.logS_hi) * kLog2e);
                const float q = ex2_fast((tQ - Q.logS_hi) * kLog2e);
                float dP = p == 0.f ? 0.f : gr * p * (((tP - tQ) - P.c_hi) - P.c_lo);
                float dQ = gr * (q - p);
                if (c * 32 + i >= ncol) dP = dQ = 0.f;
                else if (nan) dP = dQ = qnan();
                a[i] = dP;
                b[i] = dQ;
            }
            if (!valid) continue;
            const int64_t off = (int64_t)row * ldz + col0 + c * 32;
            if (dzp) store_dz32(dzp + off, a);
            if (dzq) store_dz32(dzq + off, b);
        }
    }
};

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int64_t n_vtiles(int64_t V) { return (V + kLBN - 1) / kLBN; }

size_t linear_entropy_workspace_bytes(int64_t N, int64_t V) {
    return up256((size_t)N * n_vtiles(V) * sizeof(EntTile));
}

cudaError_t launch_linear_entropy_fwd(const LinearEntArgs &a) {
    const int n_vt = (int)n_vtiles(a.V);
    EntTile *parts = static_cast<EntTile *>(a.workspace);
    const EntEpi epi{(int)a.N, n_vt, parts};
    cudaError_t e = launch_logits_gemm(a.hidden, a.weight, (int)a.N, (int)a.V, (int)a.D, epi, a.stream, kFwdPairs);
    if (e != cudaSuccess) return e;
    linear_entropy_merge_kernel<<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>((int)a.N, n_vt, parts, a.H,
                                                                                   static_cast<RowStat *>(a.stats));
    return cudaGetLastError();
}

size_t linear_entropy_bwd_workspace_bytes(int64_t N, int64_t V, int64_t D) {
    return up256((size_t)N * chunk_cols(N, V) * 2) + up256((size_t)N * D * 4);
}

cudaError_t launch_linear_entropy_bwd(const LinearEntArgs &a) {
    const int64_t vc = chunk_cols(a.N, a.V);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    __nv_bfloat16 *dz = reinterpret_cast<__nv_bfloat16 *>(ws);
    float *acc = a.dhidden ? reinterpret_cast<float *>(ws + up256((size_t)a.N * vc * 2)) : nullptr;
    const __nv_bfloat16 *h = static_cast<const __nv_bfloat16 *>(a.hidden);
    const __nv_bfloat16 *W = static_cast<const __nv_bfloat16 *>(a.weight);
    const int N = (int)a.N, V = (int)a.V, D = (int)a.D;
    cudaError_t e;
    CUtensorMap tm_h_mn;
    if (!make_map_mn(&tm_h_mn, h, N, D, D)) return cudaErrorInvalidValue;
    for (int64_t v0 = 0; v0 < V; v0 += vc) {
        const int nv = (int)(V - v0 < vc ? V - v0 : vc);
        const DzEntEpi de{N, (int)vc, static_cast<const RowStat *>(a.stats), a.g, dz};
        if ((e = launch_logits_gemm(h, W + v0 * D, N, nv, D, de, a.stream, kGemmPairs)) != cudaSuccess) return e;
        if ((e = chunk_gradient_gemms(tm_h_mn, W, N, D, v0, nv, vc, dz, acc, static_cast<__nv_bfloat16 *>(a.dW),
                                      a.stream)) != cudaSuccess)
            return e;
    }
    if (a.dhidden) return finish_dhidden(acc, (int64_t)N * D, static_cast<__nv_bfloat16 *>(a.dhidden), a.stream);
    return cudaSuccess;
}

// records of the dual epilogues: one per 128-column half tile (kDualEpiCols)
static int64_t n_dual_tiles(int64_t V) { return (V + kDualEpiCols - 1) / kDualEpiCols; }

size_t linear_kl_workspace_bytes(int64_t N, int64_t V) { return up256((size_t)N * n_dual_tiles(V) * sizeof(KLTile)); }

cudaError_t launch_linear_kl_fwd(const LinearKLArgs &a) {
    CUtensorMap tm_ha, tm_wa, tm_hb, tm_wb;
    if (!make_map(&tm_ha, a.ha, a.N, a.Da, a.Da, kLBM) || !make_map(&tm_wa, a.wa, a.V, a.Da, a.Da, kLBN) ||
        !make_map(&tm_hb, a.hb, a.N, a.Db, a.Db, kLBM) || !make_map(&tm_wb, a.wb, a.V, a.Db, a.Db, kLBN))
        return cudaErrorInvalidValue;
    const int n_vt = (int)n_dual_tiles(a.V);
    const bool p_is_a = a.direction == 0;
    KLTile *parts = static_cast<KLTile *>(a.workspace);
    const KLEpi epi{(int)a.N, n_vt, p_is_a, parts};
    cudaError_t e = launch_gemm_dual(tm_ha, tm_wa, tm_hb, tm_wb, (int)a.N, (int)a.V, (int)a.Da, (int)a.Db, epi,
                                     a.stream);
    if (e != cudaSuccess) return e;
    RowStat *sa = static_cast<RowStat *>(a.stats_a), *sb = static_cast<RowStat *>(a.stats_b);
    linear_kl_merge_kernel<<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>((int)a.N, n_vt, parts, a.kl,
                                                                              p_is_a ? sa : sb, p_is_a ? sb : sa);
    return cudaGetLastError();
}

// dz of A and of B for one chunk, then the fp32 dhidden accumulators of A and B.
size_t linear_kl_bwd_workspace_bytes(int64_t N, int64_t V, int64_t Da, int64_t Db) {
    const size_t dz = up256((size_t)N * chunk_cols(N, V) * 2);
    return 2 * dz + up256((size_t)N * Da * 4) + up256((size_t)N * Db * 4);
}

// Backward of a two-model op: per vocabulary chunk, the dual GEMM recomputes
// both logits tiles and the epilogue made by make_epi(dza, dzb) writes dz of A
// and / or B; then the gradient GEMMs of each model whose gradients are asked for.
template <class MakeEpi>
static cudaError_t two_model_bwd(const LinearKLArgs &a, MakeEpi make_epi) {
    const int64_t vc = chunk_cols(a.N, a.V);
    const size_t dz_bytes = up256((size_t)a.N * vc * 2);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    const bool want_a = a.dha || a.dwa, want_b = a.dhb || a.dwb;
    __nv_bfloat16 *dza = want_a ? reinterpret_cast<__nv_bfloat16 *>(ws) : nullptr;
    __nv_bfloat16 *dzb = want_b ? reinterpret_cast<__nv_bfloat16 *>(ws + dz_bytes) : nullptr;
    float *acc_a = a.dha ? reinterpret_cast<float *>(ws + 2 * dz_bytes) : nullptr;
    float *acc_b = a.dhb ? reinterpret_cast<float *>(ws + 2 * dz_bytes + up256((size_t)a.N * a.Da * 4)) : nullptr;
    const __nv_bfloat16 *ha = static_cast<const __nv_bfloat16 *>(a.ha), *hb = static_cast<const __nv_bfloat16 *>(a.hb);
    const __nv_bfloat16 *Wa = static_cast<const __nv_bfloat16 *>(a.wa), *Wb = static_cast<const __nv_bfloat16 *>(a.wb);
    const int N = (int)a.N, V = (int)a.V, Da = (int)a.Da, Db = (int)a.Db;
    cudaError_t e;
    CUtensorMap tm_ha, tm_hb, tm_ha_mn, tm_hb_mn;
    if (!make_map(&tm_ha, ha, N, Da, Da, kLBM) || !make_map(&tm_hb, hb, N, Db, Db, kLBM) ||
        !make_map_mn(&tm_ha_mn, ha, N, Da, Da) || !make_map_mn(&tm_hb_mn, hb, N, Db, Db))
        return cudaErrorInvalidValue;
    for (int64_t v0 = 0; v0 < V; v0 += vc) {
        const int nv = (int)(V - v0 < vc ? V - v0 : vc);
        CUtensorMap tm_wac, tm_wbc;
        if (!make_map(&tm_wac, Wa + v0 * Da, nv, Da, Da, kLBN) || !make_map(&tm_wbc, Wb + v0 * Db, nv, Db, Db, kLBN))
            return cudaErrorInvalidValue;
        const auto de = make_epi((int)vc, dza, dzb);
        if ((e = launch_gemm_dual(tm_ha, tm_wac, tm_hb, tm_wbc, N, nv, Da, Db, de, a.stream)) != cudaSuccess) return e;
        if (want_a && (e = chunk_gradient_gemms(tm_ha_mn, Wa, N, Da, v0, nv, vc, dza, acc_a,
                                                static_cast<__nv_bfloat16 *>(a.dwa), a.stream)) != cudaSuccess)
            return e;
        if (want_b && (e = chunk_gradient_gemms(tm_hb_mn, Wb, N, Db, v0, nv, vc, dzb, acc_b,
                                                static_cast<__nv_bfloat16 *>(a.dwb), a.stream)) != cudaSuccess)
            return e;
    }
    if (a.dha && (e = finish_dhidden(acc_a, (int64_t)N * Da, static_cast<__nv_bfloat16 *>(a.dha), a.stream)) !=
                     cudaSuccess)
        return e;
    if (a.dhb) return finish_dhidden(acc_b, (int64_t)N * Db, static_cast<__nv_bfloat16 *>(a.dhb), a.stream);
    return cudaSuccess;
}

cudaError_t launch_linear_kl_bwd(const LinearKLArgs &a) {
    const bool p_is_a = a.direction == 0;
    const RowStat *sa = static_cast<const RowStat *>(a.stats_a), *sb = static_cast<const RowStat *>(a.stats_b);
    return two_model_bwd(a, [&](int ldz, __nv_bfloat16 *dza, __nv_bfloat16 *dzb) {
        return DzKLEpi{(int)a.N, ldz, p_is_a, p_is_a ? sa : sb, p_is_a ? sb : sa, a.g, dza, dzb};
    });
}

// ---------------------------------------------------------------------------
// Generalized JSD of two models, interior beta ([P1], the commit message adding
// vocab_parallel_jsd: "Motivation" names teacher-student divergences computed
// from tiled LM-head projections, "Changes" the two passes: global
// normalisation first, then both KL-to-mixture expectations together).
//   pass 1  the KL forward's dual GEMM and merge: each row's exact maxima and
//           log-sums of A and B in the two records;
//   pass 2  the dual GEMM again; the epilogue (JsdEpi) forms log p, log q and
//           log mix (mix = beta q + (1 - beta) p) in base-2 units and sums
//           p (log p - log mix) and q (log q - log mix) per tile; a merge per
//           row adds the tiles, writes JSD = beta KL(q||mix) + (1 - beta)
//           KL(p||mix) and keeps the two expectations in the records' c fields;
//   backward  the dual GEMM, dA = g (1 - beta) p ((log p - log mix) - KL(p||mix))
//           and dB = g beta q ((log q - log mix) - KL(q||mix)) in the epilogue
//           (DzJsdEpi), then the gradient GEMMs of each model asked for.
// ---------------------------------------------------------------------------
struct JsdTile {
    float kp, kq;   // sum p (log2 p - log2 mix), sum q (log2 q - log2 mix) over the tile
};

struct JsdEpi {
    int N, n_vt;
    float beta;
    const RowStat *sa, *sb;   // records of pass 1
    JsdTile *parts;           // [N][n_vt]
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const int r = valid ? row : 0;
        const RowStat A = load_rowstat(sa + r), B = load_rowstat(sb + r);
        const float omb = 1.f - beta;
        float kp = 0.f, kq = 0.f;
#pragma unroll 1
        for (int c = 0; c < kDualEpiCols / 32; ++c) {
            float a[32], b[32];
            tmem_ld32(taddr + c * 32, a);
            tmem_ld32(taddr + kLBN + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (c * 32 + i >= ncol) continue;
                const float xa = ((a[i] - A.m) - A.logS_hi) * kLog2e;   // log2 p
                const float xb = ((b[i] - B.m) - B.logS_hi) * kLog2e;   // log2 q
                const float p = ex2_fast(xa), q = ex2_fast(xb);
                const float lm = fmaxf(lg2_fast(fmaf(beta, q, omb * p)), -250.f);
                if (p > 0.f) kp = fmaf(p, xa - lm, kp);                  // zero-weight terms add nothing
                if (q > 0.f) kq = fmaf(q, xb - lm, kq);
            }
        }
        if (!valid) return;
        parts[(int64_t)row * n_vt + col0 / kDualEpiCols] = JsdTile{kp, kq};
    }
};

__global__ void __launch_bounds__(256)
linear_jsd_merge_kernel(int N, int n_vt, float beta, const JsdTile *__restrict__ parts, float *__restrict__ jsd,
                        RowStat *__restrict__ sa, RowStat *__restrict__ sb) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const JsdTile *p = parts + (int64_t)row * n_vt;
    DF kp{0.f, 0.f}, kq{0.f, 0.f};
    for (int i = lane; i < n_vt; i += 32) {
        df_add(kp, p[i].kp);
        df_add(kq, p[i].kq);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        df_add(kp, shfl_xor(kp, m));
        df_add(kq, shfl_xor(kq, m));
    }
    if (lane != 0) return;
    const double ln2 = 0.69314718055994530942;
    const double KLp = df_value(kp) * ln2, KLq = df_value(kq) * ln2;
    const bool bad = ((sa[row].flags | sb[row].flags) & (kRowNanInf | kRowEmpty)) != 0;
    const DF cp = df_from(KLp), cq = df_from(KLq);
    sa[row].c_hi = cp.hi;
    sa[row].c_lo = cp.lo;
    sb[row].c_hi = cq.hi;
    sb[row].c_lo = cq.lo;
    jsd[row] = bad ? qnan() : (float)((double)beta * KLq + (1.0 - (double)beta) * KLp);
}

struct DzJsdEpi {
    int N, ldz;
    float beta;
    const RowStat *sa, *sb;
    const float *g;
    __nv_bfloat16 *dza, *dzb;   // either may be null
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const int r = valid ? row : 0;
        const RowStat A = load_rowstat(sa + r), B = load_rowstat(sb + r);
        const bool nan = ((A.flags | B.flags) & (kRowNanInf | kRowEmpty)) != 0;
        const float gr = valid ? g[row] : 0.f, omb = 1.f - beta;
        const float ka = A.c_hi + A.c_lo, kb = B.c_hi + B.c_lo;   // KL(p||mix), KL(q||mix)
        const float ln2 = 0.69314718055994530942f;
#pragma unroll 1
        for (int c = 0; c < kDualEpiCols / 32; ++c) {
            float a[32], b[32];
            tmem_ld32(taddr + c * 32, a);
            tmem_ld32(taddr + kLBN + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float la = (a[i] - A.m) - A.logS_hi, lb = (b[i] - B.m) - B.logS_hi;   // log p, log q
                const float p = ex2_fast(la * kLog2e), q = ex2_fast(lb * kLog2e);
                const float lmix = fmaxf(lg2_fast(fmaf(beta, q, omb * p)), -250.f) * ln2;
                float dA = p == 0.f ? 0.f : gr * omb * p * ((la - lmix) - ka);
                float dB = q == 0.f ? 0.f : gr * beta * q * ((lb - lmix) - kb);
                if (c * 32 + i >= ncol) dA = dB = 0.f;
                else if (nan) dA = dB = qnan();
                a[i] = dA;
                b[i] = dB;
            }
            if (!valid) continue;
            const int64_t off = (int64_t)row * ldz + col0 + c * 32;
            if (dza) store_dz32(dza + off, a);
            if (dzb) store_dz32(dzb + off, b);
        }
    }
};

cudaError_t launch_linear_jsd_fwd(const LinearKLArgs &a) {
    // pass 1: the records (the KL forward; its KL output is overwritten below)
    LinearKLArgs k = a;
    k.direction = 0;
    cudaError_t e = launch_linear_kl_fwd(k);
    if (e != cudaSuccess) return e;
    // pass 2: both KL-to-mixture expectations (the workspace is free again)
    CUtensorMap tm_ha, tm_wa, tm_hb, tm_wb;
    if (!make_map(&tm_ha, a.ha, a.N, a.Da, a.Da, kLBM) || !make_map(&tm_wa, a.wa, a.V, a.Da, a.Da, kLBN) ||
        !make_map(&tm_hb, a.hb, a.N, a.Db, a.Db, kLBM) || !make_map(&tm_wb, a.wb, a.V, a.Db, a.Db, kLBN))
        return cudaErrorInvalidValue;
    const int n_vt = (int)n_dual_tiles(a.V);
    RowStat *sa = static_cast<RowStat *>(a.stats_a), *sb = static_cast<RowStat *>(a.stats_b);
    JsdTile *parts = static_cast<JsdTile *>(a.workspace);
    const JsdEpi epi{(int)a.N, n_vt, a.beta, sa, sb, parts};
    e = launch_gemm_dual(tm_ha, tm_wa, tm_hb, tm_wb, (int)a.N, (int)a.V, (int)a.Da, (int)a.Db, epi, a.stream);
    if (e != cudaSuccess) return e;
    linear_jsd_merge_kernel<<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>((int)a.N, n_vt, a.beta, parts, a.kl, sa,
                                                                               sb);
    return cudaGetLastError();
}

cudaError_t launch_linear_jsd_bwd(const LinearKLArgs &a) {
    const RowStat *sa = static_cast<const RowStat *>(a.stats_a), *sb = static_cast<const RowStat *>(a.stats_b);
    return two_model_bwd(a, [&](int ldz, __nv_bfloat16 *dza, __nv_bfloat16 *dzb) {
        return DzJsdEpi{(int)a.N, ldz, a.beta, sa, sb, a.g, dza, dzb};
    });
}

cudaError_t read_linear_ent_kl_fault(uint32_t *value, bool clear) { return read_tu_fault(value, clear); }

}  // namespace vp
