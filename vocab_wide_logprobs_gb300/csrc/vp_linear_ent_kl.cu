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
//   forward   the dual GEMM (on CTA pairs) puts the same tile of both models'
//             logits in TMEM, P's model first; the epilogue (KLEpi) takes P's
//             columns into registers at once (freeing them for the next tile)
//             and, with Q's columns, the tile's maxima of P and Q, S_P, S_Q and
//             W = sum e^{P - m_P} ((P - m_P) - (Q - m_Q)); the merge re-centres
//             the tiles (W_i -> alpha_i (W_i - (dP_i - dQ_i) S_P,i)) and writes
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
        // each 32-column chunk summed in fp32, the chunks folded into double-floats
        DF S{0.f, 0.f}, W{0.f, 0.f};
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            float s0 = 0.f, s1 = 0.f, w0 = 0.f, w1 = 0.f;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float t0 = v[i] - m, t1 = v[i + 1] - m;
                const float e0 = c * 32 + i < ncol ? exp_fwd(t0) : 0.f;
                const float e1 = c * 32 + i + 1 < ncol ? exp_fwd(t1) : 0.f;
                s0 += e0;
                s1 += e1;
                w0 = e0 == 0.f ? w0 : fmaf(e0, t0, w0);   // zero-weight terms add nothing
                w1 = e1 == 0.f ? w1 : fmaf(e1, t1, w1);
            }
            df_add(S, s0 + s1);
            df_add(W, w0 + w1);
        }
        if (row >= N) return;
        parts[(int64_t)row * n_vt + col0 / kLBN] = EntTile{m, S.hi + S.lo, W.hi + W.lo, 0.f};
    }
};

struct KLTile {
    float mp, Sp, mq, Sq, W, pad0, pad1, pad2;
};

// Packed helpers of the dual-form full-tile paths: two columns per fp32
// instruction (f32x2), a three-input max for the tile maxima.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float max32(float m, const float (&v)[32]) {
    float m0 = m, m1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        m0 = max3f(m0, v[i], v[i + 1]);
        m1 = max3f(m1, v[i + 2], v[i + 3]);
    }
    return fmaxf(m0, m1);
}
__device__ __forceinline__ float2 splat(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 pair_at(const float (&v)[32], int i) { return make_float2(v[i], v[i + 1]); }
__device__ __forceinline__ float2 ex2_pair(float2 x) { return make_float2(ex2_fast(x.x), ex2_fast(x.y)); }
__device__ __forceinline__ float2 lg2_pair(float2 x) { return make_float2(lg2_fast(x.x), lg2_fast(x.y)); }
__device__ __forceinline__ bool finite(float x) { return fabsf(x) < INFINITY; }

__device__ __forceinline__ float2 pair128(const float (&v)[128], int i) { return make_float2(v[i], v[i + 1]); }

// q - p from p and d = log q - log p: p (e^d - 1) where |d| < 1/2 (q ~ p, where
// the difference of the two exponentials would cancel), else q - p
__device__ __forceinline__ float q_minus_p(float q, float p, float d) {
    return fabsf(d) < 0.5f ? p * expm1_small(d) : q - p;
}

// Dual-form epilogues: x holds the thread's 128 columns (one half of the
// tile) of the first product, model A, already out of TMEM; tb is the TMEM
// address of the same columns of the second product, model B, read here in
// 32-column chunks.
// KL(P||Q) with P the first product (the launcher puts the P model first).
struct KLEpi {
    int N, n_vt;
    KLTile *parts;    // [N][n_vt]

    // any tile: columns past ncol left out, zero-weight terms skipped
    __device__ __forceinline__ KLTile checked(int ncol, const float (&x)[128], uint32_t tb) const {
        float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i < ncol) {
                    ma = fmaxf(ma, x[c * 32 + i]);
                    mb = fmaxf(mb, b[i]);
                }
        }
        const float mp = ma, mq = mb;
        DF SP{0.f, 0.f}, SQ{0.f, 0.f}, WW{0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
            float sp = 0.f, sq = 0.f, w = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const bool in = c * 32 + i < ncol;
                const float vp = x[c * 32 + i], vq = b[i];
                const float tP = vp - mp, tQ = vq - mq;
                const float ep = in ? exp_fwd(tP) : 0.f;
                const float eq = in ? exp_fwd(tQ) : 0.f;
                sp += ep;
                sq += eq;
                w = ep == 0.f ? w : fmaf(ep, tP - tQ, w);
            }
            df_add(SP, sp);
            df_add(SQ, sq);
            df_add(WW, w);
        }
        return KLTile{mp, SP.hi + SP.lo, mq, SQ.hi + SQ.lo, WW.hi + WW.lo, 0.f, 0.f, 0.f};
    }

    // a full tile, two columns per instruction and no per-column tests: a zero
    // weight times an infinite (tP - tQ) makes W NaN, and such a tile is redone
    // by checked()
    __device__ __forceinline__ KLTile full(const float (&x)[128], uint32_t tb) const {
        float ma0 = -INFINITY, ma1 = -INFINITY;
#pragma unroll
        for (int i = 0; i < 128; i += 4) {
            ma0 = max3f(ma0, x[i], x[i + 1]);
            ma1 = max3f(ma1, x[i + 2], x[i + 3]);
        }
        const float ma = fmaxf(ma0, ma1);
        float mb = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
            mb = max32(mb, b);
        }
        const float2 nma = splat(-ma), nmb = splat(-mb), m1 = splat(-1.f);
        // each 32-column chunk summed in fp32 (f32x2), the chunks folded into double-floats
        DF SA{0.f, 0.f}, SB{0.f, 0.f}, WW{0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
            float2 sa[2] = {splat(0.f), splat(0.f)}, sb[2] = {splat(0.f), splat(0.f)}, w[2] = {splat(0.f), splat(0.f)};
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const int k = (i >> 1) & 1;
                const float2 tA = __fadd2_rn(pair128(x, c * 32 + i), nma), tB = __fadd2_rn(pair_at(b, i), nmb);
                const float2 eA = exp_fwd2(tA), eB = exp_fwd2(tB);
                sa[k] = __fadd2_rn(sa[k], eA);
                sb[k] = __fadd2_rn(sb[k], eB);
                w[k] = __ffma2_rn(eA, __ffma2_rn(tB, m1, tA), w[k]);   // e_P (tP - tQ)
            }
            const float2 a2 = __fadd2_rn(sa[0], sa[1]), b2 = __fadd2_rn(sb[0], sb[1]), w2 = __fadd2_rn(w[0], w[1]);
            df_add(SA, a2.x + a2.y);
            df_add(SB, b2.x + b2.y);
            df_add(WW, w2.x + w2.y);
        }
        return KLTile{ma, SA.hi + SA.lo, mb, SB.hi + SB.lo, WW.hi + WW.lo, 0.f, 0.f, 0.f};
    }

    __device__ __forceinline__ void operator()(int row, int col0, int ncol, const float (&x)[128], uint32_t tb) const {
        KLTile t;
        if (ncol == kDualEpiCols) {                 // warp-uniform: the tile's columns
            t = full(x, tb);
            const bool redo = !finite(t.W);
            if (__any_sync(0xffffffffu, redo)) {    // TMEM loads are warp-collective
                const KLTile u = checked(ncol, x, tb);
                if (redo) t = u;
            }
        } else {
            t = checked(ncol, x, tb);
        }
        if (row >= N) return;
        parts[(int64_t)row * n_vt + col0 / kDualEpiCols] = t;
    }
};

// ---------------------------------------------------------------------------
// Merges: one warp per row, the row's tiles in a fixed order (lane-strided,
// then a fixed shuffle tree), fp32 exponentials summed as double-floats, fp64
// finish; the result depends on V only, not on N (batch invariance).
// ---------------------------------------------------------------------------
// kPart: the row's record over this vocabulary shard (vp_partial: m, S, W
// about m, flags) instead of H and the row statistics.
template <bool kPart>
__global__ void __launch_bounds__(256)
linear_entropy_merge_kernel(int N, int n_vt, const EntTile *__restrict__ parts, float *__restrict__ H,
                            RowStat *__restrict__ stats, PartialRec *__restrict__ shard_parts) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const EntTile *p = parts + (int64_t)row * n_vt;
    // tiles lane, lane + 32, ... in that order, four loads issued together
    constexpr int kB = 4;
    const EntTile empty{-INFINITY, 0.f, 0.f, 0.f};
    float M = -INFINITY;
    for (int i0 = lane; i0 < n_vt; i0 += 32 * kB) {
        float m[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) m[u] = i0 + 32 * u < n_vt ? p[i0 + 32 * u].m : -INFINITY;
#pragma unroll
        for (int u = 0; u < kB; ++u) M = fmaxf(M, m[u]);
    }
    M = warp_max(M);
    DF S{0.f, 0.f}, W{0.f, 0.f};
    bool nan = false;
    for (int i0 = lane; i0 < n_vt; i0 += 32 * kB) {
        EntTile tt[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) tt[u] = i0 + 32 * u < n_vt ? p[i0 + 32 * u] : empty;
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const EntTile &t = tt[u];
            if (t.S != t.S || t.W != t.W || t.m == INFINITY) { nan = true; continue; }
            if (!(t.S > 0.f)) continue;                       // zero-weight tile
            const float a = expf(t.m - M);
            if (a == 0.f) continue;
            df_add(S, a * t.S);
            df_add(W, a * fmaf(-(M - t.m), t.S, t.W));        // both terms <= 0
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        df_add(S, shfl_xor(S, m));
        df_add(W, shfl_xor(W, m));
    }
    nan = __any_sync(0xffffffffu, nan);
    if (lane != 0) return;
    const double s = df_value(S), w = df_value(W);
    if constexpr (kPart) {
        shard_parts[row] = PartialRec{s > 0.0 ? M : kNegBig, 0.f, s, 0.0, w, 0.f, (nan || s != s) ? kPartNanInf : 0u};
        return;
    }
    uint32_t flags = 0;
    if (nan || s != s || M != M) flags |= kRowNanInf;
    else if (!(s > 0.0)) flags |= kRowEmpty;
    const double logS = log(s), c = w / s;
    store_rowstat(stats + row, M, logS, c, flags);
    H[row] = flags ? qnan() : (float)(logS - c);
}

// s *= a for a double-float and a float a in [0, 1] (the product's rounding
// error kept in lo).
__device__ __forceinline__ void df_scale(DF &s, float a) {
    const float hi = s.hi * a;
    s.lo = fmaf(s.lo, a, fmaf(s.hi, a, -hi));
    s.hi = hi;
}

// Moves KL sums (S_P, S_Q and W about the centres (cp, cq)) to the centres
// (np, nq) >= (cp, cq): S_P *= e^{cp - np}, S_Q *= e^{cq - nq} and
// W -> e^{cp - np} (W - ((np - cp) - (nq - cq)) S_P) (the merge rule of the
// KL records). Sums about -inf centres are empty and only take the new centres.
__device__ __forceinline__ void kl_recentre(DF &Sp, DF &Sq, DF &W, float &cp, float &cq, float np, float nq) {
    if (cp != -INFINITY) {
        const float dp = np - cp, dq = cq != -INFINITY ? nq - cq : 0.f;
        df_add(W, -((dp - dq) * Sp.hi));
        const float a = expf(-dp);
        df_scale(W, a);
        df_scale(Sp, a);
    }
    if (cq != -INFINITY) df_scale(Sq, expf(cq - nq));
    cp = np;
    cq = nq;
}

// kPart: the row's record over this vocabulary shard (vp_partial: both
// maxima and sum-exps, W about the maxima, flags) instead of KL and the records.
template <bool kPart>
__global__ void __launch_bounds__(256)
linear_kl_merge_kernel(int N, int n_vt, const KLTile *__restrict__ parts, float *__restrict__ kl,
                       RowStat *__restrict__ stats_p, RowStat *__restrict__ stats_q,
                       PartialRec *__restrict__ shard_parts) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const KLTile *p = parts + (int64_t)row * n_vt;
    // One pass: each lane takes tiles lane, lane + 32, ... in that order (four
    // loads in flight; an absent tile reads as an empty one) and keeps its sums
    // about its own centres (cp, cq), the maxima of the tiles it has added so
    // far, moving them up when a tile brings a larger maximum; the lanes' sums
    // are then moved to the warp's centres and added in a fixed shuffle tree.
    constexpr int kB = 4;
    const KLTile empty{-INFINITY, 0.f, -INFINITY, 0.f, 0.f, 0.f, 0.f, 0.f};
    float Mp = -INFINITY, Mq = -INFINITY;   // maxima over every tile: the records' m
    float cp = -INFINITY, cq = -INFINITY;   // this lane's centres
    DF Sp{0.f, 0.f}, Sq{0.f, 0.f}, W{0.f, 0.f};
    bool nanp = false, nanq = false;
    for (int i0 = lane; i0 < n_vt; i0 += 32 * kB) {
        KLTile tt[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) tt[u] = i0 + 32 * u < n_vt ? p[i0 + 32 * u] : empty;
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const KLTile &t = tt[u];
            Mp = fmaxf(Mp, t.mp);
            Mq = fmaxf(Mq, t.mq);
            const bool bp = t.Sp != t.Sp || t.W != t.W || t.mp == INFINITY;
            const bool bq = t.Sq != t.Sq || t.mq == INFINITY;
            nanp |= bp;
            nanq |= bq;
            if (bp || bq || !(t.Sp > 0.f || t.Sq > 0.f)) continue;
            if (t.mp > cp || t.mq > cq) kl_recentre(Sp, Sq, W, cp, cq, fmaxf(cp, t.mp), fmaxf(cq, t.mq));
            if (t.Sq > 0.f) {
                const float aq = expf(t.mq - cq);
                if (aq != 0.f) df_add(Sq, aq * t.Sq);
            }
            if (t.Sp > 0.f) {
                const float ap = expf(t.mp - cp);
                if (ap != 0.f) {
                    df_add(Sp, ap * t.Sp);
                    // W_i about the centres: W_i - ((cp - mp_i) - (cq - mq_i)) S_P,i
                    const float shift = (cp - t.mp) - (cq - t.mq);
                    df_add(W, ap * t.W);
                    df_add(W, -(ap * shift) * t.Sp);
                }
            }
        }
    }
    Mp = warp_max(Mp);
    Mq = warp_max(Mq);
    const float wp = warp_max(cp), wq = warp_max(cq);   // the warp's centres
    if (cp < wp || cq < wq) kl_recentre(Sp, Sq, W, cp, cq, wp, wq);
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
    if constexpr (kPart) {
        const uint32_t pf = ((nanp || sp != sp) ? kPartNanInf : 0u) | ((nanq || sq != sq) ? kPartNanInfB : 0u);
        shard_parts[row] = PartialRec{sp > 0.0 ? Mp : kNegBig, sq > 0.0 ? Mq : kNegBig, sp, sq, w, 0.f, pf};
        return;
    }
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
// (round to nearest even), row-major [row][col] with pitch ldz, and with
// lo_off != 0 the remainder at dz + lo_off (store_dz); the gradient GEMMs read
// both in place. Rows without valid statistics get NaN.
// ---------------------------------------------------------------------------

// Entropy: dz = -g p ((z - m) - c), c = W / S from the record (so that
// (z - m) - c = log p + H), taken as (z - K_hi) - K_lo with K = m + c as a
// double-float: where z ~ K the first difference is exact, so dz keeps its
// relative accuracy where it cancels.
struct DzEntEpi {
    int N, ldz;
    const RowStat *stats;
    const float *g;
    __nv_bfloat16 *dz;
    int64_t lo_off;
    __device__ __forceinline__ void operator()(int row, int col0, int ncol, uint32_t taddr) const {
        const bool valid = row < N;
        const RowStat s = load_rowstat(stats + (valid ? row : 0));
        const bool nan = (s.flags & (kRowNanInf | kRowEmpty)) != 0;
        const float gr = valid ? g[row] : 0.f;
        const DF K = df_from((double)s.m + ((double)s.c_hi + (double)s.c_lo));
#pragma unroll 1
        for (int c = 0; c < kLBN / 32; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float t = v[i] - s.m;
                const float p = ex2_fast((t - s.logS_hi) * kLog2e);
                float x = p == 0.f ? 0.f : -gr * p * ((v[i] - K.hi) - K.lo);
                if (c * 32 + i >= ncol) x = 0.f;
                else if (nan) x = qnan();
                v[i] = x;
            }
            if (valid) store_dz(dz + (int64_t)row * ldz + col0 + c * 32, v, lo_off);
        }
    }
};

// KL(P||Q): dP = g p ((tP - tQ) - c), dQ = g (q - p), tX = X - m_X, c from P's
// record; written to the dz of A and / or B (either may be null) by direction.

// KL(P||Q) with P the first product (the launcher puts the P model first);
// dzp, dzq: the dz of P and of Q, either may be null.
struct DzKLEpi {
    int N, ldz;
    const RowStat *sp, *sq;
    const float *g;
    __nv_bfloat16 *dzp, *dzq;
    int64_t lo_off;

    // columns j0 .. j0 + 7 of the half tile (x[j0 + u], b[i0 + u]) with the
    // per-column tests: columns past ncol give 0, zero-weight terms give 0,
    // NaN rows give NaN
    __device__ __forceinline__ void checked(int j0, int i0, int ncol, bool nan, float gr, const RowStat &P,
                                            const RowStat &Q, const DF &KP, const DF &KQ, const float (&x)[128],
                                            const float (&b)[32], float (&oa)[8], float (&ob)[8]) const {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float vp = x[j0 + u], vq = b[i0 + u];
            const float tP = vp - P.m, tQ = vq - Q.m;
            const float p = ex2_fast((tP - P.logS_hi) * kLog2e);
            const float q = ex2_fast((tQ - Q.logS_hi) * kLog2e);
            const DF s = two_sum(vp, -vq);                           // vp - vq exactly
            float dP = p == 0.f ? 0.f : gr * p * (((s.hi - KP.hi) - KP.lo) + s.lo);
            float dQ = gr * q_minus_p(q, p, ((KQ.hi - s.hi) + KQ.lo) - s.lo);
            if (j0 + u >= ncol) dP = dQ = 0.f;
            else if (nan) dP = dQ = qnan();
            oa[u] = dP;
            ob[u] = dQ;
        }
    }

    __device__ __forceinline__ void operator()(int row, int col0, int ncol, const float (&x)[128], uint32_t tb) const {
        const bool valid = row < N;
        const int r = valid ? row : 0;
        const RowStat P = load_rowstat(sp + r), Q = load_rowstat(sq + r);
        const bool nan = ((P.flags & (kRowNanInf | kRowEmpty)) | (Q.flags & kRowNanInf)) != 0;
        const float gr = valid ? g[row] : 0.f;
        const bool full = ncol == kDualEpiCols;
        const float2 nPm = splat(-P.m), nQm = splat(-Q.m), l2e = splat(kLog2e), m1 = splat(-1.f);
        const float2 nCp = splat(-P.logS_hi * kLog2e), nCq = splat(-Q.logS_hi * kLog2e);
        const float2 g2 = splat(gr);
        // with s = vp - vq (exactly, as a double-float): (tP - tQ) - c = s - KP and
        // log q - log p = KQ - s, KP = (m_P - m_Q) + c, KQ = (m_P - m_Q) + (log S_P - log S_Q);
        // where either cancels, s and the constant are close and their difference is exact
        const double dm = (double)P.m - (double)Q.m;
        const DF KP = df_from(dm + ((double)P.c_hi + (double)P.c_lo));
        const DF KQ = df_from(dm + (((double)P.logS_hi + (double)P.logS_lo) - ((double)Q.logS_hi + (double)Q.logS_lo)));
        const float2 nkph = splat(-KP.hi), nkpl = splat(-KP.lo), kqh = splat(KQ.hi), kql = splat(KQ.lo);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
                const int i0 = gq * 8, j0 = c * 32 + i0;
                // two columns per instruction, no per-column tests; a zero p
                // times an infinite (tP - tQ - c) leaves the group's sum
                // non-finite, and such a group is redone with the tests
                float oa[8], ob[8];
                float2 chk = splat(0.f);
#pragma unroll
                for (int u = 0; u < 8; u += 2) {
                    const float2 vp = pair128(x, j0 + u), vq = pair_at(b, i0 + u);
                    const float2 tP = __fadd2_rn(vp, nPm), tQ = __fadd2_rn(vq, nQm);
                    const float2 p = ex2_pair(__ffma2_rn(tP, l2e, nCp)), q = ex2_pair(__ffma2_rn(tQ, l2e, nCq));
                    // s + e = vp - vq exactly (two-sum)
                    const float2 s = __ffma2_rn(vq, m1, vp);
                    const float2 bb = __ffma2_rn(vp, m1, s);
                    const float2 e = __ffma2_rn(__fadd2_rn(vq, bb), m1, __ffma2_rn(__ffma2_rn(bb, m1, s), m1, vp));
                    const float2 d = __fadd2_rn(__fadd2_rn(__fadd2_rn(s, nkph), nkpl), e);         // (tP - tQ) - c
                    chk = __fadd2_rn(chk, d);
                    // q - p, as p (e^dd - 1) where q ~ p (q_minus_p)
                    const float2 dd = __ffma2_rn(e, m1, __fadd2_rn(__ffma2_rn(s, m1, kqh), kql));    // log q - log p
                    const float2 em = __fmul2_rn(p, expm1_small2(dd));
                    float2 qp = __ffma2_rn(p, m1, q);
                    qp.x = fabsf(dd.x) < 0.5f ? em.x : qp.x;
                    qp.y = fabsf(dd.y) < 0.5f ? em.y : qp.y;
                    const float2 dP = __fmul2_rn(__fmul2_rn(g2, p), d), dQ = __fmul2_rn(g2, qp);
                    oa[u] = dP.x;
                    oa[u + 1] = dP.y;
                    ob[u] = dQ.x;
                    ob[u + 1] = dQ.y;
                }
                if (!full || nan || !finite(chk.x + chk.y)) checked(j0, i0, ncol, nan, gr, P, Q, KP, KQ, x, b, oa, ob);
                if (!valid) continue;
                const int64_t off = (int64_t)row * ldz + col0 + j0;
                if (dzp) store_dz(dzp + off, oa, lo_off);
                if (dzq) store_dz(dzq + off, ob, lo_off);
            }
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
    if (a.parts)
        linear_entropy_merge_kernel<true><<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
            (int)a.N, n_vt, parts, nullptr, nullptr, static_cast<PartialRec *>(a.parts));
    else
        linear_entropy_merge_kernel<false><<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
            (int)a.N, n_vt, parts, a.H, static_cast<RowStat *>(a.stats), nullptr);
    return cudaGetLastError();
}

// dz of one chunk twice over (hi and lo halves of the exact form), then the
// fp32 dhidden accumulator
size_t linear_entropy_bwd_workspace_bytes(int64_t N, int64_t V, int64_t D) {
    return up256((size_t)2 * N * chunk_cols(N, V) * 2) + up256((size_t)N * D * 4);
}

cudaError_t launch_linear_entropy_bwd(const LinearEntArgs &a) {
    const int64_t vc = chunk_cols(a.N, a.V);
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    __nv_bfloat16 *dz = reinterpret_cast<__nv_bfloat16 *>(ws);
    const int64_t lo_off = a.precision == VP_GRAD_EXACT_ ? a.N * vc : 0;   // dz_lo follows dz_hi
    float *acc = a.dhidden ? reinterpret_cast<float *>(ws + up256((size_t)2 * a.N * vc * 2)) : nullptr;
    const __nv_bfloat16 *h = static_cast<const __nv_bfloat16 *>(a.hidden);
    const __nv_bfloat16 *W = static_cast<const __nv_bfloat16 *>(a.weight);
    const int N = (int)a.N, V = (int)a.V, D = (int)a.D;
    cudaError_t e;
    CUtensorMap tm_h_mn;
    if (!make_map_mn(&tm_h_mn, h, N, D, D)) return cudaErrorInvalidValue;
    for (int64_t v0 = 0; v0 < V; v0 += vc) {
        const int nv = (int)(V - v0 < vc ? V - v0 : vc);
        const DzEntEpi de{N, (int)vc, static_cast<const RowStat *>(a.stats), a.g, dz, lo_off};
        if ((e = launch_logits_gemm(h, W + v0 * D, N, nv, D, de, a.stream, kGemmPairs)) != cudaSuccess) return e;
        if ((e = chunk_gradient_gemms(tm_h_mn, W, N, D, v0, nv, vc, dz, lo_off ? dz + lo_off : nullptr, acc,
                                      static_cast<__nv_bfloat16 *>(a.dhidden), static_cast<__nv_bfloat16 *>(a.dW),
                                      v0 + vc >= V, a.stream)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

// records of the dual epilogues: one per 128-column half tile (kDualEpiCols)
static int64_t n_dual_tiles(int64_t V) { return (V + kDualEpiCols - 1) / kDualEpiCols; }

size_t linear_kl_workspace_bytes(int64_t N, int64_t V) { return up256((size_t)N * n_dual_tiles(V) * sizeof(KLTile)); }

cudaError_t launch_linear_kl_fwd(const LinearKLArgs &a) {
    CUtensorMap tm_ha, tm_wa, tm_hb, tm_wb;
    if (!make_map(&tm_ha, a.ha, a.N, a.Da, a.Da, kLBM) || !make_map(&tm_wa, a.wa, a.V, a.Da, a.Da, kPBHalf) ||
        !make_map(&tm_hb, a.hb, a.N, a.Db, a.Db, kLBM) || !make_map(&tm_wb, a.wb, a.V, a.Db, a.Db, kPBHalf))
        return cudaErrorInvalidValue;
    const int n_vt = (int)n_dual_tiles(a.V);
    const bool p_is_a = a.direction == 0;
    KLTile *parts = static_cast<KLTile *>(a.workspace);
    // P first: the forward direction, KL(B||A), runs the dual GEMM with model B first
    const int N = (int)a.N, V = (int)a.V, Da = (int)a.Da, Db = (int)a.Db;
    cudaError_t e = p_is_a ? launch_gemm_dual(tm_ha, tm_wa, tm_hb, tm_wb, N, V, Da, Db, KLEpi{N, n_vt, parts}, a.stream)
                           : launch_gemm_dual(tm_hb, tm_wb, tm_ha, tm_wa, N, V, Db, Da, KLEpi{N, n_vt, parts}, a.stream);
    if (e != cudaSuccess) return e;
    RowStat *sa = static_cast<RowStat *>(a.stats_a), *sb = static_cast<RowStat *>(a.stats_b);
    if (a.parts)
        linear_kl_merge_kernel<true><<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
            (int)a.N, n_vt, parts, nullptr, nullptr, nullptr, static_cast<PartialRec *>(a.parts));
    else
        linear_kl_merge_kernel<false><<<(unsigned)((a.N + 7) / 8), 256, 0, a.stream>>>(
            (int)a.N, n_vt, parts, a.kl, p_is_a ? sa : sb, p_is_a ? sb : sa, nullptr);
    return cudaGetLastError();
}

// dz of A and of B for one chunk (each twice over: the hi and lo halves of the
// exact form), then the fp32 dhidden accumulators of A and B.
size_t linear_kl_bwd_workspace_bytes(int64_t N, int64_t V, int64_t Da, int64_t Db) {
    const size_t dz = up256((size_t)2 * N * chunk_cols(N, V) * 2);
    return 2 * dz + up256((size_t)N * Da * 4) + up256((size_t)N * Db * 4);
}

// Backward of a two-model op: per vocabulary chunk, the dual GEMM recomputes
// both logits tiles and the epilogue made by make_epi(dza, dzb) writes dz of A
// and / or B; then the gradient GEMMs of each model whose gradients are asked for.
// b_first: the dual GEMM takes model B as its first product; make_epi(ldz,
// dz of the first product, dz of the second, lo_off) builds the epilogue.
template <class MakeEpi>
static cudaError_t two_model_bwd(const LinearKLArgs &a, bool b_first, MakeEpi make_epi) {
    const int64_t vc = chunk_cols(a.N, a.V);
    const size_t dz_bytes = up256((size_t)2 * a.N * vc * 2);
    const int64_t lo_off = a.precision == VP_GRAD_EXACT_ ? a.N * vc : 0;   // each dz_lo follows its dz_hi
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
        if (!make_map(&tm_wac, Wa + v0 * Da, nv, Da, Da, kPBHalf) ||
            !make_map(&tm_wbc, Wb + v0 * Db, nv, Db, Db, kPBHalf))
            return cudaErrorInvalidValue;
        e = b_first ? launch_gemm_dual(tm_hb, tm_wbc, tm_ha, tm_wac, N, nv, Db, Da, make_epi((int)vc, dzb, dza, lo_off),
                                       a.stream)
                    : launch_gemm_dual(tm_ha, tm_wac, tm_hb, tm_wbc, N, nv, Da, Db, make_epi((int)vc, dza, dzb, lo_off),
                                       a.stream);
        if (e != cudaSuccess) return e;
        const bool last = v0 + vc >= V;
        if (want_a && (e = chunk_gradient_gemms(tm_ha_mn, Wa, N, Da, v0, nv, vc, dza, lo_off ? dza + lo_off : nullptr,
                                                acc_a, static_cast<__nv_bfloat16 *>(a.dha),
                                                static_cast<__nv_bfloat16 *>(a.dwa), last, a.stream)) != cudaSuccess)
            return e;
        if (want_b && (e = chunk_gradient_gemms(tm_hb_mn, Wb, N, Db, v0, nv, vc, dzb, lo_off ? dzb + lo_off : nullptr,
                                                acc_b, static_cast<__nv_bfloat16 *>(a.dhb),
                                                static_cast<__nv_bfloat16 *>(a.dwb), last, a.stream)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_linear_kl_bwd(const LinearKLArgs &a) {
    const bool p_is_a = a.direction == 0;
    const RowStat *sa = static_cast<const RowStat *>(a.stats_a), *sb = static_cast<const RowStat *>(a.stats_b);
    // P first: the forward direction, KL(B||A), runs the dual GEMM with model B first
    return two_model_bwd(a, !p_is_a, [&](int ldz, __nv_bfloat16 *dzp, __nv_bfloat16 *dzq, int64_t lo_off) {
        return DzKLEpi{(int)a.N, ldz, p_is_a ? sa : sb, p_is_a ? sb : sa, a.g, dzp, dzq, lo_off};
    });
}

// ---------------------------------------------------------------------------
// Generalized JSD of two models, interior beta ([P1], the commit message adding
// vocab_parallel_jsd: "Motivation" names teacher-student divergences computed
// from tiled LM-head projections, "Changes" the two passes: global
// normalisation first, then both KL-to-mixture expectations together).
//   pass 1  each model's single-product GEMM and merge (the entropy
//           forward's): each row's exact maxima and log-sums of A and B in
//           the two records;
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

    // any tile: columns past ncol left out, zero-weight terms skipped, log2 mix
    // kept above -250
    __device__ __forceinline__ JsdTile checked(int ncol, const RowStat &A, const RowStat &B, const float (&x)[128],
                                               uint32_t tb) const {
        const float omb = 1.f - beta;
        float kp = 0.f, kq = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if (c * 32 + i >= ncol) continue;
                const float xa = ((x[c * 32 + i] - A.m) - A.logS_hi) * kLog2e;   // log2 p
                const float xb = ((b[i] - B.m) - B.logS_hi) * kLog2e;            // log2 q
                const float p = ex2_fast(xa), q = ex2_fast(xb);
                const float lm = fmaxf(lg2_fast(fmaf(beta, q, omb * p)), -250.f);
                if (p > 0.f) kp = fmaf(p, xa - lm, kp);                  // zero-weight terms add nothing
                if (q > 0.f) kq = fmaf(q, xb - lm, kq);
            }
        }
        return JsdTile{kp, kq};
    }

    // a full tile, two columns per instruction: log2 p = z log2(e) - C with
    // C = (m + log S) log2(e) rounded once; a mixture that underflows to 0 makes
    // log2 mix = -inf and the sums non-finite, and such a tile is redone by
    // checked()
    __device__ __forceinline__ JsdTile full(const RowStat &A, const RowStat &B, const float (&x)[128],
                                            uint32_t tb) const {
        const double l2e = 1.4426950408889634074;
        const float2 nCa = splat((float)(-((double)A.m + A.logS_hi + A.logS_lo) * l2e));
        const float2 nCb = splat((float)(-((double)B.m + B.logS_hi + B.logS_lo) * l2e));
        const float2 L = splat(kLog2e), bet = splat(beta), omb = splat(1.f - beta), m1 = splat(-1.f);
        float2 kp[2] = {splat(0.f), splat(0.f)}, kq[2] = {splat(0.f), splat(0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const int k = (i >> 1) & 1;
                const float2 xa = __ffma2_rn(pair128(x, c * 32 + i), L, nCa), xb = __ffma2_rn(pair_at(b, i), L, nCb);
                const float2 p = ex2_pair(xa), q = ex2_pair(xb);
                const float2 lm = lg2_pair(__ffma2_rn(bet, q, __fmul2_rn(omb, p)));
                kp[k] = __ffma2_rn(p, __ffma2_rn(lm, m1, xa), kp[k]);
                kq[k] = __ffma2_rn(q, __ffma2_rn(lm, m1, xb), kq[k]);
            }
        }
        const float2 p2 = __fadd2_rn(kp[0], kp[1]), q2 = __fadd2_rn(kq[0], kq[1]);
        return JsdTile{p2.x + p2.y, q2.x + q2.y};
    }

    __device__ __forceinline__ void operator()(int row, int col0, int ncol, const float (&x)[128], uint32_t tb) const {
        const bool valid = row < N;
        const int r = valid ? row : 0;
        const RowStat A = load_rowstat(sa + r), B = load_rowstat(sb + r);
        JsdTile t;
        if (ncol == kDualEpiCols) {                 // warp-uniform
            t = full(A, B, x, tb);
            const bool redo = !finite(t.kp) || !finite(t.kq);
            if (__any_sync(0xffffffffu, redo)) {    // TMEM loads are warp-collective
                const JsdTile u = checked(ncol, A, B, x, tb);
                if (redo) t = u;
            }
        } else {
            t = checked(ncol, A, B, x, tb);
        }
        if (!valid) return;
        parts[(int64_t)row * n_vt + col0 / kDualEpiCols] = t;
    }
};

__global__ void __launch_bounds__(256)
linear_jsd_merge_kernel(int N, int n_vt, float beta, const JsdTile *__restrict__ parts, float *__restrict__ jsd,
                        RowStat *__restrict__ sa, RowStat *__restrict__ sb) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const JsdTile *p = parts + (int64_t)row * n_vt;
    // tiles lane, lane + 32, ... in that order, four loads issued together
    constexpr int kB = 4;
    DF kp{0.f, 0.f}, kq{0.f, 0.f};
    for (int i0 = lane; i0 < n_vt; i0 += 32 * kB) {
        JsdTile tt[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) tt[u] = i0 + 32 * u < n_vt ? p[i0 + 32 * u] : JsdTile{0.f, 0.f};
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            df_add(kp, tt[u].kp);
            df_add(kq, tt[u].kq);
        }
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
    int64_t lo_off;

    // columns j0 .. j0 + 7 of the half tile with the per-column tests: columns
    // past ncol give 0, zero-weight terms give 0, log2 mix kept above -250, NaN
    // rows give NaN
    __device__ __forceinline__ void checked(int j0, int i0, int ncol, bool nan, float gr, const RowStat &A,
                                            const RowStat &B, const float (&x)[128], const float (&b)[32],
                                            float (&oa)[8], float (&ob)[8]) const {
        const float omb = 1.f - beta;
        const float ka = A.c_hi + A.c_lo, kb = B.c_hi + B.c_lo;   // KL(p||mix), KL(q||mix)
        const float ln2 = 0.69314718055994530942f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float la = (x[j0 + u] - A.m) - A.logS_hi, lb = (b[i0 + u] - B.m) - B.logS_hi;   // log p, log q
            const float p = ex2_fast(la * kLog2e), q = ex2_fast(lb * kLog2e);
            const float lmix = fmaxf(lg2_fast(fmaf(beta, q, omb * p)), -250.f) * ln2;
            float dA = p == 0.f ? 0.f : gr * omb * p * ((la - lmix) - ka);
            float dB = q == 0.f ? 0.f : gr * beta * q * ((lb - lmix) - kb);
            if (j0 + u >= ncol) dA = dB = 0.f;
            else if (nan) dA = dB = qnan();
            oa[u] = dA;
            ob[u] = dB;
        }
    }

    __device__ __forceinline__ void operator()(int row, int col0, int ncol, const float (&x)[128], uint32_t tb) const {
        const bool valid = row < N;
        const int r = valid ? row : 0;
        const RowStat A = load_rowstat(sa + r), B = load_rowstat(sb + r);
        const bool nan = ((A.flags | B.flags) & (kRowNanInf | kRowEmpty)) != 0;
        const float gr = valid ? g[row] : 0.f;
        const bool full = ncol == kDualEpiCols;
        // log p = z - C with C = m + log S rounded once
        const float2 nCa = splat((float)(-((double)A.m + A.logS_hi + A.logS_lo)));
        const float2 nCb = splat((float)(-((double)B.m + B.logS_hi + B.logS_lo)));
        const float2 L = splat(kLog2e), bet = splat(beta), omb = splat(1.f - beta), m1 = splat(-1.f);
        const float2 ln2 = splat(0.69314718055994530942f);
        const float2 nka = splat(-(A.c_hi + A.c_lo)), nkb = splat(-(B.c_hi + B.c_lo));
        const float2 ga = splat(gr * (1.f - beta)), gb = splat(gr * beta);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float b[32];
            tmem_ld32(tb + c * 32, b);
#pragma unroll
            for (int gq = 0; gq < 4; ++gq) {
                const int i0 = gq * 8, j0 = c * 32 + i0;
                // two columns per instruction, no per-column tests; an
                // underflowed mixture (log mix = -inf) leaves the group's sum
                // non-finite, and such a group is redone with the tests
                float oa[8], ob[8];
                float2 chk = splat(0.f);
#pragma unroll
                for (int u = 0; u < 8; u += 2) {
                    const float2 la = __fadd2_rn(pair128(x, j0 + u), nCa), lb = __fadd2_rn(pair_at(b, i0 + u), nCb);
                    const float2 p = ex2_pair(__fmul2_rn(la, L)), q = ex2_pair(__fmul2_rn(lb, L));
                    const float2 lmix = __fmul2_rn(lg2_pair(__ffma2_rn(bet, q, __fmul2_rn(omb, p))), ln2);
                    const float2 ua = __fadd2_rn(__ffma2_rn(lmix, m1, la), nka);
                    const float2 ub = __fadd2_rn(__ffma2_rn(lmix, m1, lb), nkb);
                    chk = __fadd2_rn(chk, __fadd2_rn(ua, ub));
                    const float2 dA = __fmul2_rn(__fmul2_rn(ga, p), ua), dB = __fmul2_rn(__fmul2_rn(gb, q), ub);
                    oa[u] = dA.x;
                    oa[u + 1] = dA.y;
                    ob[u] = dB.x;
                    ob[u + 1] = dB.y;
                }
                if (!full || nan || !finite(chk.x + chk.y)) checked(j0, i0, ncol, nan, gr, A, B, x, b, oa, ob);
                if (!valid) continue;
                const int64_t off = (int64_t)row * ldz + col0 + j0;
                if (dza) store_dz(dza + off, oa, lo_off);
                if (dzb) store_dz(dzb + off, ob, lo_off);
            }
        }
    }
};

cudaError_t launch_linear_jsd_fwd(const LinearKLArgs &a) {
    // pass 1: each model's records (row max, log-sum, flags) from its own
    // single-product forward, the entropy's (its H output, written to jsd, is
    // overwritten below): two single GEMMs cost less than one dual KL pass
    LinearEntArgs ea{a.ha, a.wa, a.N, a.V, a.Da, a.kl, a.stats_a, nullptr, nullptr, nullptr, a.workspace, a.stream};
    cudaError_t e = launch_linear_entropy_fwd(ea);
    if (e != cudaSuccess) return e;
    LinearEntArgs eb{a.hb, a.wb, a.N, a.V, a.Db, a.kl, a.stats_b, nullptr, nullptr, nullptr, a.workspace, a.stream};
    if ((e = launch_linear_entropy_fwd(eb)) != cudaSuccess) return e;
    // pass 2: both KL-to-mixture expectations (the workspace is free again)
    CUtensorMap tm_ha, tm_wa, tm_hb, tm_wb;
    if (!make_map(&tm_ha, a.ha, a.N, a.Da, a.Da, kLBM) || !make_map(&tm_wa, a.wa, a.V, a.Da, a.Da, kPBHalf) ||
        !make_map(&tm_hb, a.hb, a.N, a.Db, a.Db, kLBM) || !make_map(&tm_wb, a.wb, a.V, a.Db, a.Db, kPBHalf))
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
    return two_model_bwd(a, false, [&](int ldz, __nv_bfloat16 *dza, __nv_bfloat16 *dzb, int64_t lo_off) {
        return DzJsdEpi{(int)a.N, ldz, a.beta, sa, sb, a.g, dza, dzb, lo_off};
    });
}

cudaError_t read_linear_ent_kl_fault(uint32_t *value, bool clear) { return read_tu_fault(value, clear); }

}  // namespace vp
