// vp_bwd.cu -- fused backward kernels: logprobs, entropy and KL gradients.
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838): first commit message (fused forward
//        and backward passes per op), second commit message ("gradients are
//        returned contiguous"; rows read in place through two strides), and
//        the Codex thread (positions of zero weight get exactly zero).
//   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton", review nitpick
//        on the chunked backward: dz = onehot - exp(logits - lse), scaled by
//        the upstream gradient.
//
// Gradients, per row with upstream g, t_j = z_j - m and p_j = exp(t_j - logS),
// written with the centred mean c of the forward's vp_rowstat record:
//   logprobs  dz_j = g (onehot_{j,t} - p_j)
//   entropy   dz_j = -g p_j (log p_j + H)  = -g p_j (t_j - c)          (0 where p_j = 0)
//   KL(P||Q)  dP_j = g p_j (log p_j - log q_j - KL)
//                  = g p_j ((t^P_j - t^Q_j) - c)                       (0 where p_j = 0)
//             dQ_j = g (q_j - p_j)
//   JSD       dA_j = g (1 - beta) p_j ((log p_j - log mix_j) - KL(p || mix))
//             dB_j = g beta q_j ((log q_j - log mix_j) - KL(q || mix)), mix = beta q + (1 - beta) p
// m is the exact row max, so t_j is exact; logS and c arrive as hi + lo pairs.
// The fp32 path uses both halves and an error-free difference t^P - t^Q, so a
// gradient that cancels to near zero keeps its accuracy. The bf16 path
// subtracts both halves of c, and of log S where 1 - p of a target cancels;
// where q ~ p it forms q - p as p (e^d - 1) from d = log q - log p.
//
// Shape: each CTA (256 threads) handles one tile of one row: up to 1024
// 16-byte vectors of the input (8192 bf16 / 4096 fp32 logits), four loads in
// flight per thread, and writes the same span of the contiguous gradient with
// streaming 16-byte stores. Rows whose input and output do not share their
// address modulo 16 are processed element by element.
#include "vp_device.cuh"
#include "vp_launch.h"

namespace vp {

constexpr int kTileVec = kBwdThreads * kBwdVecPerThread;

enum RowMode { kNormal = 0, kZero = 1, kNaN = 2 };

template <typename T>
__device__ __forceinline__ uint4 splat(float v) {
    float f[Elem<T>::kVec];
#pragma unroll
    for (int i = 0; i < Elem<T>::kVec; ++i) f[i] = v;
    return Elem<T>::pack(f);
}

// --------------------------------------------------------------------------
// Element formulas. The fp32 path carries t, log p and the centred factor as
// double-floats, takes an accurate exponential and rounds each gradient once;
// the bf16 path uses fp32 arithmetic and the hardware exponential.
// --------------------------------------------------------------------------
template <int kOp, typename T>
__device__ __forceinline__ float grad_elem(float z, int64_t j, const RowStat &s, float g, int64_t loc) {
    if constexpr (Elem<T>::kPrecise) {
        // exact t and log p (double-float), p from the split-argument exponential
        // (relative error below 1.5e-7), each gradient rounded once: within 1e-6
        // of the exact gradient for |g| up to ~6
        const DF t = df_diff(z, s.m);
        const DF lp = df_sub(t, s.logS_hi, s.logS_lo);
        const float p = exp_split(lp.hi, lp.lo);
        if (kOp == 0) {                                   // g (onehot - p)
            if (j != loc) return -g * p;
            const float lpf = lp.hi + lp.lo;
            return g * (lpf > -0.5f ? -expm1_small(lpf) : 1.f - p);   // 1 - p without cancellation
        }
        if (p == 0.f) return 0.f;                         // -g p (t - c)
        const DF r = df_sub(t, s.c_hi, s.c_lo);
        return -g * p * (r.hi + r.lo);
    } else {
        const float t = z - s.m;
        const float lp = t - s.logS_hi;
        const float p = Elem<T>::exp(lp);
        if (kOp == 0) {
            if (j != loc) return -g * p;
            const float lpt = lp - s.logS_lo;                          // log p of the target, both halves
            return g * (lpt > -0.5f ? -expm1_small(lpt) : 1.f - p);   // 1 - p without cancellation
        }
        return (p == 0.f) ? 0.f : -g * p * ((t - s.c_hi) - s.c_lo);
    }
}

// fp32 inputs: grad_elem of two columns at once (f32x2, each lane rounded as
// grad_elem rounds it), both taken as non-targets (logprobs: -g p; the caller
// rewrites a target column with grad_elem).
template <int kOp>
__device__ __forceinline__ float2 grad_pair_f32(float2 z, const RowStat &s, float g) {
    const DF2 t = two_sum2(z, f2(-s.m));
    const DF2 lp = df_sub2(t, DF2{f2(s.logS_hi), f2(s.logS_lo)});
    const float2 p = exp_split2(lp);
    if (kOp == 0) return __fmul2_rn(f2(-g), p);
    const DF2 r = df_sub2(t, DF2{f2(s.c_hi), f2(s.c_lo)});
    const float2 d = __fmul2_rn(__fmul2_rn(f2(-g), p), __fadd2_rn(r.hi, r.lo));
    return make_float2(p.x == 0.f ? 0.f : d.x, p.y == 0.f ? 0.f : d.y);
}

// k_pq = log S_P - log S_Q of the row (double-float): log q_j - log p_j =
// (t^Q_j - t^P_j) + k_pq. Where that difference d is small, q - p cancels, and
// the bf16 path evaluates it as p (e^d - 1) with a series for e^d - 1.
template <typename T, bool kDP, bool kDQ>
__device__ __forceinline__ void kl_grad_elem(float zp, float zq, const RowStat &sp, const RowStat &sq, const DF &k_pq,
                                             float g, bool p_nan, float &dp, float &dq) {
    if constexpr (Elem<T>::kPrecise) {
        // as grad_elem: exact centred values and log-probabilities, split-argument
        // exponentials, q - p as p (e^d - 1) where |d| < 1/2, each gradient rounded once
        const DF tp = df_diff(zp, sp.m), tq = df_diff(zq, sq.m);
        const DF lp = df_sub(tp, sp.logS_hi, sp.logS_lo), lq = df_sub(tq, sq.logS_hi, sq.logS_lo);
        const float p = exp_split(lp.hi, lp.lo), q = exp_split(lq.hi, lq.lo);
        if (kDQ) {
            const DF dd = df_sub(lq, lp.hi, lp.lo);
            const float d = dd.hi + dd.lo;
            dq = g * (fabsf(d) < 0.5f ? p * expm1_small(d) : q - p);
        }
        if (kDP) {                                                     // g p ((tP - tQ) - c)
            if (p_nan) dp = qnan();
            else if (p == 0.f) dp = 0.f;
            else {
                const DF r = df_sub(df_sub(tp, tq.hi, tq.lo), sp.c_hi, sp.c_lo);
                dp = g * p * (r.hi + r.lo);
            }
        }
    } else {
        const float tp = zp - sp.m, tq = zq - sq.m;          // exact for bf16 values
        // base-2 arguments t log2(e) - log S log2(e) with one FMA, the operations
        // of KLGradRow::vec, so that an element's gradient does not depend on
        // which of the two paths (set by the rows' and outputs' alignment) takes it
        float p, q;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(fmaf(tp, kLog2e, -sp.logS_hi * kLog2e)));
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(q) : "f"(fmaf(tq, kLog2e, -sq.logS_hi * kLog2e)));
        if (kDQ) {
            // q - p = p (e^d - 1), d = log q - log p. Below |d| = 1/64 the difference
            // of the two exponentials would lose more than 2^-9 of itself (each carries
            // up to ~2^-18 relative error from its rounded argument), so it is taken from
            // the series d + d^2/2 (truncation below d^2/6 < 2^-14 of the result).
            const float d = ((tq - tp) + k_pq.hi) + k_pq.lo;
            const float em1 = fmaf(0.5f * d, d, d);
            dq = g * (fabsf(d) < 0.015625f ? p * em1 : q - p);
        }
        if (kDP) dp = p_nan ? qnan() : (p == 0.f) ? 0.f : g * p * (((tp - tq) - sp.c_hi) - sp.c_lo);
    }
}

// fp32 inputs: kl_grad_elem of two columns at once (f32x2, each lane rounded
// as kl_grad_elem rounds it).
template <bool kDP, bool kDQ>
__device__ __forceinline__ void kl_grad_pair_f32(float2 zp, float2 zq, const RowStat &sp, const RowStat &sq, float g,
                                                 bool p_nan, float2 &dp, float2 &dq) {
    const DF2 tp = two_sum2(zp, f2(-sp.m)), tq = two_sum2(zq, f2(-sq.m));
    const DF2 lp = df_sub2(tp, DF2{f2(sp.logS_hi), f2(sp.logS_lo)});
    const DF2 lq = df_sub2(tq, DF2{f2(sq.logS_hi), f2(sq.logS_lo)});
    const float2 p = exp_split2(lp), q = exp_split2(lq);
    if (kDQ) {
        const DF2 dd = df_sub2(lq, lp);
        const float2 d = __fadd2_rn(dd.hi, dd.lo);
        const float2 pe = __fmul2_rn(p, expm1_small2(d));
        const float2 qp = __ffma2_rn(p, f2(-1.f), q);                      // q - p
        dq = __fmul2_rn(f2(g), make_float2(fabsf(d.x) < 0.5f ? pe.x : qp.x, fabsf(d.y) < 0.5f ? pe.y : qp.y));
    }
    if (kDP) {                                                           // g p ((tP - tQ) - c)
        if (p_nan) {                                                     // the whole row (a flagged P)
            dp = f2(qnan());
        } else {
            const DF2 r = df_sub2(df_sub2(tp, tq), DF2{f2(sp.c_hi), f2(sp.c_lo)});
            const float2 v = __fmul2_rn(__fmul2_rn(f2(g), p), __fadd2_rn(r.hi, r.lo));
            dp = make_float2(p.x == 0.f ? 0.f : v.x, p.y == 0.f ? 0.f : v.y);
        }
    }
}

// --------------------------------------------------------------------------
// logprobs (kOp = 0) and entropy (kOp = 1)
// --------------------------------------------------------------------------
template <int kOp, typename T>
__global__ void __launch_bounds__(kBwdThreads)
grad_kernel(const T *__restrict__ x, int V, Rows rows, const RowStat *__restrict__ stats,
            const float *__restrict__ g_in, const int64_t *__restrict__ targets, int64_t vocab_start,
            T *__restrict__ dx, int32_t *__restrict__ err, int tiles_per_row, int64_t total_tiles) {
    pdl_enter<true>();   // no global access before this
    constexpr int kVec = Elem<T>::kVec;
    const int tid = threadIdx.x;
    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const int64_t r = tile / tiles_per_row;
        const int seg = (int)(tile - r * tiles_per_row);
        const T *in = x + rows.off(r);
        T *out = dx + r * (int64_t)V;
        // the tile's streaming loads go out first, ahead of the row header's loads
        const int hin = head_count(in, V), hout = head_count(out, V);
        const int v0 = seg * kTileVec;
        const int v1 = hin == hout ? min((V - hin) / kVec, v0 + kTileVec) : 0;
        uint4 u[kBwdVecPerThread];
#pragma unroll
        for (int k = 0; k < kBwdVecPerThread; ++k) {
            const int i = v0 + tid + k * kBwdThreads;
            if (i < v1) u[k] = ldg_stream(reinterpret_cast<const uint4 *>(in + hin) + i);
        }
        const RowStat s = load_rowstat(stats + r);
        const float g = g_in[r];
        int64_t loc = -1;
        int mode = (s.flags & (kRowNanInf | kRowEmpty | kRowBadTarget)) ? kNaN : kNormal;
        if (kOp == 0) {
            const int64_t t = targets[r];
            if (t < 0) {
                mode = kZero;
            } else {
                loc = t - vocab_start;
                if (loc < 0 || loc >= V) {
                    if (s.flags & kRowSharded) {
                        loc = -1;   // merged record: the target lies in another vocabulary shard
                    } else {
                        mode = kNaN;
                        if (err && seg == 0 && tid == 0) atomicOr(err, VP_ERRBIT_TARGET_);
                    }
                }
            }
        }

        if (hin == hout) {
            const int head = hin;
            const int nv = (V - head) / kVec;
            const int tail0 = head + nv * kVec;
            if (seg == 0) {
                for (int j = tid; j < head; j += kBwdThreads) {
                    float d = mode == kZero ? 0.f : mode == kNaN ? qnan()
                              : grad_elem<kOp, T>(Elem<T>::load1(in + j), j, s, g, loc);
                    Elem<T>::store1(out + j, d);
                }
                for (int j = tail0 + tid; j < V; j += kBwdThreads) {
                    float d = mode == kZero ? 0.f : mode == kNaN ? qnan()
                              : grad_elem<kOp, T>(Elem<T>::load1(in + j), j, s, g, loc);
                    Elem<T>::store1(out + j, d);
                }
            }
            uint4 *vout = reinterpret_cast<uint4 *>(out + head);
            if (mode != kNormal) {
                const uint4 c = splat<T>(mode == kZero ? 0.f : qnan());
                for (int i = v0 + tid; i < v1; i += kBwdThreads) stg_stream(vout + i, c);
                continue;
            }
#pragma unroll
            for (int k = 0; k < kBwdVecPerThread; ++k) {
                const int i = v0 + tid + k * kBwdThreads;
                if (i < v1) {
                    float z[kVec], d[kVec];
                    Elem<T>::unpack(u[k], z);
                    const int64_t j0 = head + (int64_t)i * kVec;
                    if (kOp == 0 && !Elem<T>::kPrecise) {
                        // every element as a non-target; the target is rewritten below
#pragma unroll
                        for (int e = 0; e < kVec; ++e) d[e] = grad_elem<0, T>(z[e], 0, s, g, -1);
                    } else if constexpr (Elem<T>::kPrecise) {
                        // pairs of columns (f32x2), then the target column, if here, alone
#pragma unroll
                        for (int e = 0; e < kVec; e += 2) {
                            const float2 dd = grad_pair_f32<kOp>(make_float2(z[e], z[e + 1]), s, g);
                            d[e] = dd.x;
                            d[e + 1] = dd.y;
                        }
                        if (kOp == 0 && loc >= j0 && loc < j0 + kVec) {
#pragma unroll
                            for (int e = 0; e < kVec; ++e)
                                if (j0 + e == loc) d[e] = grad_elem<0, T>(z[e], loc, s, g, loc);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < kVec; ++e) d[e] = grad_elem<kOp, T>(z[e], j0 + e, s, g, loc);
                    }
                    stg_stream(vout + i, Elem<T>::pack(d));
                }
            }
            if (kOp == 0 && !Elem<T>::kPrecise && loc >= head && loc < tail0) {
                // the thread that stored the target's vector rewrites the target element
                // (same thread, same address: the later store wins)
                const int it = (int)((loc - head) / kVec);
                if (it >= v0 && it < v1 && (it - v0) % kBwdThreads == tid)
                    Elem<T>::store1(out + loc, grad_elem<0, T>(Elem<T>::load1(in + loc), loc, s, g, loc));
            }
        } else {
            const int64_t e0 = (int64_t)seg * kTileVec * kVec;
            const int64_t e1 = min((int64_t)V, e0 + (int64_t)kTileVec * kVec);
            for (int64_t j = e0 + tid; j < e1; j += kBwdThreads) {
                float d = mode == kZero ? 0.f : mode == kNaN ? qnan()
                          : grad_elem<kOp, T>(Elem<T>::load1(in + j), j, s, g, loc);
                Elem<T>::store1(out + j, d);
            }
        }
    }
}

// --------------------------------------------------------------------------
// Logprobs of K ids per row (top-k): dz_j = G_j - p_j Gsum, where Gsum sums the
// upstream gradients of the ids that are not ignored and G_j those of the ids
// equal to j (duplicates add up). One CTA per row (grid-stride over rows):
// every warp reads the row's K (id, g) pairs once and reduces them in a fixed
// order (no CTA barrier; the same Gsum in every warp), the CTA writes
// -Gsum p_j over the row tile by tile, then the warp that stored an id's
// element rewrites it as G_j (1 - p_j) - p_j Gother_j in fp64 (topk_target_elem;
// after a warp barrier, so the later store wins). Duplicate ids
// rewrite the same value. A row holding an id outside the shard is NaN (error
// bit); a row whose ids are all ignored is 0.
// --------------------------------------------------------------------------
// An id's own element: G (1 - p) - p Gother, where G sums the upstream
// gradients of the ids equal to this one and Gother those of the row's other
// (not ignored) ids (a row has only K such elements). p comes from the
// double-float exponential (relative error ~1e-8), 1 - p as -(e^{log p} - 1)
// where p > e^{-1/2} (no cancellation as p -> 1), and the two terms are
// combined in fp64, so that their difference keeps its accuracy where they
// nearly cancel.
__device__ __forceinline__ float topk_target_elem(float z, const RowStat &s, double G, double Gother) {
    const DF t = df_diff(z, s.m);
    const DF lp = df_sub(t, s.logS_hi, s.logS_lo);
    const DF e = exp_df(lp.hi, lp.lo);
    const double p = (double)e.hi + (double)e.lo;
    const float lpf = lp.hi + lp.lo;
    const double omp = lpf > -0.5f ? (double)-expm1_small(lpf) : 1.0 - p;
    return (float)(G * omp - p * Gother);
}

template <typename T>
__global__ void __launch_bounds__(kBwdThreads)
topk_grad_kernel(const T *__restrict__ x, int64_t N, int V, Rows rows, const RowStat *__restrict__ stats,
                 const float *__restrict__ g_in, const int64_t *__restrict__ targets, int64_t K, int64_t vocab_start,
                 T *__restrict__ dx, int32_t *__restrict__ err) {
    pdl_enter<true>();   // no global access before this
    constexpr int kVec = Elem<T>::kVec;
    static_assert((kBwdThreads & (kBwdThreads - 1)) == 0 && kTileVec % kBwdThreads == 0, "tiles of whole blocks");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int64_t r = blockIdx.x; r < N; r += gridDim.x) {
        const T *in = x + rows.off(r);
        T *out = dx + r * (int64_t)V;
        const int64_t *tr = targets + r * K;
        const float *gr = g_in + r * K;
        const int hin = head_count(in, V), hout = head_count(out, V);
        const bool vec = hin == hout;
        const int head = vec ? hin : 0;
        const int nv = vec ? (V - head) / kVec : 0;
        const int tail0 = head + nv * kVec;
        // the first tile's streaming loads go out ahead of the row header's loads
        uint4 u[kBwdVecPerThread];
#pragma unroll
        for (int k = 0; k < kBwdVecPerThread; ++k) {
            const int i = tid + k * kBwdThreads;
            if (i < nv) u[k] = ldg_stream(reinterpret_cast<const uint4 *>(in + head) + i);
        }
        const RowStat s = load_rowstat(stats + r);
        // row header, in every warp: Gsum, any id used, any id out of the shard
        float gsum = 0.f;
        int used = 0, bad = 0;
        for (int64_t k = lane; k < K; k += 32) {
            const int64_t t = tr[k];
            if (t < 0) continue;
            used = 1;
            const int64_t loc = t - vocab_start;
            if (loc < 0 || loc >= V) bad = 1;
            gsum += gr[k];
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, m);   // fixed order
        used = __any_sync(0xffffffffu, used);
        bad = __any_sync(0xffffffffu, bad);
        const int mode = !used ? kZero : (bad || (s.flags & (kRowNanInf | kRowEmpty))) ? kNaN : kNormal;
        if (bad && err && tid == 0) atomicOr(err, VP_ERRBIT_TARGET_);

        // phase 1: -Gsum p over the row (0 / NaN rows filled)
        auto scalar_range = [&](int j0, int j1) {
            for (int j = j0 + tid; j < j1; j += kBwdThreads) {
                const float d = mode == kZero ? 0.f : mode == kNaN ? qnan()
                                : grad_elem<0, T>(Elem<T>::load1(in + j), 0, s, gsum, -1);
                Elem<T>::store1(out + j, d);
            }
        };
        if (vec) {
            scalar_range(0, head);
            scalar_range(tail0, V);
            const uint4 *vin = reinterpret_cast<const uint4 *>(in + head);
            uint4 *vout = reinterpret_cast<uint4 *>(out + head);
            const uint4 c = splat<T>(mode == kZero ? 0.f : qnan());
            for (int v0 = 0; v0 < nv; v0 += kTileVec) {
                if (v0 > 0) {
#pragma unroll
                    for (int k = 0; k < kBwdVecPerThread; ++k) {
                        const int i = v0 + tid + k * kBwdThreads;
                        if (i < nv) u[k] = ldg_stream(vin + i);
                    }
                }
#pragma unroll
                for (int k = 0; k < kBwdVecPerThread; ++k) {
                    const int i = v0 + tid + k * kBwdThreads;
                    if (i < nv) {
                        if (mode != kNormal) {
                            stg_stream(vout + i, c);
                            continue;
                        }
                        float z[kVec], d[kVec];
                        Elem<T>::unpack(u[k], z);
#pragma unroll
                        for (int e = 0; e < kVec; ++e) d[e] = grad_elem<0, T>(z[e], 0, s, gsum, -1);
                        stg_stream(vout + i, Elem<T>::pack(d));
                    }
                }
            }
        } else {
            scalar_range(0, V);
        }
        if (mode != kNormal) continue;

        // phase 2: the ids' own elements. Element j was stored in phase 1 by
        // thread owner(j) (the tiles start at multiples of kBwdThreads); the
        // lanes of each warp share out the row's ids, and an id whose element
        // this warp stored is rewritten by a lane of this warp after
        // __syncwarp, which orders the warp's phase-1 stores before it.
        auto owner = [&](int j) -> int {   // j in [0, V)
            if (!vec || j < head) return j & (kBwdThreads - 1);
            if (j >= tail0) return (j - tail0) & (kBwdThreads - 1);
            return (int)((unsigned)(j - head) / (unsigned)kVec) & (kBwdThreads - 1);
        };
        __syncwarp();
        for (int64_t k = lane; k < K; k += 32) {
            const int64_t t = tr[k];
            if (t < 0) continue;
            const int j = (int)(t - vocab_start);          // in [0, V): the row has no id outside the shard
            if ((owner(j) >> 5) != warp) continue;
            double G = 0.0, Gother = 0.0;                  // ids equal to this one / the other ids, in id order
            for (int64_t k2 = 0; k2 < K; ++k2) {
                const int64_t t2 = tr[k2];
                if (t2 == t) G += gr[k2];
                else if (t2 >= 0) Gother += gr[k2];
            }
            Elem<T>::store1(out + j, topk_target_elem(Elem<T>::load1(in + j), s, G, Gother));
        }
    }
}

// --------------------------------------------------------------------------
// Paired inputs (KL, generalized JSD): dP and / or dQ. The per-row policy
// Row gives the NaN state of the row and the element formula.
// --------------------------------------------------------------------------
// KL(P||Q). NaN row (NaN / +inf anywhere, or no finite P logit): both
// gradients NaN; support mismatch (KL = +inf): dP is NaN, dQ = g (q - p)
// stays finite.
template <typename T>
struct KLGradRow {
    RowStat sp, sq;
    DF k_pq;   // log S_P - log S_Q
    float g;
    bool all_nan, p_nan;
    __device__ __forceinline__ KLGradRow(const RowStat *stats_p, const RowStat *stats_q, const float *g_in,
                                         int64_t r) {
        sp = load_rowstat(stats_p + r);
        sq = load_rowstat(stats_q + r);
        k_pq = two_sum(sp.logS_hi, -sq.logS_hi);
        k_pq.lo = __fadd_rn(k_pq.lo, __fsub_rn(sp.logS_lo, sq.logS_lo));
        g = g_in[r];
        all_nan = (sp.flags & (kRowNanInf | kRowEmpty)) || (sq.flags & kRowNanInf);
        p_nan = all_nan || (sp.flags & kRowMismatch);
    }
    template <bool kDP, bool kDQ>
    __device__ __forceinline__ void elem(float zp, float zq, float &dp, float &dq) const {
        kl_grad_elem<T, kDP, kDQ>(zp, zq, sp, sq, k_pq, g, p_nan, dp, dq);
    }
    // One 16-byte vector of P and of Q. bf16: the formulas of kl_grad_elem two
    // columns per instruction (f32x2); the base-2 arguments are formed as
    // t log2(e) - log S log2(e) with one FMA.
    template <bool kDP, bool kDQ>
    __device__ __forceinline__ void vec(const uint4 &up, const uint4 &uq, uint4 &op, uint4 &oq) const {
        if constexpr (Elem<T>::kPrecise) {
            float zp[4], zq[4], dp[4], dq[4];
            Elem<T>::unpack(up, zp);
            Elem<T>::unpack(uq, zq);
#pragma unroll
            for (int e = 0; e < 4; e += 2) {   // kl_grad_elem's operations, two columns at once
                float2 a, b;
                kl_grad_pair_f32<kDP, kDQ>(make_float2(zp[e], zp[e + 1]), make_float2(zq[e], zq[e + 1]), sp, sq, g,
                                           p_nan, a, b);
                dp[e] = a.x; dp[e + 1] = a.y; dq[e] = b.x; dq[e + 1] = b.y;
            }
            if (kDP) op = Elem<T>::pack(dp);
            if (kDQ) oq = Elem<T>::pack(dq);
        } else {
            const float2 nmp = make_float2(-sp.m, -sp.m), nmq = make_float2(-sq.m, -sq.m);
            const float2 l2e = make_float2(kLog2e, kLog2e), m1 = make_float2(-1.f, -1.f);
            const float lp0 = -sp.logS_hi * kLog2e, lq0 = -sq.logS_hi * kLog2e;
            const float2 nlp = make_float2(lp0, lp0), nlq = make_float2(lq0, lq0);
            const float2 kh = make_float2(k_pq.hi, k_pq.hi), kl = make_float2(k_pq.lo, k_pq.lo);
            const float2 nch = make_float2(-sp.c_hi, -sp.c_hi), ncl = make_float2(-sp.c_lo, -sp.c_lo);
            const float2 g2 = make_float2(g, g), half = make_float2(0.5f, 0.5f);
            uint32_t wp[4], wq[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t a = w == 0 ? up.x : w == 1 ? up.y : w == 2 ? up.z : up.w;
                const uint32_t b = w == 0 ? uq.x : w == 1 ? uq.y : w == 2 ? uq.z : uq.w;
                const float2 tp = __fadd2_rn(make_float2(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u)), nmp);
                const float2 tq = __fadd2_rn(make_float2(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u)), nmq);
                const float2 ap = __ffma2_rn(tp, l2e, nlp), aq = __ffma2_rn(tq, l2e, nlq);
                float2 p, q;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p.x) : "f"(ap.x));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p.y) : "f"(ap.y));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(q.x) : "f"(aq.x));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(q.y) : "f"(aq.y));
                if (kDQ) {   // g (q - p), the series where |log q - log p| < 1/64 (kl_grad_elem)
                    const float2 d = __fadd2_rn(__fadd2_rn(__ffma2_rn(tp, m1, tq), kh), kl);
                    const float2 em1 = __ffma2_rn(__fmul2_rn(d, half), d, d);
                    const float2 pe = __fmul2_rn(p, em1);
                    float2 x = __ffma2_rn(p, m1, q);
                    x.x = fabsf(d.x) < 0.015625f ? pe.x : x.x;
                    x.y = fabsf(d.y) < 0.015625f ? pe.y : x.y;
                    const float2 r = __fmul2_rn(g2, x);
                    const __nv_bfloat162 h = __floats2bfloat162_rn(r.x, r.y);
                    wq[w] = *reinterpret_cast<const uint32_t *>(&h);
                }
                if (kDP) {   // g p ((tP - tQ) - c), 0 where p = 0
                    const float2 c = __fadd2_rn(__fadd2_rn(__ffma2_rn(tq, m1, tp), nch), ncl);
                    float2 r = __fmul2_rn(__fmul2_rn(g2, p), c);
                    r.x = p_nan ? qnan() : p.x == 0.f ? 0.f : r.x;
                    r.y = p_nan ? qnan() : p.y == 0.f ? 0.f : r.y;
                    const __nv_bfloat162 h = __floats2bfloat162_rn(r.x, r.y);
                    wp[w] = *reinterpret_cast<const uint32_t *>(&h);
                }
            }
            if (kDP) op = make_uint4(wp[0], wp[1], wp[2], wp[3]);
            if (kDQ) oq = make_uint4(wq[0], wq[1], wq[2], wq[3]);
        }
    }
};

// Generalized JSD with interior beta, (P, Q) = (A, B), mix = beta q + (1 - beta) p:
//   dA_j = g (1 - beta) p_j ((log p_j - log mix_j) - KL(p || mix)),
//   dB_j = g beta q_j ((log q_j - log mix_j) - KL(q || mix)),
// exactly 0 where p_j = 0 (q_j = 0); the KL-to-mixture values are the c fields
// of the forward's records. Rows with a NaN / +inf or no finite logit in A or
// B give NaN rows.
template <typename T>
struct JSDGradRow {
    float ma, mb, la_hi, la_lo, lb_hi, lb_lo, ka, kb, beta, omb, ga, gb;
    bool all_nan;
    static constexpr bool p_nan = false;
    __device__ __forceinline__ JSDGradRow(const RowStat *stats_a, const RowStat *stats_b, const float *g_in,
                                          int64_t r, float beta_) {
        const RowStat sa = load_rowstat(stats_a + r), sb = load_rowstat(stats_b + r);
        ma = sa.m; mb = sb.m;
        la_hi = sa.logS_hi; la_lo = sa.logS_lo; lb_hi = sb.logS_hi; lb_lo = sb.logS_lo;
        ka = sa.c_hi + sa.c_lo;
        kb = sb.c_hi + sb.c_lo;
        beta = beta_;
        omb = 1.f - beta_;
        const float g = g_in[r];
        ga = g * omb;
        gb = g * beta_;
        all_nan = ((sa.flags | sb.flags) & (kRowNanInf | kRowEmpty)) != 0;
    }
    template <bool kDP, bool kDQ>
    __device__ __forceinline__ void elem(float za, float zb, float &da, float &db) const {
        if constexpr (Elem<T>::kPrecise) {
            const float lp = ((za - ma) - la_hi) - la_lo, lq = ((zb - mb) - lb_hi) - lb_lo;   // z - m exact
            const float p = expf(lp), q = expf(lq);
            const float lmix = logf(fmaf(beta, q, omb * p));
            if (kDP) da = (p > 0.f) ? ga * p * ((lp - lmix) - ka) : 0.f;
            if (kDQ) db = (q > 0.f) ? gb * q * ((lq - lmix) - kb) : 0.f;
        } else {
            constexpr float kLn2f = 0.6931471805599453f;
            const float xa = fmaf(za - ma, kLog2e, -(la_hi + la_lo) * kLog2e);   // log2 p
            const float xb = fmaf(zb - mb, kLog2e, -(lb_hi + lb_lo) * kLog2e);
            float p, q;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(xa));
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(q) : "f"(xb));
            float lm;
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lm) : "f"(fmaf(beta, q, omb * p)));
            lm = fmaxf(lm, -250.f);
            if (kDP) da = (p > 0.f) ? ga * p * fmaf(xa - lm, kLn2f, -ka) : 0.f;
            if (kDQ) db = (q > 0.f) ? gb * q * fmaf(xb - lm, kLn2f, -kb) : 0.f;
        }
    }
    template <bool kDP, bool kDQ>
    __device__ __forceinline__ void vec(const uint4 &up, const uint4 &uq, uint4 &op, uint4 &oq) const {
        constexpr int kVec = Elem<T>::kVec;
        float zp[kVec], zq[kVec], dp[kVec], dq[kVec];
        Elem<T>::unpack(up, zp);
        Elem<T>::unpack(uq, zq);
#pragma unroll
        for (int e = 0; e < kVec; ++e) elem<kDP, kDQ>(zp[e], zq[e], dp[e], dq[e]);
        if (kDP) op = Elem<T>::pack(dp);
        if (kDQ) oq = Elem<T>::pack(dq);
    }
};

template <typename T, bool kDP, bool kDQ, class Row>
__device__ __forceinline__ void pair_grad_tile(const T *__restrict__ P, const T *__restrict__ Q, int V, Rows rows,
                                               const Row &row, int64_t r, int seg, T *__restrict__ dP,
                                               T *__restrict__ dQ) {
    constexpr int kVec = Elem<T>::kVec;
    const int tid = threadIdx.x;
    const int64_t off = rows.off(r);
    const T *prow = P + off, *qrow = Q + off;
    T *dprow = kDP ? dP + r * (int64_t)V : nullptr;
    T *dqrow = kDQ ? dQ + r * (int64_t)V : nullptr;
    const bool all_nan = row.all_nan;
    const bool p_nan = row.p_nan;

    uintptr_t ph = (uintptr_t)prow & 15u;
    bool vec = (((uintptr_t)qrow & 15u) == ph);
    if (kDP) vec = vec && (((uintptr_t)dprow & 15u) == ph);
    if (kDQ) vec = vec && (((uintptr_t)dqrow & 15u) == ph);

    auto scalar_range = [&](int64_t j0, int64_t j1) {
        for (int64_t j = j0 + tid; j < j1; j += kBwdThreads) {
            float dp = qnan(), dq = qnan();
            if (!all_nan) row.template elem<kDP, kDQ>(Elem<T>::load1(prow + j), Elem<T>::load1(qrow + j), dp, dq);
            if (kDP) Elem<T>::store1(dprow + j, dp);
            if (kDQ) Elem<T>::store1(dqrow + j, dq);
        }
    };

    if (vec) {
        const int head = head_count(prow, V);
        const int nv = (V - head) / kVec;
        const int tail0 = head + nv * kVec;
        if (seg == 0) {
            scalar_range(0, head);
            scalar_range(tail0, V);
        }
        const int v0 = seg * kTileVec;
        const int v1 = min(nv, v0 + kTileVec);
        const uint4 *vp = reinterpret_cast<const uint4 *>(prow + head);
        const uint4 *vq = reinterpret_cast<const uint4 *>(qrow + head);
        uint4 *vdp = kDP ? reinterpret_cast<uint4 *>(dprow + head) : nullptr;
        uint4 *vdq = kDQ ? reinterpret_cast<uint4 *>(dqrow + head) : nullptr;
        if (all_nan || (kDP && !kDQ && p_nan)) {
            const uint4 c = splat<T>(qnan());
            for (int i = v0 + tid; i < v1; i += kBwdThreads) {
                if (kDP) stg_stream(vdp + i, c);
                if (kDQ) stg_stream(vdq + i, c);
            }
            return;
        }
        uint4 up[kBwdVecPerThread], uq[kBwdVecPerThread];
#pragma unroll
        for (int k = 0; k < kBwdVecPerThread; ++k) {
            const int i = v0 + tid + k * kBwdThreads;
            if (i < v1) { up[k] = ldg_stream(vp + i); uq[k] = ldg_stream(vq + i); }
        }
#pragma unroll
        for (int k = 0; k < kBwdVecPerThread; ++k) {
            const int i = v0 + tid + k * kBwdThreads;
            if (i < v1) {
                uint4 op, oq;
                row.template vec<kDP, kDQ>(up[k], uq[k], op, oq);
                if (kDP) stg_stream(vdp + i, op);
                if (kDQ) stg_stream(vdq + i, oq);
            }
        }
    } else {
        const int64_t e0 = (int64_t)seg * kTileVec * kVec;
        scalar_range(e0, min((int64_t)V, e0 + (int64_t)kTileVec * kVec));
    }
}

// Four CTAs (32 warps) per SM: 64 registers a thread, the occupancy that keeps
// the HBM streams of both inputs and both gradients in flight (for fp32 too:
// three CTAs with the 85 registers that avoid a few spills measured slower).
template <typename T, bool kDP, bool kDQ>
__global__ void __launch_bounds__(kBwdThreads, 4)
kl_grad_kernel(const T *__restrict__ P, const T *__restrict__ Q, int V, Rows rows,
               const RowStat *__restrict__ stats_p, const RowStat *__restrict__ stats_q,
               const float *__restrict__ g_in, T *__restrict__ dP, T *__restrict__ dQ, int tiles_per_row,
               int64_t total_tiles) {
    pdl_enter<true>();   // no global access before this
    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const int64_t r = tile / tiles_per_row;
        const KLGradRow<T> row(stats_p, stats_q, g_in, r);
        pair_grad_tile<T, kDP, kDQ>(P, Q, V, rows, row, r, (int)(tile - r * tiles_per_row), dP, dQ);
    }
}

template <typename T, bool kDA, bool kDB>
__global__ void __launch_bounds__(kBwdThreads)
jsd_grad_kernel(const T *__restrict__ A, const T *__restrict__ B, int V, Rows rows, float beta,
                const RowStat *__restrict__ stats_a, const RowStat *__restrict__ stats_b,
                const float *__restrict__ g_in, T *__restrict__ dA, T *__restrict__ dB, int tiles_per_row,
                int64_t total_tiles) {
    pdl_enter<true>();   // no global access before this
    for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const int64_t r = tile / tiles_per_row;
        const JSDGradRow<T> row(stats_a, stats_b, g_in, r, beta);
        pair_grad_tile<T, kDA, kDB>(A, B, V, rows, row, r, (int)(tile - r * tiles_per_row), dA, dB);
    }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
static inline void tile_grid(int64_t N, int64_t V, int vec, int &tiles_per_row, int64_t &total, unsigned &grid) {
    const int64_t per_tile = (int64_t)kTileVec * vec;
    tiles_per_row = (int)((V + per_tile - 1) / per_tile);
    total = N * tiles_per_row;
    grid = (unsigned)(total < (int64_t)(1u << 30) ? total : (int64_t)(1u << 30));
}

template <int kOp, typename T>
static cudaError_t launch_grad(const GradArgs &a) {
    int tpr;
    int64_t total;
    unsigned grid;
    tile_grid(a.N, a.V, Elem<T>::kVec, tpr, total, grid);
    cudaError_t e = launch_pdl(grad_kernel<kOp, T>, dim3(grid), dim3(kBwdThreads), 0, a.stream,
                               static_cast<const T *>(a.x), (int)a.V, Rows{a.R, a.s_o, a.s_i},
                               static_cast<const RowStat *>(a.stats), a.g, a.targets, a.vocab_start,
                               static_cast<T *>(a.dx), a.err, tpr, total);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_logprobs_bwd(const GradArgs &a) {
    return a.bf16 ? launch_grad<0, __nv_bfloat16>(a) : launch_grad<0, float>(a);
}

cudaError_t launch_entropy_bwd(const GradArgs &a) {
    return a.bf16 ? launch_grad<1, __nv_bfloat16>(a) : launch_grad<1, float>(a);
}

template <typename T>
static cudaError_t launch_topk_grad(const GradArgs &a) {
    const unsigned grid = (unsigned)(a.N < (int64_t)(1u << 30) ? a.N : (int64_t)(1u << 30));   // one CTA per row
    cudaError_t e = launch_pdl(topk_grad_kernel<T>, dim3(grid), dim3(kBwdThreads), 0, a.stream,
                               static_cast<const T *>(a.x), a.N, (int)a.V, Rows{a.R, a.s_o, a.s_i},
                               static_cast<const RowStat *>(a.stats), a.g, a.targets, a.K, a.vocab_start,
                               static_cast<T *>(a.dx), a.err);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_logprobs_topk_bwd(const GradArgs &a) {
    return a.bf16 ? launch_topk_grad<__nv_bfloat16>(a) : launch_topk_grad<float>(a);
}

template <typename T, bool kDP, bool kDQ>
static cudaError_t launch_kl_grad_t(const KLBwdArgs &a) {
    int tpr;
    int64_t total;
    unsigned grid;
    tile_grid(a.N, a.V, Elem<T>::kVec, tpr, total, grid);
    cudaError_t e = launch_pdl(kl_grad_kernel<T, kDP, kDQ>, dim3(grid), dim3(kBwdThreads), 0, a.stream,
                               static_cast<const T *>(a.p), static_cast<const T *>(a.q), (int)a.V,
                               Rows{a.R, a.s_o, a.s_i}, static_cast<const RowStat *>(a.stats_p),
                               static_cast<const RowStat *>(a.stats_q), a.g, static_cast<T *>(a.dp),
                               static_cast<T *>(a.dq), tpr, total);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
static cudaError_t launch_kl_grad_dt(const KLBwdArgs &a) {
    if (a.dp && a.dq) return launch_kl_grad_t<T, true, true>(a);
    if (a.dp) return launch_kl_grad_t<T, true, false>(a);
    return launch_kl_grad_t<T, false, true>(a);
}

cudaError_t launch_kl_bwd(const KLBwdArgs &a) {
    return a.bf16 ? launch_kl_grad_dt<__nv_bfloat16>(a) : launch_kl_grad_dt<float>(a);
}

template <typename T, bool kDA, bool kDB>
static cudaError_t launch_jsd_grad_t(const JsdBwdArgs &a) {
    int tpr;
    int64_t total;
    unsigned grid;
    tile_grid(a.N, a.V, Elem<T>::kVec, tpr, total, grid);
    cudaError_t e = launch_pdl(jsd_grad_kernel<T, kDA, kDB>, dim3(grid), dim3(kBwdThreads), 0, a.stream,
                               static_cast<const T *>(a.a), static_cast<const T *>(a.b), (int)a.V,
                               Rows{a.R, a.s_o, a.s_i}, (float)a.beta, static_cast<const RowStat *>(a.stats_a),
                               static_cast<const RowStat *>(a.stats_b), a.g, static_cast<T *>(a.da),
                               static_cast<T *>(a.db), tpr, total);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
static cudaError_t launch_jsd_grad_dt(const JsdBwdArgs &a) {
    if (a.da && a.db) return launch_jsd_grad_t<T, true, true>(a);
    if (a.da) return launch_jsd_grad_t<T, true, false>(a);
    return launch_jsd_grad_t<T, false, true>(a);
}

cudaError_t launch_jsd_bwd(const JsdBwdArgs &a) {
    return a.bf16 ? launch_jsd_grad_dt<__nv_bfloat16>(a) : launch_jsd_grad_dt<float>(a);
}

}  // namespace vp
