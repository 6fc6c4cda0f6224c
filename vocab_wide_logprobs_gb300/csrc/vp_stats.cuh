// vp_stats.cuh -- per-lane online statistics, their merges and the fp64 row
// finish, shared by the forward kernels (vp_fwd.cu, vp_fwd_tma.cu).
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838): second commit message and the
//        reviewer's "Suggested change" (one read of each logit: online max,
//        sum-exp S and the centred weighted sum W; H = log S - W/S,
//        KL = W/S_A - log S_A + log S_B; partials re-centred on the max;
//        support mismatch decided on the logits), and the Codex thread "Guard
//        zero rescaling before applying infinite shifts" (zero-weight terms).
//   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton", "Implementation"
//        (logp = target logit - LSE).
#pragma once

#include <string.h>

#include <type_traits>

#include "vp_device.cuh"
#include "vp_launch.h"

namespace vp {

// ---------------------------------------------------------------------------
// Packed bf16 helpers (the fast path of the bf16 inputs)
// ---------------------------------------------------------------------------
constexpr uint32_t kBf16NegInf2 = 0xff80ff80u;   // two bf16 -inf

__device__ __forceinline__ __nv_bfloat162 bf162_bits(uint32_t w) {
    __nv_bfloat162 b;
    memcpy(&b, &w, 4);
    return b;
}

// max over the bf16 values held in K 16-byte words (NaN ignored, like fmaxf)
template <int K>
__device__ __forceinline__ float max_bf16(const uint4 (&u)[K]) {
    __nv_bfloat162 m0 = bf162_bits(u[0].x), m1 = bf162_bits(u[0].y), m2 = bf162_bits(u[0].z),
                   m3 = bf162_bits(u[0].w);
#pragma unroll
    for (int k = 1; k < K; ++k) {
        m0 = __hmax2(m0, bf162_bits(u[k].x));
        m1 = __hmax2(m1, bf162_bits(u[k].y));
        m2 = __hmax2(m2, bf162_bits(u[k].z));
        m3 = __hmax2(m3, bf162_bits(u[k].w));
    }
    const __nv_bfloat162 m = __hmax2(__hmax2(m0, m1), __hmax2(m2, m3));
    return fmaxf(__low2float(m), __high2float(m));
}

// min over the bf16 values held in K 16-byte words (NaN ignored)
template <int K>
__device__ __forceinline__ float min_bf16(const uint4 (&u)[K]) {
    __nv_bfloat162 m0 = bf162_bits(u[0].x), m1 = bf162_bits(u[0].y), m2 = bf162_bits(u[0].z),
                   m3 = bf162_bits(u[0].w);
#pragma unroll
    for (int k = 1; k < K; ++k) {
        m0 = __hmin2(m0, bf162_bits(u[k].x));
        m1 = __hmin2(m1, bf162_bits(u[k].y));
        m2 = __hmin2(m2, bf162_bits(u[k].z));
        m3 = __hmin2(m3, bf162_bits(u[k].w));
    }
    const __nv_bfloat162 m = __hmin2(__hmin2(m0, m1), __hmin2(m2, m3));
    return fminf(__low2float(m), __high2float(m));
}

__device__ __forceinline__ float2 bf16_pair(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float ex2_fast(float a) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(a));
    return y;
}

// e^t for the fused-linear forward tiles: the base-2 argument t log2(e) with
// log2(e) split into fp32 hi + lo parts (the product with the hi part exact
// inside the FMA), so that the sums are those of e^t and not of
// e^{t (1 - 1.3e-8)}: with the fp32 constant alone, every weight is off by a
// factor e^{-1.3e-8 t}, which moves the centred mean c = W / S by about
// 1.3e-8 Var_p(t). (The GEMM epilogues have the issue slots to spare; the
// HBM-bound logits scans do not, and there the hardware exponential's own
// error pattern is of the same size.)
constexpr float kLog2eLo = 1.925963033500011e-08f;   // log2(e) - kLog2e
__device__ __forceinline__ float exp_fwd(float t) { return ex2_fast(fmaf(t, kLog2e, t * kLog2eLo)); }
__device__ __forceinline__ float2 exp_fwd2(float2 t) {
    const float2 a = __ffma2_rn(t, make_float2(kLog2e, kLog2e), __fmul2_rn(t, make_float2(kLog2eLo, kLog2eLo)));
    return make_float2(ex2_fast(a.x), ex2_fast(a.y));
}

__device__ __forceinline__ uint32_t word(const uint4 &u, int q) {
    return q == 0 ? u.x : q == 1 ? u.y : q == 2 ? u.z : u.w;
}

// ---------------------------------------------------------------------------
// One distribution, one lane
// ---------------------------------------------------------------------------
// max(a, b) that keeps a NaN operand (fmaxf would drop it).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// A centred value of each lane with a -inf made finite: t.hi at least -200, where
// the exponential is already 0 (NaN kept), and t.lo at least -1 (below an ulp of
// t.hi wherever the exponential is not 0; NaN only where t.hi is not finite).
// Every term e, e t.hi and e t.lo is then finite, and exactly 0 for a -inf value,
// so neither the exponential nor W needs a zero-weight test; where e is not 0 the
// value is unchanged.
__device__ __forceinline__ DF2 finite_centred2(const DF2 &t) {
    return {make_float2(fmax_nan(t.hi.x, -200.f), fmax_nan(t.hi.y, -200.f)),
            make_float2(fmaxf(t.lo.x, -1.f), fmaxf(t.lo.y, -1.f))};
}

// exp_split2 of a finite centred value (finite_centred2): the same operations
// without the zero test, which only guards a_lo = NaN at an infinite t.hi.
__device__ __forceinline__ float2 exp_split2_finite(const DF2 &t) {
    constexpr float kL = 1.4426950408889634f, kLlo = 1.925963033500011e-08f, kLn2 = 0.6931471805599453f;
    const float2 a_hi = __fmul2_rn(t.hi, f2(kL));
    float2 na = __ffma2_rn(t.hi, f2(-kL), a_hi);                       // -(t_hi kL - a_hi)
    na = __ffma2_rn(t.hi, f2(-kLlo), na);
    na = __ffma2_rn(t.lo, f2(-kL), na);                                // -a_lo
    float2 e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(a_hi.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(a_hi.y));
    return __ffma2_rn(e, __fmul2_rn(na, f2(-kLn2)), e);                // e (1 + a_lo ln 2)
}

// How far a value may exceed a lane's centre before the centre moves to it. The
// fp32 path's exponential takes an exact argument, so only overflow bounds it;
// the bf16 path's takes the rounded (t log2 e), t 2^-24 relative error in e^t,
// and a move at t > 4 keeps that within the hardware exponential's own error
// scale (at most 2.4 2^-24) for the terms that carry S.
template <typename T>
__device__ __forceinline__ constexpr float centre_span() { return Elem<T>::kPrecise ? kSpan : kSpanFast; }

template <typename T, bool kW>
struct Lane1 {
    float ref, mx;
    DF S, W;
    int moved;

    __device__ __forceinline__ void init(float r) {
        ref = r; mx = kNegBig; S = {0.f, 0.f}; W = {0.f, 0.f}; moved = 0;
    }

    // Rare: a value exceeds the centre by more than centre_span<T>(). The sums are
    // re-centred in fp64 on the fp32 path; on the bf16 path, whose lane sums are
    // plain fp32, in fp32 (c - ref is exact for bf16 values, expf is within 2 ulp).
    __device__ __forceinline__ void move_centre(float c) {
        if constexpr (Elem<T>::kPrecise) {
            const double d = (double)c - (double)ref;
            const double a = exp(-d);
            double s = df_value(S), w = df_value(W);
            if (kW) w = (a == 0.0) ? 0.0 : a * (w - d * s);
            s *= a;
            S = df_from(s);
            W = df_from(w);
        } else {
            const float d = c - ref;
            const float a = expf(-d);
            const float s = S.hi + S.lo;
            if (kW) W = DF{(a == 0.f) ? 0.f : a * (W.hi + W.lo - d * s), 0.f};
            S = DF{s * a, 0.f};
        }
        ref = c;
        moved = 1;
    }

    template <int n>
    __device__ __forceinline__ void push(const float (&v)[n]) {
        float c = v[0];
#pragma unroll
        for (int i = 1; i < n; ++i) c = fmaxf(c, v[i]);
        mx = fmaxf(mx, c);
        if (c > ref + centre_span<T>()) move_centre(c);
        if constexpr (Elem<T>::kPrecise) {
            // fp32 inputs: exact centred value (double-float), exponential with an exact
            // argument (exp_split), the chunk summed in fp32 (even and odd values apart)
            // and folded into double-floats; on pairs of values (f32x2) where n is even,
            // whose centred values and exponentials round exactly as the scalar forms
            // (the scalar form takes a row's unaligned head and tail).
            // S and W are summed compensated: each addition's rounding error, and each
            // product e t's, goes to a low part. In a peaked row one term carries most
            // of S and W, and a plain fp32 running sum would leave W/S with a few 2^-24
            // of that term's distance from the centre (up to kSpan), which the gradient
            // at a mode with p near 1 resolves. The pairs use the offset fast two-sum:
            // S from K = 2^k above the chunk's exponentials, W from 2^(k+11), above
            // eight of its terms (|e t| < 2^(k+7): t >= -88 wherever e is not 0).
            float s0 = 0.f, s1 = 0.f, sl0 = 0.f, sl1 = 0.f, w0 = 0.f, w1 = 0.f, wl0 = 0.f, wl1 = 0.f;
            if constexpr (n % 2 == 0) {
                const int k = offset_log2(c, ref);
                const float K = pow2f(k), KW = pow2f(k + 11);
                const float2 nref = f2(-ref);
                float2 s2 = f2(K), sl2 = f2(0.f), w2 = f2(KW), wl2 = f2(0.f);
#pragma unroll
                for (int i = 0; i < n; i += 2) {
                    const DF2 t = finite_centred2(two_sum2(make_float2(v[i], v[i + 1]), nref));
                    const float2 e = exp_split2_finite(t);
                    fast_acc2(s2, sl2, e);
                    if (kW) {   // a zero-weight term is exactly 0 here (t is finite)
                        const float2 ph = __fmul2_rn(e, t.hi);
                        const float2 pe = __ffma2_rn(e, t.hi, make_float2(-ph.x, -ph.y));   // e t.hi - ph, exact
                        fast_acc2(w2, wl2, ph);
                        wl2 = __fadd2_rn(wl2, __ffma2_rn(e, t.lo, pe));
                    }
                }
                s0 = s2.x - K; s1 = s2.y - K; sl0 = sl2.x; sl1 = sl2.y;   // exact differences
                w0 = w2.x - KW; w1 = w2.y - KW; wl0 = wl2.x; wl1 = wl2.y;
            } else {
#pragma unroll
                for (int i = 0; i < n; ++i) {
                    const DF t = df_diff(v[i], ref);
                    const float e = exp_split(t.hi, t.lo);
                    float &si = (i & 1) ? s1 : s0;
                    float &sli = (i & 1) ? sl1 : sl0;
                    const DF ss = two_sum(si, e);
                    si = ss.hi;
                    sli += ss.lo;
                    if (kW && e != 0.f) {
                        const float ph = e * t.hi, pe = fmaf(e, t.hi, -ph);
                        float &wi = (i & 1) ? w1 : w0;
                        float &wli = (i & 1) ? wl1 : wl0;
                        const DF sw = two_sum(wi, ph);
                        wi = sw.hi;
                        wli = wli + (sw.lo + fmaf(e, t.lo, pe));
                    }
                }
            }
            df_add(S, s0);
            df_add(S, s1);
            S.lo = __fadd_rn(S.lo, sl0 + sl1);
            if (kW) {
                df_add(W, w0);
                df_add(W, w1);
                W.lo = __fadd_rn(W.lo, wl0 + wl1);
            }
        } else {
            float s0 = 0.f, s1 = 0.f, w0 = 0.f, w1 = 0.f;
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const float t = v[i] - ref;   // exact for bf16 values
                const float e = Elem<T>::exp(t);
                // e is exactly 0 below t = -104, so clamping t keeps 0 * (-inf) out of W
                if (i & 1) { s1 += e; if (kW) w1 = fmaf(e, fmaxf(t, -128.f), w1); }
                else       { s0 += e; if (kW) w0 = fmaf(e, fmaxf(t, -128.f), w0); }
            }
            df_add(S, s0 + s1);
            if (kW) df_add(W, w0 + w1);
        }
    }

    // bf16 fast path on raw 16-byte words (8 values each): packed max, packed
    // f32x2 arithmetic and four independent accumulator pairs. The chunk sums are
    // folded into the lane's double-float sums: after a lane's centre has moved to
    // a peak (S near 1), the later chunks each add far less than an ulp of S, and
    // a plain fp32 running sum would drop them whole (up to the lane's whole
    // off-peak mass, some 2^-24 of S). The warp merges the lanes as double-floats
    // and the partials likewise (warp_sum_acc). What remains is the hardware
    // exponential's error pattern (bias -5e-8 below -1, +3.3e-8 above +1, spread
    // 3e-8, measured on GB300), ~2^-23 relative on c = W / S.
    template <int K>
    __device__ __forceinline__ void push_bf16(const uint4 (&u)[K]) {
        const float c = max_bf16(u);
        mx = fmaxf(mx, c);
        if (c > ref + centre_span<T>()) move_centre(c);
        const float2 nref = make_float2(-ref, -ref), l2e = make_float2(kLog2e, kLog2e);
        float2 s[4], w[4];
#pragma unroll
        for (int k = 0; k < K; ++k) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 t = __fadd2_rn(bf16_pair(word(u[k], q)), nref);   // exact
                const float2 a = __fmul2_rn(t, l2e);
                const float2 e = make_float2(ex2_fast(a.x), ex2_fast(a.y));
                if (k == 0) {
                    s[q] = e;
                    if (kW) w[q] = __fmul2_rn(e, t);
                } else {
                    s[q] = __fadd2_rn(s[q], e);
                    if (kW) w[q] = __ffma2_rn(e, t, w[q]);
                }
            }
        }
        const float2 ss = __fadd2_rn(__fadd2_rn(s[0], s[1]), __fadd2_rn(s[2], s[3]));
        df_add(S, ss.x + ss.y);
        if (kW) {
            float2 ww = __fadd2_rn(__fadd2_rn(w[0], w[1]), __fadd2_rn(w[2], w[3]));
            float wsum = ww.x + ww.y;
            // e * t is 0 * (-inf) = NaN where t = -inf (a -inf logit or a spread beyond
            // FLT_MAX): redo W for this chunk with t clamped (e is exactly 0 below t = -104)
            if (!(fabsf(wsum) < INFINITY)) {
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < K; ++k) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 t = __fadd2_rn(bf16_pair(word(u[k], q)), nref);
                        const float2 a = __fmul2_rn(t, l2e);
                        const float2 e = make_float2(ex2_fast(a.x), ex2_fast(a.y));
                        w[q] = __ffma2_rn(e, make_float2(fmaxf(t.x, -128.f), fmaxf(t.y, -128.f)), w[q]);
                    }
                }
                ww = __fadd2_rn(__fadd2_rn(w[0], w[1]), __fadd2_rn(w[2], w[3]));
                wsum = ww.x + ww.y;
            }
            df_add(W, wsum);
        }
    }
};

// Merged partials carry their sums in fp64 on the fp32 path and as fp32 values on
// the bf16 path: one rounding of a partial (2^-24 of its share) is below the
// hardware exponential's error floor on c (~2^-23, see Lane1::push_bf16), and
// GB300's fp64 pipe is narrow, so the bf16 path keeps fp64 for the one-thread row
// finish only. Sums over several partials are taken as double-floats and rounded
// once (warp_sum_acc): repeated fp32 roundings would add up where one partial
// carries the row.
template <typename T>
using AccT = typename std::conditional<Elem<T>::kPrecise, double, float>::type;

__device__ __forceinline__ double exp_acc(double x) { return exp(x); }
__device__ __forceinline__ float exp_acc(float x) { return expf(x); }

template <typename V>
__device__ __forceinline__ V df_to(const DF &a) { return (V)a.hi + (V)a.lo; }

template <typename V>
__device__ __forceinline__ V warp_sum_t(V v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// Sum over the warp's lanes for the merges of partials: fp64 values as they are;
// fp32 values (the bf16 path) as double-floats, rounded once at the end. A plain
// fp32 butterfly rounds at each of its five levels, and where one lane carries the
// sum (the partial that holds a peaked row's mode) each rounding can take half an
// ulp of it: up to 5 2^-24 of S in log S, which gradients at p near 1, and q - p
// where q ~ p, resolve. The double-float add is symmetric, so all lanes agree;
// a non-finite sum keeps the fp32 butterfly's value (W = +inf in a row whose
// support mismatches stays +inf rather than turning NaN through its low part).
__device__ __forceinline__ double warp_sum_acc(double v) { return warp_sum_t(v); }
__device__ __forceinline__ float warp_sum_acc(float v) {
    DF s{v, 0.f};
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) df_add(s, shfl_xor(s, m));
    return isfinite(s.hi) ? s.hi + s.lo : s.hi;
}

template <typename V>
struct Part1 {  // a merged partial, centre `ref`
    float ref, mx;
    V S, W;
};

template <typename T, bool kW>
__device__ __forceinline__ Part1<AccT<T>> warp_merge(const Lane1<T, kW> &L) {
    using V = AccT<T>;
    Part1<V> o;
    o.mx = warp_max(L.mx);
    if (__all_sync(0xffffffffu, L.moved == 0)) {
        DF S = L.S, W = L.W;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            df_add(S, shfl_xor(S, m));
            if (kW) df_add(W, shfl_xor(W, m));
        }
        o.ref = L.ref;
        o.S = df_to<V>(S);
        o.W = kW ? df_to<V>(W) : V(0);
    } else {
        const float M = warp_max(L.ref);
        const V s = df_to<V>(L.S), w = df_to<V>(L.W);
        const V a = (L.ref == M) ? V(1) : exp_acc((V)L.ref - (V)M);
        V sc = a * s, wc = V(0);
        if (sc != V(0)) { if (kW) wc = a * (w - ((V)M - (V)L.ref) * s); }
        else sc = V(0);
        o.ref = M;
        o.S = warp_sum_acc(sc);
        o.W = kW ? warp_sum_acc(wc) : V(0);
    }
    return o;
}

// Merge the partials held by the lanes of one warp (lane i holds partial i; an
// empty partial where there is none), re-centred on the largest centre and
// added in a fixed shuffle order; the result is valid in all lanes.
template <bool kW, typename V>
__device__ __forceinline__ Part1<V> merge_lane_parts(const Part1<V> &q) {
    const float M = warp_max(q.ref);
    const V a = (q.ref == M) ? V(1) : exp_acc((V)q.ref - (V)M);
    V sc = a * q.S, wc = V(0);
    if (sc != V(0)) { if (kW) wc = a * (q.W - ((V)M - (V)q.ref) * q.S); }
    else sc = V(0);
    Part1<V> o;
    o.ref = M;
    o.mx = warp_max(q.mx);
    o.S = warp_sum_acc(sc);
    o.W = kW ? warp_sum_acc(wc) : V(0);
    return o;
}

template <typename V>
__device__ __forceinline__ Part1<V> empty_part() { return Part1<V>{kNegBig, kNegBig, V(0), V(0)}; }

// Merge `count` (<= 32) warp partials in a fixed order; called by one whole
// warp, the result is valid in all lanes.
template <bool kW, typename V>
__device__ __forceinline__ Part1<V> merge_parts(const Part1<V> *parts, int count) {
    const int lane = threadIdx.x & 31;
    return merge_lane_parts<kW>(lane < count ? parts[lane] : empty_part<V>());
}

// ---------------------------------------------------------------------------
// KL(P||Q): paired statistics from one read of P and Q
// ---------------------------------------------------------------------------
// kW = false keeps the two distributions' sums only (no cross term W and no
// mismatch flag): the JSD's first pass, which needs each row's maxima and sums.
template <typename T, bool kW = true>
struct LaneKL {
    float rp, rq, mxp, mxq;
    DF Sp, Sq, W;
    int flag, moved;

    __device__ __forceinline__ void init(float p, float q) {
        rp = p; rq = q; mxp = mxq = kNegBig;
        Sp = Sq = W = DF{0.f, 0.f};
        flag = 0; moved = 0;
    }

    // as Lane1::move_centre, for both centres
    __device__ __forceinline__ void move_centres(float np, float nq) {
        if constexpr (Elem<T>::kPrecise) {
            const double dp = (double)np - (double)rp, dq = (double)nq - (double)rq;
            const double ap = exp(-dp), aq = exp(-dq);
            const double sp = df_value(Sp), sq = df_value(Sq), w = df_value(W);
            W = df_from(ap == 0.0 ? 0.0 : ap * (w - (dp - dq) * sp));
            Sp = df_from(sp * ap);
            Sq = df_from(sq * aq);
        } else {
            const float dp = np - rp, dq = nq - rq;
            const float ap = expf(-dp), aq = expf(-dq);
            const float sp = Sp.hi + Sp.lo, sq = Sq.hi + Sq.lo;
            W = DF{ap == 0.f ? 0.f : ap * (W.hi + W.lo - (dp - dq) * sp), 0.f};
            Sp = DF{sp * ap, 0.f};
            Sq = DF{sq * aq, 0.f};
        }
        rp = np;
        rq = nq;
        moved = 1;
    }

    template <int n>
    __device__ __forceinline__ void push(const float (&p)[n], const float (&q)[n]) {
        float cp = p[0], cq = q[0];
#pragma unroll
        for (int i = 1; i < n; ++i) { cp = fmaxf(cp, p[i]); cq = fmaxf(cq, q[i]); }
        mxp = fmaxf(mxp, cp);
        mxq = fmaxf(mxq, cq);
        const bool up = cp > rp + centre_span<T>(), uq = cq > rq + centre_span<T>();
        if (up || uq) move_centres(up ? cp : rp, uq ? cq : rq);
        int fl = 0;
        if constexpr (Elem<T>::kPrecise) {
            // fp32 inputs: as Lane1::push (exact centred values, exp_split, chunk sums
            // of the even and the odd values folded into double-floats, pairs of values
            // in f32x2 where n is even)
            float sp0 = 0.f, sp1 = 0.f, sq0 = 0.f, sq1 = 0.f, w0 = 0.f, w1 = 0.f;
            // All three sums are compensated (see Lane1::push). Sp and Sq take the offset
            // fast two-sum from 2^k above each chunk's exponentials; W's terms (the
            // product's rounding error from an FMA, the sum's from a two-sum, both into
            // wl) have no such bound, d = tp - tq growing without limit where Q is far
            // below its centre. Where one term carries most of W (a peaked P whose mode Q
            // puts far below its own), a plain fp32 sum would leave c = W / S_P with
            // 2^-24 of that term's size
            float wl0 = 0.f, wl1 = 0.f, spl0 = 0.f, sql0 = 0.f;   // low parts of the compensated sums
            if constexpr (n % 2 == 0) {
                const float2 nrp = f2(-rp), nrq = f2(-rq);
                const float Kp = pow2f(offset_log2(cp, rp)), Kq = pow2f(offset_log2(cq, rq));
                float2 sp = f2(Kp), sq = f2(Kq), spl = f2(0.f), sql = f2(0.f), w = f2(0.f), wl = f2(0.f);
                float qmin = q[0];
#pragma unroll
                for (int i = 0; i < n; i += 2) {
                    const DF2 tp = two_sum2(make_float2(p[i], p[i + 1]), nrp);
                    const DF2 tq = two_sum2(make_float2(q[i], q[i + 1]), nrq);
                    const float2 ep = exp_split2(tp), eq = exp_split2(tq);
                    fast_acc2(sp, spl, ep);
                    fast_acc2(sq, sql, eq);
                    if constexpr (kW) {
                        const DF2 d = df_sub2(tp, tq);
                        const float2 ph = __fmul2_rn(ep, d.hi);
                        const float2 pe = __ffma2_rn(ep, d.hi, make_float2(-ph.x, -ph.y));   // ep d.hi - ph, exact
                        const DF2 sw = two_sum2(w, ph);
                        const float2 wln = __fadd2_rn(wl, __fadd2_rn(sw.lo, __ffma2_rn(ep, d.lo, pe)));
                        w = make_float2(ep.x != 0.f ? sw.hi.x : w.x, ep.y != 0.f ? sw.hi.y : w.y);   // zero weights add nothing
                        wl = make_float2(ep.x != 0.f ? wln.x : wl.x, ep.y != 0.f ? wln.y : wl.y);
                        qmin = fminf(qmin, fminf(q[i], q[i + 1]));
                    }
                }
                if (kW && qmin == -INFINITY) {   // the support-mismatch flag, decided on the logits
#pragma unroll
                    for (int i = 0; i < n; ++i) fl |= (q[i] == -INFINITY) & (p[i] > -INFINITY);
                }
                sp0 = sp.x - Kp; sp1 = sp.y - Kp; sq0 = sq.x - Kq; sq1 = sq.y - Kq;   // exact differences
                w0 = w.x; w1 = w.y; wl0 = wl.x; wl1 = wl.y;
                spl0 = spl.x + spl.y;
                sql0 = sql.x + sql.y;
            } else {
#pragma unroll
                for (int i = 0; i < n; ++i) {
                    const DF tp = df_diff(p[i], rp), tq = df_diff(q[i], rq);
                    const float ep = exp_split(tp.hi, tp.lo), eq = exp_split(tq.hi, tq.lo);
                    if (kW && ep != 0.f) {           // zero-weight terms add nothing
                        const DF d = df_sub(tp, tq.hi, tq.lo);
                        const float ph = ep * d.hi, pe = fmaf(ep, d.hi, -ph);
                        float &wi = (i & 1) ? w1 : w0;
                        float &wli = (i & 1) ? wl1 : wl0;
                        const DF sw = two_sum(wi, ph);
                        wi = sw.hi;
                        wli = wli + (sw.lo + fmaf(ep, d.lo, pe));
                    }
                    float &spi = (i & 1) ? sp1 : sp0;
                    float &sqi = (i & 1) ? sq1 : sq0;
                    const DF ssp = two_sum(spi, ep), ssq = two_sum(sqi, eq);
                    spi = ssp.hi;
                    sqi = ssq.hi;
                    spl0 += ssp.lo;
                    sql0 += ssq.lo;
                    if (kW) fl |= (q[i] == -INFINITY) & (p[i] > -INFINITY);
                }
            }
            df_add(Sp, sp0);
            df_add(Sp, sp1);
            Sp.lo = __fadd_rn(Sp.lo, spl0);
            df_add(Sq, sq0);
            df_add(Sq, sq1);
            Sq.lo = __fadd_rn(Sq.lo, sql0);
            df_add(W, w0);
            df_add(W, w1);
            W.lo = __fadd_rn(W.lo, wl0 + wl1);
        } else {
            float sp0 = 0.f, sp1 = 0.f, sq0 = 0.f, sq1 = 0.f, w0 = 0.f, w1 = 0.f;
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const float tp = p[i] - rp, tq = q[i] - rq;
                const float ep = Elem<T>::exp(tp), eq = Elem<T>::exp(tq);
                const float dl = (ep > 0.f) ? (tp - tq) : 0.f;  // zero-weight terms add nothing
                if (i & 1) { sp1 += ep; sq1 += eq; w1 = fmaf(ep, dl, w1); }
                else       { sp0 += ep; sq0 += eq; w0 = fmaf(ep, dl, w0); }
                if (kW) fl |= (q[i] == -INFINITY) & (p[i] > -INFINITY);
            }
            df_add(Sp, sp0 + sp1);
            df_add(Sq, sq0 + sq1);
            df_add(W, w0 + w1);
        }
        flag |= fl;
    }

    // bf16 fast path on raw 16-byte words of P and Q (see Lane1::push_bf16); the
    // mismatch flag is taken on the raw halves: Q = -inf where P is not -inf.
    template <int K>
    __device__ __forceinline__ void push_bf16(const uint4 (&up)[K], const uint4 (&uq)[K]) {
        const float cp = max_bf16(up), cq = max_bf16(uq);
        mxp = fmaxf(mxp, cp);
        mxq = fmaxf(mxq, cq);
        const bool mp = cp > rp + centre_span<T>(), mq = cq > rq + centre_span<T>();
        if (mp || mq) move_centres(mp ? cp : rp, mq ? cq : rq);
        const float2 nrp = make_float2(-rp, -rp), nrq = make_float2(-rq, -rq);
        const float2 l2e = make_float2(kLog2e, kLog2e), m1 = make_float2(-1.f, -1.f);
        float2 sp[4], sq[4], w[4];
#pragma unroll
        for (int k = 0; k < K; ++k) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 tp = __fadd2_rn(bf16_pair(word(up[k], q)), nrp);
                const float2 tq = __fadd2_rn(bf16_pair(word(uq[k], q)), nrq);
                const float2 ap = __fmul2_rn(tp, l2e), aq = __fmul2_rn(tq, l2e);
                const float2 ep = make_float2(ex2_fast(ap.x), ex2_fast(ap.y));
                const float2 eq = make_float2(ex2_fast(aq.x), ex2_fast(aq.y));
                if (k == 0) {
                    sp[q] = ep;
                    sq[q] = eq;
                    if (kW) w[q] = __fmul2_rn(ep, __ffma2_rn(tq, m1, tp));       // ep (tp - tq)
                } else {
                    sp[q] = __fadd2_rn(sp[q], ep);
                    sq[q] = __fadd2_rn(sq[q], eq);
                    if (kW) w[q] = __ffma2_rn(ep, __ffma2_rn(tq, m1, tp), w[q]);
                }
            }
        }
        float2 c = f2(0.f);
        float wsum = 0.f;
        if (kW) {
            c = __fadd2_rn(__fadd2_rn(w[0], w[1]), __fadd2_rn(w[2], w[3]));
            wsum = c.x + c.y;
        }
        // A -inf logit in P or Q (or a spread beyond FLT_MAX) makes some tp - tq
        // infinite or NaN and so W non-finite: redo W with zero-weight terms
        // skipped and take the support-mismatch flag (Q = -inf where P is not).
        if (kW && !(fabsf(wsum) < INFINITY)) {
            uint32_t fl = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) w[q] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < K; ++k) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t pw = word(up[k], q), qw = word(uq[k], q);
                    fl |= __vcmpeq2(qw, kBf16NegInf2) & ~__vcmpeq2(pw, kBf16NegInf2);
                    const float2 tp = __fadd2_rn(bf16_pair(pw), nrp), tq = __fadd2_rn(bf16_pair(qw), nrq);
                    const float2 ap = __fmul2_rn(tp, l2e);
                    const float2 ep = make_float2(ex2_fast(ap.x), ex2_fast(ap.y));
                    float2 d = __ffma2_rn(tq, m1, tp);                            // tp - tq
                    d.x = ep.x > 0.f ? d.x : 0.f;                                 // zero-weight terms add nothing
                    d.y = ep.y > 0.f ? d.y : 0.f;
                    w[q] = __ffma2_rn(ep, d, w[q]);
                }
            }
            c = __fadd2_rn(__fadd2_rn(w[0], w[1]), __fadd2_rn(w[2], w[3]));
            wsum = c.x + c.y;
            flag |= (fl != 0);
        }
        const float2 a = __fadd2_rn(__fadd2_rn(sp[0], sp[1]), __fadd2_rn(sp[2], sp[3]));
        const float2 b = __fadd2_rn(__fadd2_rn(sq[0], sq[1]), __fadd2_rn(sq[2], sq[3]));
        // double-float lane sums: the terms of W take both signs (tp - tq), so its
        // fp32 running sum would lose the digits of c = W / S_P that cancel
        df_add(Sp, a.x + a.y);
        df_add(Sq, b.x + b.y);
        df_add(W, wsum);
    }
};

template <typename V>
struct PartKL {
    float rp, rq, mxp, mxq;
    V Sp, Sq, W;
    int flag;
};

// Re-centre one partial on (Mp, Mq) and return its contributions.
template <typename V>
__device__ __forceinline__ void kl_recentred(float rp, float rq, V sp, V sq, V w, float Mp, float Mq, V &osp, V &osq,
                                             V &ow) {
    const V ap = (rp == Mp) ? V(1) : exp_acc((V)rp - (V)Mp);
    const V aq = (rq == Mq) ? V(1) : exp_acc((V)rq - (V)Mq);
    osq = aq * sq;
    if (osq == V(0)) osq = V(0);
    osp = ap * sp;
    ow = V(0);
    if (osp != V(0)) ow = ap * (w - (((V)Mp - (V)rp) - ((V)Mq - (V)rq)) * sp);
    else osp = V(0);
}

template <typename T, bool kW>
__device__ __forceinline__ PartKL<AccT<T>> kl_warp_merge(const LaneKL<T, kW> &L) {
    using V = AccT<T>;
    PartKL<V> o;
    o.mxp = warp_max(L.mxp);
    o.mxq = warp_max(L.mxq);
    o.flag = __any_sync(0xffffffffu, L.flag);
    if (__all_sync(0xffffffffu, L.moved == 0)) {
        DF Sp = L.Sp, Sq = L.Sq, W = L.W;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            df_add(Sp, shfl_xor(Sp, m));
            df_add(Sq, shfl_xor(Sq, m));
            df_add(W, shfl_xor(W, m));
        }
        o.rp = L.rp; o.rq = L.rq;
        o.Sp = df_to<V>(Sp); o.Sq = df_to<V>(Sq); o.W = df_to<V>(W);
    } else {
        const float Mp = warp_max(L.rp), Mq = warp_max(L.rq);
        V sp, sq, w;
        kl_recentred<V>(L.rp, L.rq, df_to<V>(L.Sp), df_to<V>(L.Sq), df_to<V>(L.W), Mp, Mq, sp, sq, w);
        o.rp = Mp; o.rq = Mq;
        o.Sp = warp_sum_acc(sp); o.Sq = warp_sum_acc(sq); o.W = warp_sum_acc(w);
    }
    return o;
}

template <typename V>
__device__ __forceinline__ PartKL<V> empty_kl_part() {
    return PartKL<V>{kNegBig, kNegBig, kNegBig, kNegBig, V(0), V(0), V(0), 0};
}

// KL counterpart of merge_lane_parts.
template <typename V>
__device__ __forceinline__ PartKL<V> kl_merge_lane_parts(const PartKL<V> &q) {
    const float Mp = warp_max(q.rp), Mq = warp_max(q.rq);
    V sp, sq, w;
    kl_recentred<V>(q.rp, q.rq, q.Sp, q.Sq, q.W, Mp, Mq, sp, sq, w);
    PartKL<V> o;
    o.rp = Mp; o.rq = Mq;
    o.mxp = warp_max(q.mxp);
    o.mxq = warp_max(q.mxq);
    o.Sp = warp_sum_acc(sp); o.Sq = warp_sum_acc(sq); o.W = warp_sum_acc(w);
    o.flag = __any_sync(0xffffffffu, q.flag);
    return o;
}

// KL counterpart of merge_parts.
template <typename V>
__device__ __forceinline__ PartKL<V> kl_merge_parts(const PartKL<V> *parts, int count) {
    const int lane = threadIdx.x & 31;
    return kl_merge_lane_parts(lane < count ? parts[lane] : empty_kl_part<V>());
}

// ---------------------------------------------------------------------------
// Row finish in fp64 against the exact row max; writes the output and records.
// ---------------------------------------------------------------------------
// kOp 0 (logprobs): t is the target id, zt the target logit (read when in range).
template <int kOp, typename Acc>
__device__ __forceinline__ void finish_stats(const Part1<Acc> &p, int64_t r, int V, int64_t t, int64_t vocab_start,
                                             float zt, float *out, RowStat *stats, int32_t *err) {
    uint32_t flags = 0;
    const double S = p.S;
    if (S != S) flags |= kRowNanInf;
    else if (S == 0.0) flags |= kRowEmpty;
    const double sh = (double)p.mx - (double)p.ref;
    const double logS = log(S) - sh;
    const double c = kOp == 1 ? (double)p.W / S - sh : 0.0;
    store_rowstat(stats + r, p.mx, logS, c, flags);
    const bool bad = flags != 0;
    if (kOp == 1) {
        out[r] = bad ? qnan() : (float)(logS - c);
        return;
    }
    if (t < 0) { out[r] = 0.f; return; }            // ignored target
    const int64_t loc = t - vocab_start;
    if (loc < 0 || loc >= V) {
        out[r] = qnan();
        if (err) atomicOr(err, VP_ERRBIT_TARGET_);
        return;
    }
    out[r] = bad ? qnan() : (float)(((double)zt - (double)p.mx) - logS);
}

// Several target ids per row (top-k): the row's record as for logprobs, then
// logp for each of the K ids, lanes of the finisher warp taking ids k = lane,
// lane + 32, ... (per id: negative = ignored, 0; outside the shard = NaN and
// the error bit). Called by a whole warp; `p` is valid in every lane.
template <typename T, typename Acc>
__device__ __forceinline__ void finish_topk(const Part1<Acc> &p, int64_t r, int V, int64_t K,
                                            const int64_t *targets, int64_t vocab_start, const T *row, float *out,
                                            RowStat *stats, int32_t *err, int lane) {
    double logS = 0.0;
    uint32_t flags = 0;
    if (lane == 0) {
        const double S = p.S;
        if (S != S) flags |= kRowNanInf;
        else if (S == 0.0) flags |= kRowEmpty;
        logS = log(S) - ((double)p.mx - (double)p.ref);
        store_rowstat(stats + r, p.mx, logS, 0.0, flags);
    }
    logS = __shfl_sync(0xffffffffu, logS, 0);
    flags = __shfl_sync(0xffffffffu, flags, 0);
    for (int64_t k = lane; k < K; k += 32) {
        const int64_t t = targets[r * K + k];
        float v;
        if (t < 0) {
            v = 0.f;
        } else {
            const int64_t loc = t - vocab_start;
            if (loc < 0 || loc >= V) {
                v = qnan();
                if (err) atomicOr(err, VP_ERRBIT_TARGET_);
            } else {
                v = flags ? qnan() : (float)(((double)Elem<T>::load1(row + loc) - (double)p.mx) - logS);
            }
        }
        out[r * K + k] = v;
    }
}

template <typename Acc>
__device__ __forceinline__ void finish_kl(const PartKL<Acc> &s, int64_t r, float *kl, RowStat *stats_p,
                                          RowStat *stats_q) {
    uint32_t fp = 0, fq = 0;
    const double Sp = s.Sp, Sq = s.Sq, W = s.W;
    if (Sp != Sp) fp |= kRowNanInf;
    else if (Sp == 0.0) fp |= kRowEmpty;
    if (Sq != Sq) fq |= kRowNanInf;
    else if (Sq == 0.0) fq |= kRowEmpty;
    if (s.flag) fp |= kRowMismatch;
    const double shp = (double)s.mxp - (double)s.rp, shq = (double)s.mxq - (double)s.rq;
    const double logSp = log(Sp) - shp, logSq = log(Sq) - shq;
    const double c = W / Sp - shp + shq;   // E_p[(P - m_P) - (Q - m_Q)]
    store_rowstat(stats_p + r, s.mxp, logSp, c, fp);
    store_rowstat(stats_q + r, s.mxq, logSq, 0.0, fq);
    float res;
    if ((fp & (kRowNanInf | kRowEmpty)) || (fq & kRowNanInf)) res = qnan();
    else if (fp & kRowMismatch) res = pinf();
    else res = (float)(c - logSp + logSq);
    if (kl) kl[r] = res;   // NULL: the records only (first pass of the JSD)
}

// ---------------------------------------------------------------------------
// Generalized JSD, second pass ([P1] commit message adding vocab_parallel_jsd:
// "reuse global normalization and reduce the two KL-to-mixture expectations
// together"). With the rows' (m, logS) of A and B from the first pass, the two
// expectations are plain sums, no centre needed:
//   KL(p || mix) = sum p (log p - log mix),  KL(q || mix) = sum q (log q - log mix),
//   mix = beta q + (1 - beta) p,
// accumulated in base-2 units (log2 p, log2 mix) and scaled by ln 2 at the end.
// ---------------------------------------------------------------------------
struct JsdRow {
    float ma, mb;                         // exact row maxima of A and B
    float la_hi, la_lo, lb_hi, lb_lo;     // logS of A and B
    float beta, omb;                      // beta, 1 - beta
};

__device__ __forceinline__ JsdRow jsd_row_constants(const RowStat &sa, const RowStat &sb, float beta) {
    return JsdRow{sa.m, sb.m, sa.logS_hi, sa.logS_lo, sb.logS_hi, sb.logS_lo, beta, 1.f - beta};
}

__device__ __forceinline__ float lg2_fast(float a) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(a));
    return y;
}

template <typename T>
struct LaneJSD {
    DF ka, kb;   // base-2 units

    __device__ __forceinline__ void init() { ka = kb = DF{0.f, 0.f}; }

    // Scalar path. fp32 inputs: accurate exponentials and logarithms,
    // double-float sums. bf16 (the unaligned head and tail of a row): the
    // hardware base-2 forms of the fast path.
    template <int n>
    __device__ __forceinline__ void push(const float (&a)[n], const float (&b)[n], const JsdRow &c) {
#pragma unroll
        for (int i = 0; i < n; ++i) {
            if constexpr (Elem<T>::kPrecise) {
                const float lp = ((a[i] - c.ma) - c.la_hi) - c.la_lo;   // a - m is exact
                const float lq = ((b[i] - c.mb) - c.lb_hi) - c.lb_lo;
                const float p = expf(lp), q = expf(lq);
                const float lmix = logf(fmaf(c.beta, q, c.omb * p));
                if (p > 0.f) df_add(ka, p * (lp - lmix) * kLog2e);
                if (q > 0.f) df_add(kb, q * (lq - lmix) * kLog2e);
            } else {
                const float xa = fmaf(a[i] - c.ma, kLog2e, -(c.la_hi + c.la_lo) * kLog2e);   // log2 p
                const float xb = fmaf(b[i] - c.mb, kLog2e, -(c.lb_hi + c.lb_lo) * kLog2e);
                const float p = ex2_fast(xa), q = ex2_fast(xb);
                const float lm = fmaxf(lg2_fast(fmaf(c.beta, q, c.omb * p)), -250.f);
                if (p > 0.f) df_add(ka, p * (xa - lm));
                if (q > 0.f) df_add(kb, q * (xb - lm));
            }
        }
    }

    // bf16 fast path on raw 16-byte words: packed f32x2 arithmetic, MUFU ex2 and
    // lg2. Terms are taken unguarded; a chunk whose sums come out non-finite (a
    // -inf logit gives 0 * inf) is redone with zero-weight terms skipped.
    template <int K>
    __device__ __forceinline__ void push_bf16(const uint4 (&ua)[K], const uint4 (&ub)[K], const JsdRow &c) {
        const float2 nma = make_float2(-c.ma, -c.ma), nmb = make_float2(-c.mb, -c.mb);
        const float la2 = -(c.la_hi + c.la_lo) * kLog2e, lb2 = -(c.lb_hi + c.lb_lo) * kLog2e;
        const float2 nla = make_float2(la2, la2), nlb = make_float2(lb2, lb2);
        const float2 l2e = make_float2(kLog2e, kLog2e), m1 = make_float2(-1.f, -1.f);
        const float2 bt = make_float2(c.beta, c.beta), ob = make_float2(c.omb, c.omb);
        float2 sa[2], sb[2];
#pragma unroll
        for (int k = 0; k < K; ++k) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 xa = __ffma2_rn(__fadd2_rn(bf16_pair(word(ua[k], q)), nma), l2e, nla);   // log2 p
                const float2 xb = __ffma2_rn(__fadd2_rn(bf16_pair(word(ub[k], q)), nmb), l2e, nlb);   // log2 q
                const float2 p = make_float2(ex2_fast(xa.x), ex2_fast(xa.y));
                const float2 qv = make_float2(ex2_fast(xb.x), ex2_fast(xb.y));
                const float2 mix = __ffma2_rn(bt, qv, __fmul2_rn(ob, p));
                const float2 lm = make_float2(fmaxf(lg2_fast(mix.x), -250.f), fmaxf(lg2_fast(mix.y), -250.f));
                const float2 da = __ffma2_rn(lm, m1, xa), db = __ffma2_rn(lm, m1, xb);
                if (k == 0 && q < 2) {
                    sa[q] = __fmul2_rn(p, da);
                    sb[q] = __fmul2_rn(qv, db);
                } else {
                    sa[q & 1] = __ffma2_rn(p, da, sa[q & 1]);
                    sb[q & 1] = __ffma2_rn(qv, db, sb[q & 1]);
                }
            }
        }
        float2 ra = __fadd2_rn(sa[0], sa[1]);
        float2 rb = __fadd2_rn(sb[0], sb[1]);
        float suma = ra.x + ra.y, sumb = rb.x + rb.y;
        if (!(fabsf(suma) < INFINITY && fabsf(sumb) < INFINITY)) {
            suma = sumb = 0.f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 xa = __ffma2_rn(__fadd2_rn(bf16_pair(word(ua[k], q)), nma), l2e, nla);
                    const float2 xb = __ffma2_rn(__fadd2_rn(bf16_pair(word(ub[k], q)), nmb), l2e, nlb);
                    const float xs[4] = {xa.x, xa.y, xb.x, xb.y};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float p = ex2_fast(xs[h]), qv = ex2_fast(xs[2 + h]);
                        const float lm = fmaxf(lg2_fast(fmaf(c.beta, qv, c.omb * p)), -250.f);
                        if (p > 0.f) suma = fmaf(p, xs[h] - lm, suma);       // zero-weight terms add nothing
                        if (qv > 0.f) sumb = fmaf(qv, xs[2 + h] - lm, sumb);
                    }
                }
            }
        }
        df_add(ka, suma);   // double-float lane sums (see Lane1::push_bf16)
        df_add(kb, sumb);
    }
};

template <typename V>
struct PartJSD {
    V ka, kb;
};

template <typename T>
__device__ __forceinline__ PartJSD<AccT<T>> jsd_warp_merge(const LaneJSD<T> &L) {
    DF a = L.ka, b = L.kb;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        df_add(a, shfl_xor(a, m));
        df_add(b, shfl_xor(b, m));
    }
    return PartJSD<AccT<T>>{df_to<AccT<T>>(a), df_to<AccT<T>>(b)};
}

// Finishes a row: JSD = ln 2 (beta KB + (1 - beta) KA) from the warps' partials
// (summed in a fixed order in fp64), and KL(p || mix), KL(q || mix) into the c
// fields of the two records (flags keep only the NaN / empty bits).
template <typename V>
__device__ __forceinline__ void finish_jsd(const PartJSD<V> *parts, int count, int64_t r, double beta, float *jsd,
                                           RowStat *stats_a, RowStat *stats_b) {
    double ka = 0.0, kb = 0.0;
    for (int w = 0; w < count; ++w) {
        ka += (double)parts[w].ka;
        kb += (double)parts[w].kb;
    }
    constexpr double kLn2 = 0.69314718055994530942;
    ka *= kLn2;
    kb *= kLn2;
    const uint32_t fa = stats_a[r].flags & (kRowNanInf | kRowEmpty), fb = stats_b[r].flags & (kRowNanInf | kRowEmpty);
    const DF ca = df_from(ka), cb = df_from(kb);
    stats_a[r].c_hi = ca.hi;
    stats_a[r].c_lo = ca.lo;
    stats_a[r].flags = fa;
    stats_b[r].c_hi = cb.hi;
    stats_b[r].c_lo = cb.lo;
    stats_b[r].flags = fb;
    jsd[r] = (fa | fb) ? qnan() : (float)(beta * kb + (1.0 - beta) * ka);
}

// Per-shard record of a row (vocabulary-sharded forms): the merged partial
// re-centred in fp64 from its centre `ref` onto the shard's exact max.
template <int kOp, typename Acc>
__device__ __forceinline__ void finish_partial(const Part1<Acc> &p, int64_t r, int V, int64_t t, int64_t vocab_start,
                                               float zt, PartialRec *parts) {
    PartialRec o;
    const double sh = (double)p.mx - (double)p.ref;   // >= 0
    const double a = exp(-sh);
    const double S = (double)p.S;
    o.m = p.mx;
    o.m_b = 0.f;
    o.S = a * S;
    o.S_b = 0.0;
    o.W = (kOp == 1 && o.S > 0.0) ? a * ((double)p.W - sh * S) : 0.0;
    o.z_t = 0.f;
    uint32_t flags = (S != S) ? kPartNanInf : 0u;
    if (kOp == 0) {
        const int64_t loc = t - vocab_start;
        if (t < 0) flags |= kPartIgnored;
        else if (loc >= 0 && loc < V) { flags |= kPartHasTarget; o.z_t = zt; }
    }
    o.flags = flags;
    parts[r] = o;
}

template <typename Acc>
__device__ __forceinline__ void finish_partial_kl(const PartKL<Acc> &s, int64_t r, PartialRec *parts) {
    PartialRec o;
    const double shp = (double)s.mxp - (double)s.rp, shq = (double)s.mxq - (double)s.rq;
    const double ap = exp(-shp), aq = exp(-shq);
    const double Sp = (double)s.Sp, Sq = (double)s.Sq;
    o.m = s.mxp;
    o.m_b = s.mxq;
    o.S = ap * Sp;
    o.S_b = aq * Sq;
    o.W = (o.S > 0.0) ? ap * ((double)s.W - (shp - shq) * Sp) : 0.0;
    o.z_t = 0.f;
    o.flags = ((Sp != Sp) ? kPartNanInf : 0u) | ((Sq != Sq) ? kPartNanInfB : 0u) | (s.flag ? kPartMismatch : 0u);
    parts[r] = o;
}

// The warp's shared centre: the max over its first round of values.
__device__ __forceinline__ float warp_centre(float c) { return fmaxf(warp_max(c), kNegBig); }

}  // namespace vp
