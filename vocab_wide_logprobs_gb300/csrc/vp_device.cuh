// vp_device.cuh -- device helpers shared by the libvp kernels (sm_103a).
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838): second commit message and the
//        reviewer's "Suggested change" (online max, sum-exp S and centred
//        weighted sum W in one read; partials re-centred on the max), and the
//        Codex thread "Guard zero rescaling before applying infinite shifts".
//
// Numerics of the online statistics (one distribution):
//   Every lane keeps S = sum_j e^{z_j - ref} and W = sum_j e^{z_j - ref} (z_j - ref)
//   against a centre `ref` that all 32 lanes of a warp share: the max of the
//   warp's first round of loads. Terms are summed in fp32 over one round of
//   loads and folded into double-float (hi + lo) accumulators with an
//   error-free two-sum; on the fp32 path every addition inside the round is
//   compensated as well (the offset fast two-sum below, FMA product errors), so
//   the row sums keep ~2^-40 relative accuracy beyond the per-term
//   exponentials. Because a warp shares one centre, the warp merge is a plain
//   double-float sum; the warp partials are re-centred on the largest centre
//   (S <- a S, W <- a (W - d S), a = e^{-d}; in fp64 on the fp32 path, and with
//   fp32 factors and double-float sums on the bf16 path), terms of zero weight
//   skipped [P1], and the row is finished in fp64.
//   A lane moves its own centre only when a value exceeds it by more than
//   kSpan (so e^{z - ref} cannot overflow); this happens only in rows whose
//   values span more than kSpan natural-log units, and the warp then merges
//   in fp64 with explicit re-centring. bf16 inputs move sooner, beyond
//   kSpanFast: their exponential takes the rounded product (z - ref) log2(e),
//   whose error is (z - ref) 2^-24 relative in e^{z - ref}, so a large value
//   far above the centre (a peak that arrives after the centre was chosen)
//   would carry that error into S whole.
//   The empty state has ref = -FLT_MAX and S = W = 0: an all -inf slice leaves
//   it unchanged and needs no special case.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vp {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -3.4028234663852886e38f;  // -FLT_MAX
constexpr float kSpan = 64.0f;                       // largest exponent a lane accumulates
constexpr float kSpanFast = 4.0f;                    // the same on the bf16 path
constexpr int kFwdThreads = 512;
constexpr int kFwdWarps = kFwdThreads / 32;
constexpr int kBwdThreads = 256;
constexpr int kBwdVecPerThread = 4;

constexpr uint32_t kRowNanInf = 1u, kRowEmpty = 2u, kRowMismatch = 4u;  // = VP_ROW_* of vp.h
constexpr uint32_t kRowSharded = 8u, kRowBadTarget = 16u;
// = VP_PART_* of vp.h
constexpr uint32_t kPartNanInf = 1u, kPartNanInfB = 2u, kPartMismatch = 4u, kPartHasTarget = 8u, kPartIgnored = 16u;

// Layout of vp_partial (40 bytes): one row's statistics over one vocabulary shard.
struct PartialRec {
    float m, m_b;
    double S, S_b, W;
    float z_t;
    uint32_t flags;
};
static_assert(sizeof(PartialRec) == 40, "vp_partial is 40 bytes");

// Device-side image of vp_rowstat (32 bytes).
struct RowStat {
    float m, logS_hi, logS_lo, c_hi, c_lo;
    uint32_t flags, r0, r1;
};
static_assert(sizeof(RowStat) == 32, "vp_rowstat is 32 bytes");

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }
__device__ __forceinline__ float pinf() { return __int_as_float(0x7f800000); }

// ---------------------------------------------------------------------------
// Row addressing: row r starts at (r / R) * s_o + (r % R) * s_i elements.
// ---------------------------------------------------------------------------
struct Rows {
    int64_t R, s_o, s_i;
    __device__ __forceinline__ int64_t off(int64_t r) const { return (r / R) * s_o + (r % R) * s_i; }
};

// ---------------------------------------------------------------------------
// Element traits: 16-byte vectors of bf16 (8) or fp32 (4).
// ---------------------------------------------------------------------------
template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int kVec = 4;
    static constexpr bool kPrecise = true;   // fp32 gradients are held to 1e-6 (absolute up to 1, relative above)
    static __device__ __forceinline__ float load1(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ void unpack(const uint4 &u, float *v) {
        v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
    }
    static __device__ __forceinline__ uint4 pack(const float *v) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
    static __device__ __forceinline__ void store1(float *p, float v) { *p = v; }
    static __device__ __forceinline__ float exp(float t) { return expf(t); }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    static constexpr bool kPrecise = false;  // bf16 gradients are held to one bf16 ulp
    static __device__ __forceinline__ float load1(const __nv_bfloat16 *p) {
        unsigned short u = __ldg(reinterpret_cast<const unsigned short *>(p));
        return __uint_as_float(((uint32_t)u) << 16);
    }
    static __device__ __forceinline__ void unpack2(uint32_t w, float &lo, float &hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
    static __device__ __forceinline__ void unpack(const uint4 &u, float *v) {
        unpack2(u.x, v[0], v[1]); unpack2(u.y, v[2], v[3]);
        unpack2(u.z, v[4], v[5]); unpack2(u.w, v[6], v[7]);
    }
    static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<uint32_t *>(&b);
    }
    static __device__ __forceinline__ uint4 pack(const float *v) {
        return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    }
    static __device__ __forceinline__ void store1(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
    // Hardware base-2 exponential (MUFU.EX2); results below 2^-126 flush to 0.
    static __device__ __forceinline__ float exp(float t) {
        float y;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t * kLog2e));
        return y;
    }
};

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void stg_stream(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Elements before the first 16-byte boundary of a row (0 .. kVec-1), capped at V.
template <typename T>
__device__ __forceinline__ int head_count(const T *p, int V) {
    int h = (int)(((16u - ((uint32_t)(uintptr_t)p & 15u)) & 15u) / sizeof(T));
    return h < V ? h : V;
}

// ---------------------------------------------------------------------------
// Double-float accumulation (error-free transformations of Knuth's two-sum).
// ---------------------------------------------------------------------------
struct DF {
    float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

// acc += x
__device__ __forceinline__ void df_add(DF &acc, float x) {
    const DF t = two_sum(acc.hi, x);
    acc.hi = t.hi;
    acc.lo = __fadd_rn(acc.lo, t.lo);
}

// acc += y (both double-float)
__device__ __forceinline__ void df_add(DF &acc, const DF &y) {
    const DF t = two_sum(acc.hi, y.hi);
    acc.hi = t.hi;
    acc.lo = __fadd_rn(__fadd_rn(acc.lo, y.lo), t.lo);
}

__device__ __forceinline__ double df_value(const DF &a) { return (double)a.hi + (double)a.lo; }

__device__ __forceinline__ DF df_from(double v) {
    const float hi = (float)v;
    // NaN / inf pass through hi; lo is 0 then
    const float lo = isfinite(v) ? (float)(v - (double)hi) : 0.f;
    return {hi, lo};
}

// hi + lo when |hi| >= |lo| (Dekker's fast two-sum)
__device__ __forceinline__ DF fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// a - b as a double-float (exact)
__device__ __forceinline__ DF df_diff(float a, float b) { return two_sum(a, -b); }

// (x_hi + x_lo) - (y_hi + y_lo) as a double-float, accurate to ~2^-44 relative
__device__ __forceinline__ DF df_sub(const DF &x, float y_hi, float y_lo) {
    const DF d = two_sum(x.hi, -y_hi);
    return {d.hi, __fadd_rn(d.lo, __fsub_rn(x.lo, y_lo))};
}

// Accurate e^(a_hi + a_lo) as a double-float (relative error ~1e-8).
// Method (Cody and Waite's argument reduction followed by a Taylor series):
//   k = nearest integer to a / ln 2, r = a - k ln 2 with ln 2 split into three
//   parts so that k * part is exact for the first two (|k| < 256), giving r as
//   a double-float with |r| <= ln 2 / 2; then e^r = 1 + r + sum_{n=2..9} r^n / n!
//   (truncation error < 3e-10), the tail evaluated in fp32 by Horner's rule;
//   finally the result is scaled by 2^k. Arguments below -104 give 0 (the
//   fp32 result underflows); NaN propagates.
__device__ __forceinline__ DF exp_df(float a_hi, float a_lo) {
    constexpr float kL1 = 0.693145751953125f;        // ln 2, 16 significant bits
    constexpr float kL2 = 1.4286197256296873e-06f;   // next 16 bits
    constexpr float kL3 = -1.2905320041778356e-11f;  // remainder
    if (!(a_hi > -104.f)) return {a_hi != a_hi ? a_hi : 0.f, 0.f};
    const float k = rintf(a_hi * kLog2e);
    const float x1 = fmaf(-k, kL1, a_hi);             // exact
    DF r = two_sum(x1, -k * kL2);                     // k * kL2 exact
    r.lo = __fadd_rn(r.lo, fmaf(-k, kL3, a_lo));
    const float h = r.hi;
    float t = 2.7557318844628753e-06f;                // 1/9!
    t = fmaf(t, h, 2.4801587642286904e-05f);          // 1/8!
    t = fmaf(t, h, 1.9841270113829523e-04f);          // 1/7!
    t = fmaf(t, h, 1.3888889225199819e-03f);          // 1/6!
    t = fmaf(t, h, 8.3333337679505350e-03f);          // 1/5!
    t = fmaf(t, h, 4.1666667908430100e-02f);          // 1/4!
    t = fmaf(t, h, 1.6666667163372040e-01f);          // 1/3!
    t = fmaf(t, h, 0.5f);                             // 1/2!
    const float tail = (h * h) * t;                   // r^2/2! + ... + r^9/9!
    const DF s = fast_two_sum(1.f, h);                // 1 + r_hi
    const float lo = __fadd_rn(__fadd_rn(s.lo, r.lo), fmaf(h, r.lo, tail));
    DF e = fast_two_sum(s.hi, lo);
    // scale by 2^k in two exact steps (k in [-151, 128])
    const int ki = (int)k;
    const int k1 = ki / 2, k2 = ki - k1;
    const float f1 = __int_as_float((k1 + 127) << 23), f2 = __int_as_float((k2 + 127) << 23);
    e.hi = (e.hi * f1) * f2;
    e.lo = (e.lo * f1) * f2;
    return e;
}

// e^x - 1 for |x| < 1/2 by its Taylor series to x^8/8! (relative error < 1e-8 there):
// used where e^x - 1 would cancel.
__device__ __forceinline__ float expm1_small(float x) {
    float t = 2.4801587301587302e-05f;      // 1/8!
    t = fmaf(t, x, 1.9841269841269841e-04f);  // 1/7!
    t = fmaf(t, x, 1.3888888888888889e-03f);  // 1/6!
    t = fmaf(t, x, 8.3333333333333333e-03f);  // 1/5!
    t = fmaf(t, x, 4.1666666666666667e-02f);  // 1/4!
    t = fmaf(t, x, 1.6666666666666667e-01f);  // 1/3!
    t = fmaf(t, x, 0.5f);                     // 1/2!
    return fmaf(t * x, x, x);                 // x + x^2 (1/2 + x/6 + ...)
}

// expm1_small of each lane (f32x2, the same operations)
__device__ __forceinline__ float2 expm1_small2(float2 x) {
    float2 t = make_float2(2.4801587301587302e-05f, 2.4801587301587302e-05f);
    t = __ffma2_rn(t, x, make_float2(1.9841269841269841e-04f, 1.9841269841269841e-04f));
    t = __ffma2_rn(t, x, make_float2(1.3888888888888889e-03f, 1.3888888888888889e-03f));
    t = __ffma2_rn(t, x, make_float2(8.3333333333333333e-03f, 8.3333333333333333e-03f));
    t = __ffma2_rn(t, x, make_float2(4.1666666666666667e-02f, 4.1666666666666667e-02f));
    t = __ffma2_rn(t, x, make_float2(1.6666666666666667e-01f, 1.6666666666666667e-01f));
    t = __ffma2_rn(t, x, make_float2(0.5f, 0.5f));
    return __ffma2_rn(__fmul2_rn(t, x), x, x);
}

// e^(t_hi + t_lo) as one fp32 value, from the hardware base-2 exponential
// with its argument a = (t_hi + t_lo) log2(e) carried as a_hi + a_lo (the
// product with the fp32 part of log2(e) exact inside an FMA, the low part of
// log2(e) and t_lo added to a_lo): e = 2^a_hi (1 + a_lo ln 2). The relative
// error is that of the hardware unit (below 1.5e-7, measured on GB300 over
// dense argument sweeps) plus (a_lo ln 2)^2 / 2 < 2^-38; a plain fp32 argument
// t log2(e) would add up to |a| 2^-24 (3.5e-6 at |t| = 40). Used by the fp32
// forward sums, whose results are held to 1e-6 (gradients) and 2e-5 (outputs).
__device__ __forceinline__ float exp_split(float t_hi, float t_lo) {
    constexpr float kL = 1.4426950408889634f, kLlo = 1.925963033500011e-08f, kLn2 = 0.6931471805599453f;
    const float a_hi = t_hi * kL;
    float a_lo = fmaf(t_hi, kL, -a_hi);
    a_lo = fmaf(t_hi, kLlo, a_lo);
    a_lo = fmaf(t_lo, kL, a_lo);
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(a_hi));
    return e == 0.f ? 0.f : fmaf(e, a_lo * kLn2, e);   // a_lo is NaN where t_hi is infinite
}

// ---------------------------------------------------------------------------
// Packed (f32x2) forms of two_sum, df_sub and exp_split: two independent
// values per instruction, each lane rounded exactly as the scalar form rounds
// it (negations are folded into FMAs with -1 or with negated constants, which
// round symmetrically), so the results are bitwise those of the scalar forms.
// ---------------------------------------------------------------------------
struct DF2 {
    float2 hi, lo;
};

__device__ __forceinline__ float2 f2(float x) { return make_float2(x, x); }

// two_sum of each lane
__device__ __forceinline__ DF2 two_sum2(float2 a, float2 b) {
    const float2 m1 = f2(-1.f);
    const float2 s = __fadd2_rn(a, b);
    const float2 bb = __ffma2_rn(a, m1, s);                            // s - a
    const float2 r = __ffma2_rn(__ffma2_rn(bb, m1, s), m1, a);         // a - (s - bb)
    return {s, __fadd2_rn(r, __ffma2_rn(bb, m1, b))};                  // + (b - bb)
}

// two_sum(a, -y) of each lane
__device__ __forceinline__ DF2 two_diff2(float2 a, float2 y) {
    const float2 m1 = f2(-1.f);
    const float2 s = __ffma2_rn(y, m1, a);                             // a - y
    const float2 bb = __ffma2_rn(a, m1, s);                            // s - a
    const float2 r = __ffma2_rn(__ffma2_rn(bb, m1, s), m1, a);         // a - (s - bb)
    return {s, __ffma2_rn(__fadd2_rn(y, bb), m1, r)};                  // + (-y - bb)
}

// df_sub(x, y.hi, y.lo) of each lane
__device__ __forceinline__ DF2 df_sub2(const DF2 &x, const DF2 &y) {
    const DF2 d = two_diff2(x.hi, y.hi);
    return {d.hi, __fadd2_rn(d.lo, __ffma2_rn(y.lo, f2(-1.f), x.lo))};
}

// exp_split of each lane, its zero test included (bitwise exp_split's)
__device__ __forceinline__ float2 exp_split2(const DF2 &t) {
    constexpr float kL = 1.4426950408889634f, kLlo = 1.925963033500011e-08f, kLn2 = 0.6931471805599453f;
    const float2 a_hi = __fmul2_rn(t.hi, f2(kL));
    float2 na = __ffma2_rn(t.hi, f2(-kL), a_hi);                       // -(t_hi kL - a_hi)
    na = __ffma2_rn(t.hi, f2(-kLlo), na);
    na = __ffma2_rn(t.lo, f2(-kL), na);                                // -a_lo
    float2 e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(a_hi.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(a_hi.y));
    const float2 r = __ffma2_rn(e, __fmul2_rn(na, f2(-kLn2)), e);      // e (1 + a_lo ln 2)
    return make_float2(e.x == 0.f ? 0.f : r.x, e.y == 0.f ? 0.f : r.y);   // a_lo is NaN where t_hi is infinite
}

// ---------------------------------------------------------------------------
// Offset fast two-sum. A running sum started at a power of two K that exceeds
// every addend keeps an exponent at least that of each addend, so Dekker's fast
// two-sum (h = s + e; error = e - (h - s)) gives each addition's rounding error
// exactly in three operations, against the six of two_sum; at the end s - K is
// exact too (K is a multiple of the final sum's ulp).
// ---------------------------------------------------------------------------
// k of K = 2^k above e^{c - ref} for a chunk whose largest value is c: the 2^-8
// margin covers the rounding of (c - ref) log2(e) and of exp_split (both below
// 2e-5 in log2 units), so every exponential of the chunk is below 2^k. Clamped
// to [-100, 100]: a chunk below 2^-100 of its centre is negligible in the row's
// sum however it is added, and a non-finite c belongs to a row whose sums are
// NaN already.
__device__ __forceinline__ int offset_log2(float c, float ref) {
    const float x = fmaf(c - ref, 1.4426950408889634f, 0.00390625f);
    return min(max(__float2int_rd(x), -101), 99) + 1;
}

__device__ __forceinline__ float pow2f(int k) { return __int_as_float((k + 127) << 23); }   // k in [-126, 127]

// s += e in each lane, its rounding error added to lo (requires |s| >= 2^j > |e| for some j)
__device__ __forceinline__ void fast_acc2(float2 &s, float2 &lo, float2 e) {
    const float2 m1 = f2(-1.f);
    const float2 h = __fadd2_rn(s, e);
    lo = __fadd2_rn(lo, __ffma2_rn(__ffma2_rn(s, m1, h), m1, e));   // e - (h - s)
    s = h;
}

// Product (x_hi + x_lo) * (y_hi + y_lo) rounded once to fp32.
__device__ __forceinline__ float df_mul_round(const DF &x, const DF &y) {
    const float p = x.hi * y.hi;
    const float pe = fmaf(x.hi, y.hi, -p);
    return p + fmaf(x.hi, y.lo, fmaf(x.lo, y.hi, pe));
}

__device__ __forceinline__ DF shfl_xor(const DF &a, int m) {
    return {__shfl_xor_sync(0xffffffffu, a.hi, m), __shfl_xor_sync(0xffffffffu, a.lo, m)};
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ void store_rowstat(RowStat *dst, float m, double logS, double c, uint32_t flags) {
    const DF l = df_from(logS), cc = df_from(c);
    RowStat s{m, l.hi, l.lo, cc.hi, cc.lo, flags, 0u, 0u};
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    const uint4 *src = reinterpret_cast<const uint4 *>(&s);
    d[0] = src[0];
    d[1] = src[1];
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization (launch_pdl) may be scheduled while the stream's previous grid
// is still finishing: it calls pdl_enter() before its first global-memory
// access, and the wait returns once every grid it depends on has completed and
// that grid's memory operations are visible.
// kTrigger also lets the stream's next grid be scheduled once every CTA of this
// grid has done so or exited, so that every CTA of this grid is resident by
// then and a waiting dependent never holds a slot one of them needs. The
// elementwise backward grids (many short CTAs) trigger: their dependents then
// arrive as the last wave drains. The persistent forward grids do not: they
// would trigger at once, and a dependent CTA would sit waiting beside them for
// the whole scan (measured on GB300: the step took 3.47-3.51 ms with every
// kernel triggering, 3.34 ms with the backwards only, 3.37 ms without PDL).
// Without the launch attribute both instructions are no-ops.
// ---------------------------------------------------------------------------
template <bool kTrigger>
__device__ __forceinline__ void pdl_enter() {
    if (kTrigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

#ifndef VP_PDL
#define VP_PDL 1
#endif

// kernel<<<grid, block, smem, stream>>>(args...) with programmatic stream
// serialization (VP_PDL = 0 launches without it)
template <typename K, typename... Args>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = VP_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ RowStat load_rowstat(const RowStat *p) {
    RowStat s;
    uint4 *d = reinterpret_cast<uint4 *>(&s);
    d[0] = __ldg(reinterpret_cast<const uint4 *>(p));
    d[1] = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
    return s;
}

}  // namespace vp
