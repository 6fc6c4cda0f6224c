// vp_device.cuh -- device helpers shared by the libvp kernels (sm_103a).
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838).
//
// Online statistics of one row slice, kept per thread and merged across
// threads, warps and CTAs [P1, second commit message and the reviewer's
// "Suggested change"]:
//   m  running centre. On the fp32 path it is the exact running max. On the
//      bf16 path it is a stale max that only moves when a value exceeds it by
//      more than kTau (so the per-element exponent stays <= kTau and the
//      rescale is rare); each thread also tracks its true max and re-centres
//      on it before the merge, so the merged m is the exact row max on both
//      paths,
//   S  = sum_j e^{z_j - m},
//   W  = sum_j e^{z_j - m} (z_j - m).
// When the centre moves from m to m' the partial becomes
//   S <- a S,  W <- a (W - (m' - m) S),  a = e^{m - m'},
// and a term whose weight a S is exactly 0 is dropped, so an overflowing shift
// (a row spanning +-3e38) never meets a zero weight as 0 * inf [P1, Codex
// thread "Guard zero rescaling before applying infinite shifts"].
//
// The empty state has m = -FLT_MAX, S = W = 0: an all -inf slice leaves it
// unchanged, and e^{-inf - (-FLT_MAX)} = 0 needs no special case.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vp {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -3.4028234663852886e38f;  // -FLT_MAX
constexpr int kFwdThreads = 512;
constexpr int kBwdThreads = 256;
constexpr int kBwdVecPerThread = 4;

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
    // Accurate exponential for the fp32 path (gradients are held to 1e-6).
    static __device__ __forceinline__ float exp(float t) { return expf(t); }
    static constexpr float kTau = 0.0f;  // exact running max
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
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
    static constexpr float kTau = 8.0f;  // allowed staleness of the centre (natural-log units)
    // Hardware base-2 exponential; bf16 results need far less than fp32 accuracy.
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
// (m, S, W) of one distribution.
// ---------------------------------------------------------------------------
struct Stat {
    float m, S, W;
    __device__ __forceinline__ static Stat empty() { return {kNegBig, 0.f, 0.f}; }
};

// Move the centre of a partial up to m_new (> s.m).
template <bool kW>
__device__ __forceinline__ void recentre(Stat &s, float m_new) {
    float d = m_new - s.m;          // > 0, may overflow to +inf
    float a = expf(-d);             // 0 when the shift is huge
    if (kW) s.W = (a == 0.f) ? 0.f : a * (s.W - d * s.S);
    s.S *= a;                       // keeps a NaN
    s.m = m_new;
}

// Fold partial b into the running merge o (o.m already the max of both).
template <bool kW>
__device__ __forceinline__ void fold(Stat &o, const Stat &b) {
    float a = (b.m == o.m) ? 1.f : expf(b.m - o.m);
    float w = a * b.S;
    if (w != 0.f) {                 // zero-weight partials are skipped; NaN is kept
        o.S += w;
        if (kW) o.W += a * (b.W - (o.m - b.m) * b.S);
    }
}

template <bool kW>
__device__ __forceinline__ Stat merge(const Stat &x, const Stat &y) {
    Stat o;
    o.m = fmaxf(x.m, y.m);
    o.S = 0.f;
    o.W = 0.f;
    fold<kW>(o, x);
    fold<kW>(o, y);
    return o;
}

template <bool kW>
__device__ __forceinline__ Stat shfl_down(const Stat &s, int off) {
    Stat o;
    o.m = __shfl_down_sync(0xffffffffu, s.m, off);
    o.S = __shfl_down_sync(0xffffffffu, s.S, off);
    o.W = kW ? __shfl_down_sync(0xffffffffu, s.W, off) : 0.f;
    return o;
}

// Block-wide merge in a fixed order; the result is valid in thread 0.
template <bool kW, int kThreads>
__device__ __forceinline__ Stat block_merge(Stat s) {
    __shared__ Stat part[kThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s = merge<kW>(s, shfl_down<kW>(s, off));
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = s;
    __syncthreads();
    if (warp == 0) {
        s = lane < kThreads / 32 ? part[lane] : Stat::empty();
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s = merge<kW>(s, shfl_down<kW>(s, off));
    }
    return s;
}

// ---------------------------------------------------------------------------
// Paired statistics for KL(P||Q): (m_P, S_P, m_Q, S_Q, W, flag) with
// W = sum_{p_j > 0} e^{P_j - m_P} ((P_j - m_P) - (Q_j - m_Q)) and flag set
// when some P_j > -inf has Q_j = -inf [P1, reviewer's suggested change].
// Moving the centres by (dp, dq) turns W into a_P (W - (dp - dq) S_P).
// ---------------------------------------------------------------------------
struct KLStat {
    float mp, Sp, mq, Sq, W;
    int flag;
    __device__ __forceinline__ static KLStat empty() { return {kNegBig, 0.f, kNegBig, 0.f, 0.f, 0}; }
};

__device__ __forceinline__ void kl_recentre(KLStat &s, float mp_new, float mq_new) {
    float dp = mp_new - s.mp, dq = mq_new - s.mq;   // >= 0
    float ap = (dp == 0.f) ? 1.f : expf(-dp);
    float aq = (dq == 0.f) ? 1.f : expf(-dq);
    s.W = (ap == 0.f) ? 0.f : ap * (s.W - (dp - dq) * s.Sp);
    s.Sp *= ap;
    s.Sq *= aq;
    s.mp = mp_new;
    s.mq = mq_new;
}

__device__ __forceinline__ void kl_fold(KLStat &o, const KLStat &b) {
    float ap = (b.mp == o.mp) ? 1.f : expf(b.mp - o.mp);
    float aq = (b.mq == o.mq) ? 1.f : expf(b.mq - o.mq);
    float wq = aq * b.Sq;
    if (wq != 0.f) o.Sq += wq;
    float wp = ap * b.Sp;
    if (wp != 0.f) {
        o.Sp += wp;
        o.W += ap * (b.W - ((o.mp - b.mp) - (o.mq - b.mq)) * b.Sp);
    }
    o.flag |= b.flag;
}

__device__ __forceinline__ KLStat kl_merge(const KLStat &x, const KLStat &y) {
    KLStat o;
    o.mp = fmaxf(x.mp, y.mp);
    o.mq = fmaxf(x.mq, y.mq);
    o.Sp = o.Sq = o.W = 0.f;
    o.flag = 0;
    kl_fold(o, x);
    kl_fold(o, y);
    return o;
}

__device__ __forceinline__ KLStat kl_shfl_down(const KLStat &s, int off) {
    KLStat o;
    o.mp = __shfl_down_sync(0xffffffffu, s.mp, off);
    o.Sp = __shfl_down_sync(0xffffffffu, s.Sp, off);
    o.mq = __shfl_down_sync(0xffffffffu, s.mq, off);
    o.Sq = __shfl_down_sync(0xffffffffu, s.Sq, off);
    o.W = __shfl_down_sync(0xffffffffu, s.W, off);
    o.flag = __shfl_down_sync(0xffffffffu, s.flag, off);
    return o;
}

template <int kThreads>
__device__ __forceinline__ KLStat kl_block_merge(KLStat s) {
    __shared__ KLStat part[kThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s = kl_merge(s, kl_shfl_down(s, off));
    int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = s;
    __syncthreads();
    if (warp == 0) {
        s = lane < kThreads / 32 ? part[lane] : KLStat::empty();
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s = kl_merge(s, kl_shfl_down(s, off));
    }
    return s;
}

}  // namespace vp
