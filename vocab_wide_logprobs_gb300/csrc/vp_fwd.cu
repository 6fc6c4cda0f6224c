// vp_fwd.cu -- single-read forward kernels: logprobs, entropy, KL statistics.
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838): second commit message and the
//        reviewer's "Suggested change" (one read of each logit: online max,
//        sum-exp S and the max-centred weighted sum W; H = log S - W/S and
//        KL = W/S_A - log S_A + log S_B; partial results re-centred on the
//        max), the support-mismatch flag, and the Codex thread on zero-weight
//        terms.
//   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton", "Implementation"
//        (logp = target logit - LSE).
//
// Shape: one CTA of 512 threads per row. The row is read once with 16-byte
// non-caching loads (four in flight per thread); a scalar head and tail cover
// rows that do not start on a 16-byte boundary. Each thread keeps its own
// online statistics with two interleaved accumulators, then the CTA merges
// them (warp shuffles, then one warp over the per-warp partials) in a fixed
// order. The decomposition depends only on V, the dtype and the row's
// address modulo 16, so a row's result does not depend on N or on the other
// rows (batch invariance).
#include "vp_device.cuh"
#include "vp_launch.h"

namespace vp {

// Per-thread accumulator for one distribution: two interleaved partial sums
// that share the centre m; mx is the thread's true running max.
template <typename T, bool kW>
struct Acc {
    float m, mx, S0, S1, W0, W1;

    __device__ __forceinline__ static Acc empty() { return {kNegBig, kNegBig, 0.f, 0.f, 0.f, 0.f}; }

    __device__ __forceinline__ void move_centre(float m_new) {
        float d = m_new - m;
        float a = expf(-d);
        if (kW) {
            W0 = (a == 0.f) ? 0.f : a * (W0 - d * S0);
            W1 = (a == 0.f) ? 0.f : a * (W1 - d * S1);
        }
        S0 *= a;
        S1 *= a;
        m = m_new;
    }

    template <int n>
    __device__ __forceinline__ void push(const float (&v)[n]) {
        float c = v[0];
#pragma unroll
        for (int i = 1; i < n; ++i) c = fmaxf(c, v[i]);
        mx = fmaxf(mx, c);
        if (c > m + Elem<T>::kTau) move_centre(c);
#pragma unroll
        for (int i = 0; i < n; ++i) {
            float t = v[i] - m;
            float e = Elem<T>::exp(t);
            // e is exactly 0 below t = -104, so clamping t keeps 0 * (-inf) out of W
            if (i & 1) { S1 += e; if (kW) W1 = fmaf(e, fmaxf(t, -128.f), W1); }
            else       { S0 += e; if (kW) W0 = fmaf(e, fmaxf(t, -128.f), W0); }
        }
    }

    __device__ __forceinline__ Stat result() {
        if (mx > m) move_centre(mx);
        return {m, S0 + S1, W0 + W1};
    }
};

template <typename T>
struct KLAcc {
    float mp, mq, mxp, mxq, Sp0, Sp1, Sq0, Sq1, W0, W1;
    int flag;

    __device__ __forceinline__ static KLAcc empty() {
        return {kNegBig, kNegBig, kNegBig, kNegBig, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0};
    }

    __device__ __forceinline__ void move_centres(float mp_new, float mq_new) {
        float dp = mp_new - mp, dq = mq_new - mq;
        float ap = (dp == 0.f) ? 1.f : expf(-dp);
        float aq = (dq == 0.f) ? 1.f : expf(-dq);
        float sh = dp - dq;
        W0 = (ap == 0.f) ? 0.f : ap * (W0 - sh * Sp0);
        W1 = (ap == 0.f) ? 0.f : ap * (W1 - sh * Sp1);
        Sp0 *= ap; Sp1 *= ap;
        Sq0 *= aq; Sq1 *= aq;
        mp = mp_new;
        mq = mq_new;
    }

    template <int n>
    __device__ __forceinline__ void push(const float (&p)[n], const float (&q)[n]) {
        float cp = p[0], cq = q[0];
#pragma unroll
        for (int i = 1; i < n; ++i) { cp = fmaxf(cp, p[i]); cq = fmaxf(cq, q[i]); }
        mxp = fmaxf(mxp, cp);
        mxq = fmaxf(mxq, cq);
        bool up = cp > mp + Elem<T>::kTau, uq = cq > mq + Elem<T>::kTau;
        if (up || uq) move_centres(up ? cp : mp, uq ? cq : mq);
        int fl = 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            float tp = p[i] - mp, tq = q[i] - mq;
            float ep = Elem<T>::exp(tp), eq = Elem<T>::exp(tq);
            float dl = (ep > 0.f) ? (tp - tq) : 0.f;  // zero-weight terms add nothing
            if (i & 1) { Sp1 += ep; Sq1 += eq; W1 = fmaf(ep, dl, W1); }
            else       { Sp0 += ep; Sq0 += eq; W0 = fmaf(ep, dl, W0); }
            fl |= (q[i] == -INFINITY) & (p[i] > -INFINITY);
        }
        flag |= fl;
    }

    __device__ __forceinline__ KLStat result() {
        if (mxp > mp || mxq > mq) move_centres(fmaxf(mxp, mp), fmaxf(mxq, mq));
        return {mp, Sp0 + Sp1, mq, Sq0 + Sq1, W0 + W1, flag};
    }
};

// kOp: 0 = logprobs (S only), 1 = entropy (S and W).
template <int kOp, typename T>
__global__ void __launch_bounds__(kFwdThreads)
stats_fwd_kernel(const T *__restrict__ x, int V, Rows rows, const int64_t *__restrict__ targets,
                 int64_t vocab_start, float *__restrict__ out, float *__restrict__ m_out,
                 float *__restrict__ logS_out, int32_t *__restrict__ err) {
    constexpr bool kW = kOp == 1;
    constexpr int kVec = Elem<T>::kVec;
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
    const T *row = x + rows.off(r);
    Acc<T, kW> acc = Acc<T, kW>::empty();

    const int head = head_count(row, V);
    const int nv = (V - head) / kVec;
    const int tail0 = head + nv * kVec;
    if (tid < head) { float v[1] = {Elem<T>::load1(row + tid)}; acc.push(v); }
    if (tid < V - tail0) { float v[1] = {Elem<T>::load1(row + tail0 + tid)}; acc.push(v); }

    const uint4 *vrow = reinterpret_cast<const uint4 *>(row + head);
    int i = tid;
    for (; i + 3 * kFwdThreads < nv; i += 4 * kFwdThreads) {
        uint4 u[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) u[k] = ldg_stream(vrow + i + k * kFwdThreads);
        float v[4 * kVec];
#pragma unroll
        for (int k = 0; k < 4; ++k) Elem<T>::unpack(u[k], v + k * kVec);
        acc.push(v);
    }
    for (; i < nv; i += kFwdThreads) {
        float v[kVec];
        Elem<T>::unpack(ldg_stream(vrow + i), v);
        acc.push(v);
    }

    Stat s = block_merge<kW, kFwdThreads>(acc.result());
    if (tid != 0) return;
    const float logS = logf(s.S);
    m_out[r] = s.m;
    logS_out[r] = logS;
    const bool invalid = !(s.S > 0.f);          // NaN / +inf seen, or an all -inf row
    if (kOp == 1) {
        out[r] = invalid ? __int_as_float(0x7fc00000) : logS - s.W / s.S;
    } else {
        const int64_t t = targets[r];
        if (t < 0) { out[r] = 0.f; return; }    // ignored target
        const int64_t loc = t - vocab_start;
        if (loc < 0 || loc >= V) {
            out[r] = __int_as_float(0x7fc00000);
            if (err) atomicOr(err, VP_ERRBIT_TARGET_);
            return;
        }
        out[r] = invalid ? __int_as_float(0x7fc00000) : (Elem<T>::load1(row + loc) - s.m) - logS;
    }
}

// KL(P||Q) statistics from one read of P and Q. P and Q share the row layout;
// when their addresses differ modulo 16 the row is read element by element.
template <typename T>
__global__ void __launch_bounds__(kFwdThreads)
kl_fwd_kernel(const T *__restrict__ P, const T *__restrict__ Q, int V, Rows rows,
              float *__restrict__ kl, float *__restrict__ mp_out, float *__restrict__ logSp_out,
              float *__restrict__ mq_out, float *__restrict__ logSq_out) {
    constexpr int kVec = Elem<T>::kVec;
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t off = rows.off(r);
    const T *prow = P + off, *qrow = Q + off;
    KLAcc<T> acc = KLAcc<T>::empty();

    const bool same_phase = (((uintptr_t)prow ^ (uintptr_t)qrow) & 15u) == 0;
    const int head = same_phase ? head_count(prow, V) : V;
    const int nv = (V - head) / kVec;
    const int tail0 = head + nv * kVec;
    for (int j = tid; j < head; j += kFwdThreads) {
        float p[1] = {Elem<T>::load1(prow + j)}, q[1] = {Elem<T>::load1(qrow + j)};
        acc.push(p, q);
    }
    if (tid < V - tail0) {
        float p[1] = {Elem<T>::load1(prow + tail0 + tid)}, q[1] = {Elem<T>::load1(qrow + tail0 + tid)};
        acc.push(p, q);
    }
    const uint4 *vp = reinterpret_cast<const uint4 *>(prow + head);
    const uint4 *vq = reinterpret_cast<const uint4 *>(qrow + head);
    int i = tid;
    for (; i + kFwdThreads < nv; i += 2 * kFwdThreads) {
        uint4 up[2], uq[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            up[k] = ldg_stream(vp + i + k * kFwdThreads);
            uq[k] = ldg_stream(vq + i + k * kFwdThreads);
        }
        float p[2 * kVec], q[2 * kVec];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            Elem<T>::unpack(up[k], p + k * kVec);
            Elem<T>::unpack(uq[k], q + k * kVec);
        }
        acc.push(p, q);
    }
    for (; i < nv; i += kFwdThreads) {
        float p[kVec], q[kVec];
        Elem<T>::unpack(ldg_stream(vp + i), p);
        Elem<T>::unpack(ldg_stream(vq + i), q);
        acc.push(p, q);
    }

    KLStat s = kl_block_merge<kFwdThreads>(acc.result());
    if (tid != 0) return;
    const float logSp = logf(s.Sp), logSq = logf(s.Sq);
    mp_out[r] = s.mp;
    logSp_out[r] = logSp;
    mq_out[r] = s.mq;
    logSq_out[r] = logSq;
    float res;
    if (s.Sp != s.Sp || s.Sq != s.Sq || !(s.Sp > 0.f)) res = __int_as_float(0x7fc00000);
    else if (s.flag) res = __int_as_float(0x7f800000);
    else res = s.W / s.Sp - logSp + logSq;
    kl[r] = res;
}

// ---------------------------------------------------------------------------
// Launchers (called by the C ABI after argument checks).
// ---------------------------------------------------------------------------
template <int kOp, typename T>
static cudaError_t launch_stats(const StatsArgs &a) {
    stats_fwd_kernel<kOp, T><<<(unsigned)a.N, kFwdThreads, 0, a.stream>>>(
        static_cast<const T *>(a.x), (int)a.V, Rows{a.R, a.s_o, a.s_i}, a.targets, a.vocab_start, a.out,
        a.m, a.logS, a.err);
    return cudaGetLastError();
}

cudaError_t launch_logprobs_fwd(const StatsArgs &a) {
    return a.bf16 ? launch_stats<0, __nv_bfloat16>(a) : launch_stats<0, float>(a);
}

cudaError_t launch_entropy_fwd(const StatsArgs &a) {
    return a.bf16 ? launch_stats<1, __nv_bfloat16>(a) : launch_stats<1, float>(a);
}

template <typename T>
static cudaError_t launch_kl_t(const KLFwdArgs &a) {
    kl_fwd_kernel<T><<<(unsigned)a.N, kFwdThreads, 0, a.stream>>>(
        static_cast<const T *>(a.p), static_cast<const T *>(a.q), (int)a.V, Rows{a.R, a.s_o, a.s_i}, a.kl,
        a.mp, a.logSp, a.mq, a.logSq);
    return cudaGetLastError();
}

cudaError_t launch_kl_fwd(const KLFwdArgs &a) {
    return a.bf16 ? launch_kl_t<__nv_bfloat16>(a) : launch_kl_t<float>(a);
}

}  // namespace vp
