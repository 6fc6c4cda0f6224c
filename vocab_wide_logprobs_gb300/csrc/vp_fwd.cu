// vp_fwd.cu -- CTA-per-row KL forward, for A and B rows that differ modulo 16 bytes.
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838): second commit message and the
//        reviewer's "Suggested change" (one read of each logit: online max,
//        sum-exp S and the max-centred weighted sum W; H = log S - W/S and
//        KL = W/S_A - log S_A + log S_B; partial results re-centred on the
//        max; support mismatch as a flag decided on the logits), and the
//        Codex thread "Guard zero rescaling before applying infinite shifts".
//   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton", "Implementation"
//        (logp = target logit - LSE).
//
// The persistent TMA-ring kernels of vp_fwd_tma.cu copy P and Q rows with one
// shared 16-byte phase; when A and B differ modulo 16 bytes this kernel reads
// them instead. Shape: one CTA of 512 threads (16 warps) per row, the row read
// once with 16-byte non-caching loads (two of P and two of Q in flight per
// thread), or element by element when P and Q cannot both be read as vectors. Each warp accumulates against one shared centre (the max of its
// first round of loads), so merging its lanes is a double-float sum; the 16
// warp partials are re-centred and merged in fp64 by warp 0, which also
// finishes the row in fp64 and writes the fp32 output and the vp_rowstat
// record. The decomposition depends only on V, the dtype and the row's address
// modulo 16, so a row's result does not depend on N or on the other rows.
#include "vp_stats.cuh"

namespace vp {

// ---------------------------------------------------------------------------
// KL(P||Q): paired statistics from one read of P and Q
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kFwdThreads)
kl_fwd_kernel(const T *__restrict__ P, const T *__restrict__ Q, int V, Rows rows, float *__restrict__ kl,
              RowStat *__restrict__ stats_p, RowStat *__restrict__ stats_q, PartialRec *__restrict__ shard_parts) {
    constexpr int kVec = Elem<T>::kVec;
    constexpr int kRound = 2;
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t off = rows.off(r);
    const T *prow = P + off, *qrow = Q + off;

    // P and Q read as vectors only when they share their address modulo 16
    const bool same_phase = (((uintptr_t)prow ^ (uintptr_t)qrow) & 15u) == 0;
    const int head = same_phase ? head_count(prow, V) : V;
    const int nv = (V - head) / kVec;
    const int tail0 = head + nv * kVec;
    const uint4 *vp = reinterpret_cast<const uint4 *>(prow + head);
    const uint4 *vq = reinterpret_cast<const uint4 *>(qrow + head);

    LaneKL<T> acc;
    {
        uint4 up[kRound], uq[kRound];
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            const int i = tid + k * kFwdThreads;
            if (i < nv) { up[k] = ldg_stream(vp + i); uq[k] = ldg_stream(vq + i); }
        }
        float p[kRound * kVec], q[kRound * kVec];
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            if (tid + k * kFwdThreads < nv) {
                Elem<T>::unpack(up[k], p + k * kVec);
                Elem<T>::unpack(uq[k], q + k * kVec);
            } else {
#pragma unroll
                for (int e = 0; e < kVec; ++e) p[k * kVec + e] = q[k * kVec + e] = -INFINITY;
            }
        }
        float cp = p[0], cq = q[0];
#pragma unroll
        for (int i = 1; i < kRound * kVec; ++i) { cp = fmaxf(cp, p[i]); cq = fmaxf(cq, q[i]); }
        acc.init(warp_centre(cp), warp_centre(cq));
        acc.push(p, q);
    }
    int i = tid + kRound * kFwdThreads;
    for (; i + (kRound - 1) * kFwdThreads < nv; i += kRound * kFwdThreads) {
        uint4 up[kRound], uq[kRound];
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            up[k] = ldg_stream(vp + i + k * kFwdThreads);
            uq[k] = ldg_stream(vq + i + k * kFwdThreads);
        }
        float p[kRound * kVec], q[kRound * kVec];
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
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
    for (int j = tid; j < head; j += kFwdThreads) {
        float p[1] = {Elem<T>::load1(prow + j)}, q[1] = {Elem<T>::load1(qrow + j)};
        acc.push(p, q);
    }
    if (tid < V - tail0) {
        float p[1] = {Elem<T>::load1(prow + tail0 + tid)}, q[1] = {Elem<T>::load1(qrow + tail0 + tid)};
        acc.push(p, q);
    }

    __shared__ PartKL<AccT<T>> parts[kFwdWarps];
    const PartKL<AccT<T>> w = kl_warp_merge(acc);
    if ((tid & 31) == 0) parts[tid >> 5] = w;
    __syncthreads();
    if (tid >= 32) return;
    const PartKL<AccT<T>> s = kl_merge_parts(parts, kFwdWarps);
    if (tid == 0) {
        if (shard_parts) finish_partial_kl(s, r, shard_parts);
        else finish_kl(s, r, kl, stats_p, stats_q);
    }
}

// ---------------------------------------------------------------------------
// Generalized JSD, second pass, when A and B do not share their address modulo
// 16: one CTA per row, element by element (vp_stats.cuh, LaneJSD::push).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kFwdThreads)
jsd_fwd_kernel(const T *__restrict__ A, const T *__restrict__ B, int V, Rows rows, float beta,
               float *__restrict__ jsd, RowStat *__restrict__ stats_a, RowStat *__restrict__ stats_b) {
    const int64_t r = blockIdx.x;
    const int tid = threadIdx.x;
    const int64_t off = rows.off(r);
    const T *arow = A + off, *brow = B + off;
    const JsdRow c = jsd_row_constants(load_rowstat(stats_a + r), load_rowstat(stats_b + r), beta);
    LaneJSD<T> acc;
    acc.init();
    for (int j = tid; j < V; j += kFwdThreads) {
        float a[1] = {Elem<T>::load1(arow + j)}, b[1] = {Elem<T>::load1(brow + j)};
        acc.push(a, b, c);
    }
    __shared__ PartJSD<AccT<T>> parts[kFwdWarps];
    const PartJSD<AccT<T>> w = jsd_warp_merge(acc);
    if ((tid & 31) == 0) parts[tid >> 5] = w;
    __syncthreads();
    if (tid == 0) finish_jsd(parts, kFwdWarps, r, (double)beta, jsd, stats_a, stats_b);
}

// ---------------------------------------------------------------------------
// Launchers (called by the C ABI after argument checks).
// ---------------------------------------------------------------------------
template <typename T>
static cudaError_t launch_kl_t(const KLFwdArgs &a) {
    kl_fwd_kernel<T><<<(unsigned)a.N, kFwdThreads, 0, a.stream>>>(
        static_cast<const T *>(a.p), static_cast<const T *>(a.q), (int)a.V, Rows{a.R, a.s_o, a.s_i}, a.kl,
        static_cast<RowStat *>(a.stats_p), static_cast<RowStat *>(a.stats_q), static_cast<PartialRec *>(a.parts));
    return cudaGetLastError();
}

cudaError_t launch_kl_fwd_rowwise(const KLFwdArgs &a) {
    return a.bf16 ? launch_kl_t<__nv_bfloat16>(a) : launch_kl_t<float>(a);
}

template <typename T>
static cudaError_t launch_jsd_rowwise_t(const JsdFwdArgs &a) {
    jsd_fwd_kernel<T><<<(unsigned)a.N, kFwdThreads, 0, a.stream>>>(
        static_cast<const T *>(a.a), static_cast<const T *>(a.b), (int)a.V, Rows{a.R, a.s_o, a.s_i}, (float)a.beta,
        a.jsd, static_cast<RowStat *>(a.stats_a), static_cast<RowStat *>(a.stats_b));
    return cudaGetLastError();
}

cudaError_t launch_jsd_fwd_rowwise(const JsdFwdArgs &a) {
    return a.bf16 ? launch_jsd_rowwise_t<__nv_bfloat16>(a) : launch_jsd_rowwise_t<float>(a);
}

}  // namespace vp
