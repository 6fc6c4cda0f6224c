// vp_merge.cu -- merge of per-shard records (the vocabulary-sharded forms).
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838): second commit message and the
//        reviewer's "Suggested change" (each rank reduces its shard's max,
//        sum-exp and centred weighted sum; the ranks' values are combined by
//        re-centring on the global max, there with a MAX then a SUM
//        all-reduce), and the Codex thread "Guard zero rescaling before
//        applying infinite shifts" (a shard whose re-centred weight is 0 is
//        skipped, so 0 * inf never enters a sum).
//
// Shape: one warp per row. Lane k reads the records of shards k, k + 32, ...
// (a fixed assignment), the row max is a warp max, the re-centred sums are
// fp64, lane-sequential then a fixed butterfly; a row's result therefore
// depends on its K records only. Lane 0 finishes the row exactly like the
// unsharded forward (fp64 log, the same record layout and special values).
#include "vp_launch.h"
#include "vp_stats.cuh"

namespace vp {

constexpr int kMergeWarps = 8;

__device__ __forceinline__ double nan64() { return __longlong_as_double(0x7ff8000000000000ll); }

template <int kOp>  // 0 = logprobs, 1 = entropy
__global__ void __launch_bounds__(kMergeWarps * 32)
merge_stats_kernel(const PartialRec *__restrict__ parts, int64_t K, int64_t N, float *__restrict__ out,
                   RowStat *__restrict__ stats, int32_t *__restrict__ err) {
    const int64_t r = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= N) return;   // warp-uniform
    float M = kNegBig;
    uint32_t flags = 0;
    int owners = 0;
    float zt = 0.f;
    for (int64_t k = lane; k < K; k += 32) {
        const PartialRec &p = parts[k * N + r];
        M = fmaxf(M, p.m);
        flags |= p.flags;
        if (p.flags & kPartHasTarget) { ++owners; zt = p.z_t; }
    }
    M = warp_max(M);
    flags = __reduce_or_sync(0xffffffffu, flags);
    const unsigned holders = __ballot_sync(0xffffffffu, owners > 0);
    owners = __reduce_add_sync(0xffffffffu, owners);
    zt = __shfl_sync(0xffffffffu, zt, holders ? __ffs(holders) - 1 : 0);

    double S = 0.0, W = 0.0;
    for (int64_t k = lane; k < K; k += 32) {
        const PartialRec &p = parts[k * N + r];
        const double d = (double)M - (double)p.m;   // >= 0
        const double a = exp(-d);
        const double w = a * p.S;
        if (w > 0.0) {                               // zero-weight shards are skipped
            S += w;
            if (kOp == 1) W += a * (p.W - d * p.S);
        }
    }
    S = warp_sum(S);
    if (kOp == 1) W = warp_sum(W);
    if (lane != 0) return;

    uint32_t rf = 0;
    if ((flags & kPartNanInf) || S != S) { S = nan64(); rf |= kRowNanInf; }
    else if (S == 0.0) rf |= kRowEmpty;
    const double logS = log(S);
    const double c = kOp == 1 ? W / S : 0.0;
    const bool bad = rf != 0;
    if (kOp == 1) {
        store_rowstat(stats + r, M, logS, c, rf);
        out[r] = bad ? qnan() : (float)(logS - c);
        return;
    }
    rf |= kRowSharded;
    const bool ignored = (flags & kPartIgnored) != 0;
    const bool bad_target = !ignored && owners != 1;
    if (bad_target) rf |= kRowBadTarget;
    store_rowstat(stats + r, M, logS, c, rf);
    if (ignored) out[r] = 0.f;
    else if (bad_target) {
        out[r] = qnan();
        if (err) atomicOr(err, VP_ERRBIT_TARGET_);
    } else out[r] = bad ? qnan() : (float)(((double)zt - (double)M) - logS);
}

__global__ void __launch_bounds__(kMergeWarps * 32)
merge_kl_kernel(const PartialRec *__restrict__ parts, int64_t K, int64_t N, float *__restrict__ kl,
                RowStat *__restrict__ stats_p, RowStat *__restrict__ stats_q) {
    const int64_t r = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= N) return;
    float Mp = kNegBig, Mq = kNegBig;
    uint32_t flags = 0;
    for (int64_t k = lane; k < K; k += 32) {
        const PartialRec &p = parts[k * N + r];
        Mp = fmaxf(Mp, p.m);
        Mq = fmaxf(Mq, p.m_b);
        flags |= p.flags;
    }
    Mp = warp_max(Mp);
    Mq = warp_max(Mq);
    flags = __reduce_or_sync(0xffffffffu, flags);

    double Sp = 0.0, Sq = 0.0, W = 0.0;
    for (int64_t k = lane; k < K; k += 32) {
        const PartialRec &p = parts[k * N + r];
        const double dp = (double)Mp - (double)p.m, dq = (double)Mq - (double)p.m_b;
        const double ap = exp(-dp), aq = exp(-dq);
        const double wq = aq * p.S_b;
        if (wq > 0.0) Sq += wq;
        const double wp = ap * p.S;
        if (wp > 0.0) {
            Sp += wp;
            W += ap * (p.W - (dp - dq) * p.S);
        }
    }
    Sp = warp_sum(Sp);
    Sq = warp_sum(Sq);
    W = warp_sum(W);
    if (lane != 0) return;
    if (flags & kPartNanInf) Sp = nan64();
    if (flags & kPartNanInfB) Sq = nan64();
    PartKL<double> s;
    s.rp = s.mxp = Mp;
    s.rq = s.mxq = Mq;
    s.Sp = Sp;
    s.Sq = Sq;
    s.W = W;
    s.flag = (flags & kPartMismatch) ? 1 : 0;
    finish_kl(s, r, kl, stats_p, stats_q);
}

static unsigned merge_grid(int64_t N) { return (unsigned)((N + kMergeWarps - 1) / kMergeWarps); }

cudaError_t launch_logprobs_merge(const MergeArgs &a) {
    merge_stats_kernel<0><<<merge_grid(a.N), kMergeWarps * 32, 0, a.stream>>>(
        static_cast<const PartialRec *>(a.parts), a.K, a.N, a.out, static_cast<RowStat *>(a.stats_p), a.err);
    return cudaGetLastError();
}

cudaError_t launch_entropy_merge(const MergeArgs &a) {
    merge_stats_kernel<1><<<merge_grid(a.N), kMergeWarps * 32, 0, a.stream>>>(
        static_cast<const PartialRec *>(a.parts), a.K, a.N, a.out, static_cast<RowStat *>(a.stats_p), nullptr);
    return cudaGetLastError();
}

cudaError_t launch_kl_merge(const MergeArgs &a) {
    merge_kl_kernel<<<merge_grid(a.N), kMergeWarps * 32, 0, a.stream>>>(
        static_cast<const PartialRec *>(a.parts), a.K, a.N, a.out, static_cast<RowStat *>(a.stats_p),
        static_cast<RowStat *>(a.stats_q));
    return cudaGetLastError();
}

}  // namespace vp
