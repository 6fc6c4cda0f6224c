// vp_fwd_tma.cu -- persistent forward kernels fed by a TMA (bulk-copy) ring.
//
// Sources:
//   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
//        (DeepSpeed pull request 8838): second commit message and the
//        reviewer's "Suggested change" (one read of each logit, online (m, S,
//        W), re-centring on the max, the support-mismatch flag); the Codex
//        thread on zero-weight terms.
//   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton", "Implementation".
//
// Shape: a persistent grid of up to two CTAs per SM; CTA b owns rows b, b + G,
// b + 2G, ... Each CTA has eight consumer warps, one producer warp and one
// finisher warp. One
// producer thread walks the CTA's rows and streams each row's 16-byte-aligned
// body through a ring of kStages shared-memory stages (16 KB each) with 1-D
// bulk copies (cp.async.bulk, non-multicast, L2 evict-first), each completing
// on a "full" mbarrier; consumers read the stage with 16-byte shared loads,
// and each warp arrives once on the stage's "empty" mbarrier before folding
// the words into its per-lane statistics (vp_stats.cuh). The producer runs ahead across row boundaries, so
// HBM keeps streaming across rows. At the end of a row each consumer warp
// merges its lanes (double-float sums) and hands its partial to the finisher
// warp through a double-buffered slot (mbarriers, no CTA barrier); the
// finisher merges the 8 partials in a fixed order, so the consumers go
// straight on to the next row, and finishes rows in fp64 in batches of 32,
// one lane per row (fp64 is slow on this part: a lone fp64 log per row costs
// about as much as streaming a short row). The unaligned head and tail of a
// row (< 16 bytes each) are read directly.
// A row's arithmetic depends only on V, the dtype, its address modulo 16 and
// the row-split setting, never on N or on which CTA handles it.
#include "vp_stats.cuh"
#include "vp_tma.cuh"

#include <algorithm>
#include <atomic>

namespace vp {

// Ring geometry (compile-time; the defaults are the measured best on GB300).
#ifndef VP_FWD_STAGE_BYTES
#define VP_FWD_STAGE_BYTES 16384
#endif
#ifndef VP_FWD_STAGES
#define VP_FWD_STAGES 6
#endif
#ifndef VP_FWD_CTAS_PER_SM
#define VP_FWD_CTAS_PER_SM 2
#endif
#ifndef VP_FWD_CONSUMER_WARPS
#define VP_FWD_CONSUMER_WARPS 8
#endif
constexpr int kTmaConsumerWarps = VP_FWD_CONSUMER_WARPS;
constexpr int kTmaConsumers = kTmaConsumerWarps * 32;
constexpr int kProducerWarp = kTmaConsumerWarps;       // warp 8
constexpr int kFinisherWarp = kTmaConsumerWarps + 1;   // warp 9
constexpr int kTmaThreads = kTmaConsumers + 64;
constexpr int kStageBytes = VP_FWD_STAGE_BYTES;
constexpr int kStages = VP_FWD_STAGES;
constexpr int kCtasPerSm = VP_FWD_CTAS_PER_SM;
constexpr int kRingBytes = kStages * kStageBytes;
static_assert(kStageBytes % (2 * 16 * kTmaConsumers) == 0, "a stage splits evenly over the consumers (P and Q halves)");

// Set (OR) when a bounded wait gave up: 1 = producer, 2 = consumer or finisher.
__device__ uint32_t g_tma_fault;

// 16-byte word of -inf values (padding of a partial last stage)
template <typename T>
__device__ __forceinline__ uint4 splat_neg_inf() {
    const uint32_t w = sizeof(T) == 2 ? kBf16NegInf2 : 0xff800000u;
    return make_uint4(w, w, w, w);
}

template <typename T, int K>
__device__ __forceinline__ float chunk_max(const uint4 (&u)[K]) {
    if constexpr (sizeof(T) == 2) {
        return max_bf16(u);
    } else {
        float c = -INFINITY;
#pragma unroll
        for (int k = 0; k < K; ++k)
            c = fmaxf(fmaxf(c, fmaxf(__uint_as_float(u[k].x), __uint_as_float(u[k].y))),
                      fmaxf(__uint_as_float(u[k].z), __uint_as_float(u[k].w)));
        return c;
    }
}

struct Ring {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t parts_full[2];   // the 8 consumer warps have written a row's partials
    uint64_t parts_empty[2];  // the finisher has read them
};

__device__ __forceinline__ void ring_init(Ring &ring) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ring.full[s], 1);
            mbar_init(&ring.empty[s], kTmaConsumerWarps);   // one arrival per consumer warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ring.parts_full[b], kTmaConsumerWarps);
            mbar_init(&ring.parts_empty[b], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
}

// Consumer warp side of the hand-over of a row's partial to the finisher warp
// (slot rowi & 1, reused every second row). Returns false on a timeout.
template <typename P>
__device__ __forceinline__ bool hand_over(Ring &ring, P (*parts)[kTmaConsumerWarps], int rowi, const P &w,
                                          int warp, int lane) {
    bool ok = true;
    if (lane == 0) {
        const int slot = rowi & 1, use = rowi >> 1;
        if (use > 0) ok = mbar_wait(&ring.parts_empty[slot], (use - 1) & 1);
        parts[slot][warp] = w;
        mbar_arrive(&ring.parts_full[slot]);
    }
    return __shfl_sync(0xffffffffu, ok, 0);
}

// A consumer's position in the ring: stage index and the parity of its use.
struct RingPos {
    uint32_t st = 0, ph = 0;
    __device__ __forceinline__ void next() {
        if (++st == (uint32_t)kStages) { st = 0; ph ^= 1u; }
    }
};

// Consumer warp side: the warp's shared loads of stage `st` are done (ordered
// before lane 0's release-arrive by the warp barrier), so the producer may
// refill it.
__device__ __forceinline__ void release_stage(Ring &ring, uint32_t st, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[st]);
}

// Producer side: stage `it`'s slot, waiting for the consumers to free it.
__device__ __forceinline__ bool acquire_stage(Ring &ring, uint32_t it, uint32_t &st) {
    st = it % kStages;
    const uint32_t use = it / kStages;
    return use == 0 || mbar_wait(&ring.empty[st], (use - 1) & 1);
}

// After a failed wait the producer waits (bounded) for its copies in flight
// before the CTA may exit.
__device__ __forceinline__ void drain(Ring &ring, uint32_t issued) {
    atomicOr(&g_tma_fault, 1u);
    for (uint32_t k = issued > (uint32_t)kStages ? issued - kStages : 0; k < issued; ++k)
        mbar_wait(&ring.full[k % kStages], (k / kStages) & 1);
}

// ---------------------------------------------------------------------------
// Vocabulary split across the CTAs of a cluster. With kC > 1 CTAs per cluster,
// the cluster takes rows u, u + U, ... (U clusters) and CTA k of it streams
// segment k of each row's aligned body (seg_range: kC contiguous pieces, 32
// vectors apart, the head with segment 0 and the tail with the last). Every
// CTA merges its 8 warp partials as before; a CTA other than the leader
// (rank 0) sends its segment's partial to the leader's shared memory with
// asynchronous DSMEM stores that complete on the leader's "full" mbarrier (no
// fence on the sender's side); the leader's finisher merges the kC partials in
// rank order (re-centred on the largest centre, as the warp partials) and
// finishes the row, then frees each peer's slot with a remote arrival. The
// split depends on V only, so a row's arithmetic does not depend on N.
// ---------------------------------------------------------------------------
template <int C>
__device__ __forceinline__ void seg_range(int nv, int k, int &lo, int &hi) {
    if constexpr (C == 1) {
        lo = 0;
        hi = nv;
    } else {
        const int step = ((nv + C - 1) / C + 31) & ~31;
        lo = min(nv, k * step);
        hi = min(nv, lo + step);
    }
}

// Slots of the segment partials of two rows in flight (double-buffered, as
// the warp partials) and their barriers: full (in the leader: one arrival, the
// leader's own arming of the phase, plus the bytes of the kC - 1 peers'
// partials) and empty (in each peer: the leader has read its partial).
template <typename P, int kC>
struct alignas(16) ClusterSlots {
    P part[2][kC];                 // 8-byte aligned words (st_async_u64)
    uint64_t full[2], empty[2];
    static constexpr uint32_t kBytes = (kC - 1) * sizeof(P);   // transaction bytes of one phase of full
};

// Before the cluster barrier that publishes the initialisation; the leader
// arms the first phase of both slots (a peer's bytes may land before or after).
template <typename P, int kC>
__device__ __forceinline__ void cluster_slots_init(ClusterSlots<P, kC> &cs, uint32_t rank) {
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&cs.full[b], 1);
            mbar_init(&cs.empty[b], 1);
        }
        fence_mbar_init();
        if (rank == 0)
            for (int b = 0; b < 2; ++b) mbar_arrive_expect_tx(&cs.full[b], ClusterSlots<P, kC>::kBytes);
    }
}

// A peer's side: its segment partial p of the row (slot rowi & 1) into the
// leader's slot, once the leader has read the slot's previous use. Lane 0.
template <typename P, int kC>
__device__ __forceinline__ bool peer_hand_over(ClusterSlots<P, kC> &cs, const P &p, int rowi, uint32_t rank) {
    static_assert(sizeof(P) % 8 == 0, "partials are whole 8-byte words");
    const int slot = rowi & 1, use = rowi >> 1;
    const bool ok = use == 0 || mbar_wait(&cs.empty[slot], (use - 1) & 1);
    uint64_t w[sizeof(P) / 8];
    memcpy(w, &p, sizeof(P));
    const uint32_t dst = cluster_addr(&cs.part[slot][rank], 0), bar = cluster_addr(&cs.full[slot], 0);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(P) / 8); ++i) st_async_u64(dst + 8 * i, w[i], bar);
    return ok;
}

// The leader's side, after merging the slot's partials (whole warp): re-arm
// the slot's next phase and free each peer's slot.
template <typename P, int kC>
__device__ __forceinline__ void leader_release(ClusterSlots<P, kC> &cs, int slot, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(&cs.full[slot], ClusterSlots<P, kC>::kBytes);
    if (lane > 0 && lane < kC) mbar_arrive_cluster_relaxed(cluster_addr(&cs.empty[slot], lane));
}

// ---------------------------------------------------------------------------
// logprobs (kOp = 0), entropy (kOp = 1), logprobs of K ids per row (kOp = 2)
// ---------------------------------------------------------------------------
template <int kOp, typename T, int kC>
__global__ void __launch_bounds__(kTmaThreads, kCtasPerSm)
stats_fwd_tma_kernel(const T *__restrict__ x, int64_t N, int V, Rows rows, const int64_t *__restrict__ targets,
                     int64_t vocab_start, float *__restrict__ out, RowStat *__restrict__ stats,
                     int32_t *__restrict__ err, PartialRec *__restrict__ shard_parts, int64_t K) {
    constexpr bool kW = kOp == 1;
    constexpr int kSt = kOp == 1 ? 1 : 0;                       // statistics of logprobs or entropy
    constexpr int kVec = Elem<T>::kVec;
    constexpr int kChunkVec = kStageBytes / 16;                 // 16-byte vectors per stage
    constexpr int kPerThread = kChunkVec / kTmaConsumers;       // 4
    using P = Part1<AccT<T>>;
    extern __shared__ __align__(128) uint8_t ring_mem[];
    __shared__ Ring ring;
    __shared__ P parts[2][kTmaConsumerWarps];
    __shared__ ClusterSlots<P, kC> cs;
    ring_init(ring);
    const uint32_t rank = kC > 1 ? cluster_rank() : 0u;
    if constexpr (kC > 1) {
        cluster_slots_init(cs, rank);
        cluster_sync();                                         // every CTA's barriers are initialised
    }
    pdl_enter<false>();                                                // no global access before this
    const int64_t unit0 = blockIdx.x / kC, n_units = gridDim.x / kC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kFinisherWarp) {
        // merges the 8 warp partials of each row (segment) in a fixed order; the
        // leader merges the segments. Logprobs and entropy rows are finished in
        // batches of 32 (lane j keeps the batch's j-th merged partial; one fp64
        // pass, 32 lanes wide, per batch), their target ids and target logits
        // read a batch ahead: a lone fp64 log or a dependent load per row would
        // cost more than streaming a short row.
        constexpr bool kBatch = kOp != 2;
        const bool loads = kOp == 0 && rank == 0;
        auto row_of = [&](int i) { return unit0 + (int64_t)i * n_units; };
        auto target_logit = [&](int64_t r, int64_t t) {
            const int64_t loc = t - vocab_start;
            return r < N && t >= 0 && loc >= 0 && loc < V ? Elem<T>::load1(x + rows.off(r) + loc) : 0.f;
        };
        int64_t t_cur = 0, t_nxt = 0;
        float z_cur = 0.f;
        if (loads) {
            const int64_t r0 = row_of(lane), r1 = row_of(32 + lane);
            t_cur = r0 < N ? targets[r0] : -1;
            t_nxt = r1 < N ? targets[r1] : -1;
            z_cur = target_logit(r0, t_cur);
        }
        P keep = empty_part<AccT<T>>();
        int rowi = 0;
        for (int64_t r = unit0; r < N; r += n_units, ++rowi) {
            const int slot = rowi & 1;
            if (!mbar_wait(&ring.parts_full[slot], (rowi >> 1) & 1)) {
                atomicOr(&g_tma_fault, 2u);
                break;
            }
            P p = merge_parts<kW>(parts[slot], kTmaConsumerWarps);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring.parts_empty[slot]);
            if constexpr (kC > 1) {
                if (rank != 0) {
                    if (lane == 0 && !peer_hand_over(cs, p, rowi, rank)) atomicOr(&g_tma_fault, 2u);
                    continue;
                }
                if (!mbar_wait_cluster(&cs.full[slot], (rowi >> 1) & 1)) {
                    atomicOr(&g_tma_fault, 2u);
                    break;
                }
                p = merge_lane_parts<kW>(lane == 0 ? p : lane < kC ? cs.part[slot][lane] : empty_part<AccT<T>>());
                leader_release(cs, slot, lane);
            }
            if constexpr (!kBatch) {
                finish_topk(p, r, V, K, targets, vocab_start, x + rows.off(r), out, stats, err, lane);
            } else {
                const int j = rowi & 31;
                if (lane == j) keep = p;
                if (j == 31 || r + n_units >= N) {   // the batch is complete
                    if (lane <= j) {
                        const int64_t rr = r - (int64_t)(j - lane) * n_units;
                        if (shard_parts) finish_partial<kSt>(keep, rr, V, t_cur, vocab_start, z_cur, shard_parts);
                        else finish_stats<kSt>(keep, rr, V, t_cur, vocab_start, z_cur, out, stats, err);
                    }
                    if (loads) {
                        t_cur = t_nxt;
                        z_cur = target_logit(row_of(rowi + 1 + lane), t_cur);
                        const int64_t rn = row_of(rowi + 33 + lane);
                        t_nxt = rn < N ? targets[rn] : -1;
                    }
                }
            }
        }
    } else if (warp == kProducerWarp) {
        // producer: the whole warp walks the stages (converged, so that no idle
        // lane holds up lane 0 at a barrier); lane 0 issues the copies
        const uint64_t pol = policy_evict_first();
        uint32_t it = 0;
        bool ok = true;
        for (int64_t r = unit0; r < N && ok; r += n_units) {
            const T *row = x + rows.off(r);
            const int head = head_count(row, V);
            const int nv = (V - head) / kVec;
            int lo, hi;
            seg_range<kC>(nv, (int)rank, lo, hi);
            const uint8_t *body = reinterpret_cast<const uint8_t *>(row + head);
            for (int c0 = lo; c0 < hi; c0 += kChunkVec, ++it) {
                uint32_t st;
                if (!__all_sync(0xffffffffu, acquire_stage(ring, it, st))) {
                    if (lane == 0) drain(ring, it);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t bytes = (uint32_t)min(kChunkVec, hi - c0) * 16u;
                    mbar_arrive_expect_tx(&ring.full[st], bytes);
                    bulk_g2s(ring_mem + st * kStageBytes, body + (int64_t)c0 * 16, bytes, &ring.full[st], pol);
                }
                __syncwarp();
            }
        }
    } else {
        // consumers
        const int ct = threadIdx.x;
        RingPos pos;
        bool ok = true;
        int rowi = 0;
        for (int64_t r = unit0; r < N; r += n_units, ++rowi) {
            const T *row = x + rows.off(r);
            const int head = head_count(row, V);
            const int nv = (V - head) / kVec;
            const int tail0 = head + nv * kVec;
            int lo, hi;
            seg_range<kC>(nv, (int)rank, lo, hi);
            Lane1<T, kW> acc;
            acc.init(kNegBig);
            for (int c0 = lo; c0 < hi; c0 += kChunkVec, pos.next()) {
                const uint32_t st = pos.st;
                if (ok && !mbar_wait(&ring.full[st], pos.ph)) {
                    ok = false;
                    atomicOr(&g_tma_fault, 2u);
                }
                const int cnt = min(kChunkVec, hi - c0);
                const uint4 *sv = reinterpret_cast<const uint4 *>(ring_mem + st * kStageBytes);
                const uint4 pad = splat_neg_inf<T>();
                uint4 u[kPerThread];
                if (cnt == kChunkVec) {
#pragma unroll
                    for (int k = 0; k < kPerThread; ++k) u[k] = sv[ct + k * kTmaConsumers];
                } else {
#pragma unroll
                    for (int k = 0; k < kPerThread; ++k) {
                        const int i = ct + k * kTmaConsumers;
                        u[k] = i < cnt ? sv[i] : pad;
                    }
                }
                release_stage(ring, st, lane);                      // the words are in registers
                if (c0 == lo) acc.init(warp_centre(chunk_max<T>(u)));   // the warp's centre for this segment
                if constexpr (Elem<T>::kPrecise) {
                    float v[kPerThread * kVec];
#pragma unroll
                    for (int k = 0; k < kPerThread; ++k) Elem<T>::unpack(u[k], v + k * kVec);
                    acc.push(v);
                } else {
                    acc.push_bf16(u);
                }
            }
            if (rank == 0 && ct < head) { float v[1] = {Elem<T>::load1(row + ct)}; acc.push(v); }
            if (rank == kC - 1 && ct < V - tail0) { float v[1] = {Elem<T>::load1(row + tail0 + ct)}; acc.push(v); }

            P w = warp_merge(acc);
            if (!ok) w.S = AccT<T>(__int_as_float(0x7fc00000));   // a timed-out row finishes as NaN
            if (!hand_over(ring, parts, rowi, w, warp, lane)) {
                atomicOr(&g_tma_fault, 2u);
                break;
            }
        }
    }
    // no DSMEM store or remote arrival may target a CTA that has exited
    __syncwarp();
    if constexpr (kC > 1) cluster_sync();
}

// ---------------------------------------------------------------------------
// KL(P||Q); P and Q share their address modulo 16 (checked by the launcher).
// The vocabulary split across a cluster is that of stats_fwd_tma_kernel.
// ---------------------------------------------------------------------------
template <typename T, int kC, bool kW = true>
__global__ void __launch_bounds__(kTmaThreads, kCtasPerSm)
kl_fwd_tma_kernel(const T *__restrict__ P, const T *__restrict__ Q, int64_t N, int V, Rows rows,
                  float *__restrict__ kl, RowStat *__restrict__ stats_p, RowStat *__restrict__ stats_q,
                  PartialRec *__restrict__ shard_parts) {
    constexpr int kVec = Elem<T>::kVec;
    constexpr int kHalf = kStageBytes / 2;                      // P and Q halves of a stage
    constexpr int kChunkVec = kHalf / 16;                       // 512 vectors of each
    constexpr int kPerThread = kChunkVec / kTmaConsumers;       // 2
    using PK = PartKL<AccT<T>>;
    extern __shared__ __align__(128) uint8_t ring_mem[];
    __shared__ Ring ring;
    __shared__ PK parts[2][kTmaConsumerWarps];
    __shared__ ClusterSlots<PK, kC> cs;
    ring_init(ring);
    const uint32_t rank = kC > 1 ? cluster_rank() : 0u;
    if constexpr (kC > 1) {
        cluster_slots_init(cs, rank);
        cluster_sync();
    }
    pdl_enter<false>();
    const int64_t unit0 = blockIdx.x / kC, n_units = gridDim.x / kC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kFinisherWarp) {
        // rows finished in batches of 32, one lane each (as in stats_fwd_tma_kernel)
        PK keep = empty_kl_part<AccT<T>>();
        int rowi = 0;
        for (int64_t r = unit0; r < N; r += n_units, ++rowi) {
            const int slot = rowi & 1;
            if (!mbar_wait(&ring.parts_full[slot], (rowi >> 1) & 1)) {
                atomicOr(&g_tma_fault, 2u);
                break;
            }
            PK p = kl_merge_parts(parts[slot], kTmaConsumerWarps);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring.parts_empty[slot]);
            if constexpr (kC > 1) {
                if (rank != 0) {
                    if (lane == 0 && !peer_hand_over(cs, p, rowi, rank)) atomicOr(&g_tma_fault, 2u);
                    continue;
                }
                if (!mbar_wait_cluster(&cs.full[slot], (rowi >> 1) & 1)) {
                    atomicOr(&g_tma_fault, 2u);
                    break;
                }
                p = kl_merge_lane_parts(lane == 0 ? p : lane < kC ? cs.part[slot][lane] : empty_kl_part<AccT<T>>());
                leader_release(cs, slot, lane);
            }
            const int j = rowi & 31;
            if (lane == j) keep = p;
            if ((j == 31 || r + n_units >= N) && lane <= j) {
                const int64_t rr = r - (int64_t)(j - lane) * n_units;
                if (shard_parts) finish_partial_kl(keep, rr, shard_parts);
                else finish_kl(keep, rr, kl, stats_p, stats_q);
            }
        }
    } else if (warp == kProducerWarp) {
        // producer: as in stats_fwd_tma_kernel, the warp converged, lane 0 issuing
        const uint64_t pol = policy_evict_first();
        uint32_t it = 0;
        bool ok = true;
        for (int64_t r = unit0; r < N && ok; r += n_units) {
            const int64_t off = rows.off(r);
            const T *prow = P + off, *qrow = Q + off;
            const int head = head_count(prow, V);
            const int nv = (V - head) / kVec;
            int lo, hi;
            seg_range<kC>(nv, (int)rank, lo, hi);
            const uint8_t *pb = reinterpret_cast<const uint8_t *>(prow + head);
            const uint8_t *qb = reinterpret_cast<const uint8_t *>(qrow + head);
            for (int c0 = lo; c0 < hi; c0 += kChunkVec, ++it) {
                uint32_t st;
                if (!__all_sync(0xffffffffu, acquire_stage(ring, it, st))) {
                    if (lane == 0) drain(ring, it);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t bytes = (uint32_t)min(kChunkVec, hi - c0) * 16u;
                    mbar_arrive_expect_tx(&ring.full[st], 2u * bytes);
                    uint8_t *dst = ring_mem + st * kStageBytes;
                    bulk_g2s(dst, pb + (int64_t)c0 * 16, bytes, &ring.full[st], pol);
                    bulk_g2s(dst + kHalf, qb + (int64_t)c0 * 16, bytes, &ring.full[st], pol);
                }
                __syncwarp();
            }
        }
    } else {
        const int ct = threadIdx.x;
        RingPos pos;
        bool ok = true;
        int rowi = 0;
        for (int64_t r = unit0; r < N; r += n_units, ++rowi) {
            const int64_t off = rows.off(r);
            const T *prow = P + off, *qrow = Q + off;
            const int head = head_count(prow, V);
            const int nv = (V - head) / kVec;
            const int tail0 = head + nv * kVec;
            int lo, hi;
            seg_range<kC>(nv, (int)rank, lo, hi);
            LaneKL<T, kW> acc;
            acc.init(kNegBig, kNegBig);
            for (int c0 = lo; c0 < hi; c0 += kChunkVec, pos.next()) {
                const uint32_t st = pos.st;
                if (ok && !mbar_wait(&ring.full[st], pos.ph)) {
                    ok = false;
                    atomicOr(&g_tma_fault, 2u);
                }
                const int cnt = min(kChunkVec, hi - c0);
                const uint4 *sp = reinterpret_cast<const uint4 *>(ring_mem + st * kStageBytes);
                const uint4 *sq = reinterpret_cast<const uint4 *>(ring_mem + st * kStageBytes + kHalf);
                const uint4 pad = splat_neg_inf<T>();
                uint4 up[kPerThread], uq[kPerThread];
                if (cnt == kChunkVec) {
#pragma unroll
                    for (int k = 0; k < kPerThread; ++k) {
                        up[k] = sp[ct + k * kTmaConsumers];
                        uq[k] = sq[ct + k * kTmaConsumers];
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < kPerThread; ++k) {
                        const int i = ct + k * kTmaConsumers;
                        up[k] = i < cnt ? sp[i] : pad;
                        uq[k] = i < cnt ? sq[i] : pad;
                    }
                }
                release_stage(ring, st, lane);
                if (c0 == lo) acc.init(warp_centre(chunk_max<T>(up)), warp_centre(chunk_max<T>(uq)));
                if constexpr (Elem<T>::kPrecise) {
                    float p[kPerThread * kVec], q[kPerThread * kVec];
#pragma unroll
                    for (int k = 0; k < kPerThread; ++k) {
                        Elem<T>::unpack(up[k], p + k * kVec);
                        Elem<T>::unpack(uq[k], q + k * kVec);
                    }
                    acc.push(p, q);
                } else {
                    acc.push_bf16(up, uq);
                }
            }
            if (rank == 0 && ct < head) {
                float p[1] = {Elem<T>::load1(prow + ct)}, q[1] = {Elem<T>::load1(qrow + ct)};
                acc.push(p, q);
            }
            if (rank == kC - 1 && ct < V - tail0) {
                float p[1] = {Elem<T>::load1(prow + tail0 + ct)}, q[1] = {Elem<T>::load1(qrow + tail0 + ct)};
                acc.push(p, q);
            }

            PK w = kl_warp_merge(acc);
            if (!ok) w.Sp = AccT<T>(__int_as_float(0x7fc00000));  // a timed-out row finishes as NaN
            if (!hand_over(ring, parts, rowi, w, warp, lane)) {
                atomicOr(&g_tma_fault, 2u);
                break;
            }
        }
    }
    __syncwarp();
    if constexpr (kC > 1) cluster_sync();
}

// ---------------------------------------------------------------------------
// Generalized JSD, second pass: KL(p || mix) and KL(q || mix) per row from a
// second read of A and B, with the first pass's records (vp_stats.cuh). A and
// B share their address modulo 16 (checked by the launcher).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kTmaThreads, kCtasPerSm)
jsd_fwd_tma_kernel(const T *__restrict__ A, const T *__restrict__ B, int64_t N, int V, Rows rows, float beta,
                   float *__restrict__ jsd, RowStat *__restrict__ stats_a, RowStat *__restrict__ stats_b) {
    constexpr int kVec = Elem<T>::kVec;
    constexpr int kHalf = kStageBytes / 2;                      // A and B halves of a stage
    constexpr int kChunkVec = kHalf / 16;
    constexpr int kPerThread = kChunkVec / kTmaConsumers;
    extern __shared__ __align__(128) uint8_t ring_mem[];
    __shared__ Ring ring;
    __shared__ PartJSD<AccT<T>> parts[2][kTmaConsumerWarps];
    ring_init(ring);
    pdl_enter<false>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kFinisherWarp) {
        int rowi = 0;
        for (int64_t r = blockIdx.x; r < N; r += gridDim.x, ++rowi) {
            const int slot = rowi & 1;
            if (!mbar_wait(&ring.parts_full[slot], (rowi >> 1) & 1)) {
                atomicOr(&g_tma_fault, 2u);
                return;
            }
            __syncwarp();
            if (lane == 0) finish_jsd(parts[slot], kTmaConsumerWarps, r, (double)beta, jsd, stats_a, stats_b);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring.parts_empty[slot]);
        }
        return;
    }
    if (warp == kProducerWarp) {
        if (lane != 0) return;
        const uint64_t pol = policy_evict_first();
        uint32_t it = 0;
        for (int64_t r = blockIdx.x; r < N; r += gridDim.x) {
            const int64_t off = rows.off(r);
            const T *arow = A + off, *brow = B + off;
            const int head = head_count(arow, V);
            const int nv = (V - head) / kVec;
            const uint8_t *ab = reinterpret_cast<const uint8_t *>(arow + head);
            const uint8_t *bb = reinterpret_cast<const uint8_t *>(brow + head);
            for (int c0 = 0; c0 < nv; c0 += kChunkVec, ++it) {
                uint32_t st;
                if (!acquire_stage(ring, it, st)) { drain(ring, it); return; }
                const uint32_t bytes = (uint32_t)min(kChunkVec, nv - c0) * 16u;
                mbar_arrive_expect_tx(&ring.full[st], 2u * bytes);
                uint8_t *dst = ring_mem + st * kStageBytes;
                bulk_g2s(dst, ab + (int64_t)c0 * 16, bytes, &ring.full[st], pol);
                bulk_g2s(dst + kHalf, bb + (int64_t)c0 * 16, bytes, &ring.full[st], pol);
            }
        }
        return;
    }

    const int ct = threadIdx.x;
    RingPos pos;
    bool ok = true;
    int rowi = 0;
    for (int64_t r = blockIdx.x; r < N; r += gridDim.x, ++rowi) {
        const int64_t off = rows.off(r);
        const T *arow = A + off, *brow = B + off;
        const int head = head_count(arow, V);
        const int nv = (V - head) / kVec;
        const int tail0 = head + nv * kVec;
        const JsdRow c = jsd_row_constants(load_rowstat(stats_a + r), load_rowstat(stats_b + r), beta);
        LaneJSD<T> acc;
        acc.init();
        for (int c0 = 0; c0 < nv; c0 += kChunkVec, pos.next()) {
            const uint32_t st = pos.st;
            if (ok && !mbar_wait(&ring.full[st], pos.ph)) {
                ok = false;
                atomicOr(&g_tma_fault, 2u);
            }
            const int cnt = min(kChunkVec, nv - c0);
            const uint4 *sa = reinterpret_cast<const uint4 *>(ring_mem + st * kStageBytes);
            const uint4 *sb = reinterpret_cast<const uint4 *>(ring_mem + st * kStageBytes + kHalf);
            const uint4 pad = splat_neg_inf<T>();
            uint4 ua[kPerThread], ub[kPerThread];
            if (cnt == kChunkVec) {
#pragma unroll
                for (int k = 0; k < kPerThread; ++k) {
                    ua[k] = sa[ct + k * kTmaConsumers];
                    ub[k] = sb[ct + k * kTmaConsumers];
                }
            } else {
#pragma unroll
                for (int k = 0; k < kPerThread; ++k) {
                    const int i = ct + k * kTmaConsumers;
                    ua[k] = i < cnt ? sa[i] : pad;
                    ub[k] = i < cnt ? sb[i] : pad;
                }
            }
            release_stage(ring, st, lane);
            if constexpr (Elem<T>::kPrecise) {
                float a[kPerThread * kVec], b[kPerThread * kVec];
#pragma unroll
                for (int k = 0; k < kPerThread; ++k) {
                    Elem<T>::unpack(ua[k], a + k * kVec);
                    Elem<T>::unpack(ub[k], b + k * kVec);
                }
                acc.push(a, b, c);
            } else {
                acc.push_bf16(ua, ub, c);
            }
        }
        if (ct < head) {
            float a[1] = {Elem<T>::load1(arow + ct)}, b[1] = {Elem<T>::load1(brow + ct)};
            acc.push(a, b, c);
        }
        if (ct < V - tail0) {
            float a[1] = {Elem<T>::load1(arow + tail0 + ct)}, b[1] = {Elem<T>::load1(brow + tail0 + ct)};
            acc.push(a, b, c);
        }
        PartJSD<AccT<T>> w = jsd_warp_merge(acc);
        if (!ok) w.ka = AccT<T>(__int_as_float(0x7fc00000));   // a timed-out row finishes as NaN
        if (!hand_over(ring, parts, rowi, w, warp, lane)) {
            atomicOr(&g_tma_fault, 2u);
            return;
        }
    }
}

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
static int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaGetDevice(&dev);
    int n = (dev >= 0 && dev < 64) ? cached[dev].load() : 0;
    if (n == 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (dev >= 0 && dev < 64) cached[dev].store(n);
    }
    return n > 0 ? n : 1;
}

// The ring is dynamic shared memory above the 48 KB default: raise the limit
// once per kernel and device.
template <typename K>
static cudaError_t allow_ring(K kernel, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load() & bit) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (e == cudaSuccess) done.fetch_or(bit);
    return e;
}

static unsigned persistent_grid(int64_t N) {
    const int64_t g = kCtasPerSm * (int64_t)sm_count();
    return (unsigned)(N < g ? N : g);
}

// CTAs that split one row's vocabulary (a thread-block cluster): the
// process-wide setting (1 by default), applied to rows of 64 KB or more, where
// each segment still spans at least two ring stages. A function of the setting,
// V and the element size only, so that a row's arithmetic is the same at every N.
static std::atomic<int> g_row_split{1};
constexpr int64_t kSplitMinBytes = 65536;

bool set_row_split(int ctas) {
    if (ctas != 1 && ctas != 2) return false;
    g_row_split.store(ctas);
    return true;
}

int row_split() { return g_row_split.load(); }

static int fwd_split(int64_t V, int elem_bytes) {
    return g_row_split.load() == 2 && V * elem_bytes >= kSplitMinBytes ? 2 : 1;
}

// Persistent launch of a forward kernel over N rows in clusters of kC CTAs:
// as many clusters as can be resident at once (cudaOccupancyMaxActiveClusters,
// taken once per device), each looping over its rows.
template <int kC, typename K, typename... Args>
static cudaError_t launch_rows(K kernel, std::atomic<int> (&resident)[64], int64_t N, cudaStream_t stream,
                               Args... args) {
    if constexpr (kC == 1)   // no cluster
        return launch_pdl(kernel, dim3(persistent_grid(N)), dim3(kTmaThreads), kRingBytes, stream, args...);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = kRingBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = VP_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int dev = 0;
    cudaGetDevice(&dev);
    int max_units = (dev >= 0 && dev < 64) ? resident[dev].load() : 0;
    if (max_units <= 0) {
        cfg.gridDim = dim3((unsigned)(kC * kCtasPerSm * sm_count()));
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0)
            n = kCtasPerSm * sm_count() / kC;
        max_units = n;
        if (dev >= 0 && dev < 64) resident[dev].store(n);
    }
    const int64_t units = std::max<int64_t>(1, std::min<int64_t>(N, max_units));
    cfg.gridDim = dim3((unsigned)(units * kC));
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int kOp, typename T, int kC>
static cudaError_t launch_stats_tma_c(const StatsArgs &a) {
    static std::atomic<uint64_t> done{0};
    static std::atomic<int> resident[64];
    auto k = stats_fwd_tma_kernel<kOp, T, kC>;
    cudaError_t e = allow_ring(k, done);
    if (e != cudaSuccess) return e;
    e = launch_rows<kC>(k, resident, a.N, a.stream, static_cast<const T *>(a.x), a.N, (int)a.V, Rows{a.R, a.s_o, a.s_i},
                        a.targets, a.vocab_start, a.out, static_cast<RowStat *>(a.stats), a.err,
                        static_cast<PartialRec *>(a.parts), a.K);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int kOp, typename T>
static cudaError_t launch_stats_tma(const StatsArgs &a) {
    return fwd_split(a.V, sizeof(T)) == 2 ? launch_stats_tma_c<kOp, T, 2>(a) : launch_stats_tma_c<kOp, T, 1>(a);
}

cudaError_t launch_logprobs_fwd(const StatsArgs &a) {
    return a.bf16 ? launch_stats_tma<0, __nv_bfloat16>(a) : launch_stats_tma<0, float>(a);
}

cudaError_t launch_entropy_fwd(const StatsArgs &a) {
    return a.bf16 ? launch_stats_tma<1, __nv_bfloat16>(a) : launch_stats_tma<1, float>(a);
}

cudaError_t launch_logprobs_topk_fwd(const StatsArgs &a) {
    return a.bf16 ? launch_stats_tma<2, __nv_bfloat16>(a) : launch_stats_tma<2, float>(a);
}

template <typename T, int kC, bool kW = true>
static cudaError_t launch_kl_tma_c(const KLFwdArgs &a) {
    static std::atomic<uint64_t> done{0};
    static std::atomic<int> resident[64];
    auto k = kl_fwd_tma_kernel<T, kC, kW>;
    cudaError_t e = allow_ring(k, done);
    if (e != cudaSuccess) return e;
    e = launch_rows<kC>(k, resident, a.N, a.stream, static_cast<const T *>(a.p), static_cast<const T *>(a.q), a.N, (int)a.V,
                        Rows{a.R, a.s_o, a.s_i}, a.kl, static_cast<RowStat *>(a.stats_p),
                        static_cast<RowStat *>(a.stats_q), static_cast<PartialRec *>(a.parts));
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
static cudaError_t launch_kl_tma(const KLFwdArgs &a) {
    return fwd_split(a.V, sizeof(T)) == 2 ? launch_kl_tma_c<T, 2>(a) : launch_kl_tma_c<T, 1>(a);
}

cudaError_t launch_kl_fwd(const KLFwdArgs &a) {
    // the ring copies P and Q rows with one shared 16-byte phase; otherwise the
    // element-wise CTA-per-row kernel reads them
    if ((((uintptr_t)a.p ^ (uintptr_t)a.q) & 15u) != 0) return launch_kl_fwd_rowwise(a);
    return a.bf16 ? launch_kl_tma<__nv_bfloat16>(a) : launch_kl_tma<float>(a);
}

template <typename T>
static cudaError_t launch_jsd_pass2(const JsdFwdArgs &a) {
    static std::atomic<uint64_t> done{0};
    auto k = jsd_fwd_tma_kernel<T>;
    cudaError_t e = allow_ring(k, done);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k, dim3(persistent_grid(a.N)), dim3(kTmaThreads), kRingBytes, a.stream,
                   static_cast<const T *>(a.a), static_cast<const T *>(a.b), a.N, (int)a.V, Rows{a.R, a.s_o, a.s_i},
                   (float)a.beta, a.jsd, static_cast<RowStat *>(a.stats_a), static_cast<RowStat *>(a.stats_b));
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The JSD's first pass on the ring: each row's (m, logS) of A and of B, the
// KL scan without its cross term and mismatch flag (the second pass rewrites
// the records' c fields and keeps only their NaN and empty flags).
template <typename T>
static cudaError_t launch_pair_stats_tma(const KLFwdArgs &a) {
    return fwd_split(a.V, sizeof(T)) == 2 ? launch_kl_tma_c<T, 2, false>(a) : launch_kl_tma_c<T, 1, false>(a);
}

cudaError_t launch_jsd_fwd(const JsdFwdArgs &a) {
    KLFwdArgs k{a.a, a.b, a.bf16, a.N, a.V, a.R, a.s_o, a.s_i, nullptr, a.stats_a, a.stats_b, a.stream};
    if ((((uintptr_t)a.a ^ (uintptr_t)a.b) & 15u) != 0) {   // element-wise kernels for both passes
        cudaError_t e = launch_kl_fwd_rowwise(k);
        return e != cudaSuccess ? e : launch_jsd_fwd_rowwise(a);
    }
    cudaError_t e = a.bf16 ? launch_pair_stats_tma<__nv_bfloat16>(k) : launch_pair_stats_tma<float>(k);
    if (e != cudaSuccess) return e;
    return a.bf16 ? launch_jsd_pass2<__nv_bfloat16>(a) : launch_jsd_pass2<float>(a);
}

cudaError_t read_fault(uint32_t *value, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(value, g_tma_fault, sizeof(uint32_t));
    if (e == cudaSuccess && clear && *value) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_tma_fault, &zero, sizeof(uint32_t));
    }
    return e;
}

}  // namespace vp
