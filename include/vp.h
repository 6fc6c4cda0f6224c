/*
 * vp.h -- C ABI of libvp: vocab-wide logprobs, entropy and KL on one GB300.
 *
 * Sources cited below:
 *   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
 *        (DeepSpeed pull request 8838).
 *   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton" (RL-Kernel pull
 *        request 208).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers.  Every array argument is a DEVICE pointer owned by the caller; the
 *   library never allocates, frees, copies to the host or synchronises. The
 *   arrays must stay alive until the work queued on `stream` has finished.
 *   `stream` is a cudaStream_t (NULL = the legacy default stream); all work is
 *   queued on it in call order and the call returns without waiting.
 *
 * Rows.  An input holds N rows of V logits. Row r (0 <= r < N) starts at
 *   element offset (r / R) * s_o + (r % R) * s_i from the base pointer and its
 *   V logits are consecutive (unit stride) [P1, second commit message: "rows
 *   are addressed with up to two strides, so a slice such as logits[:, :-1]
 *   is read in place"]. Strides and R are counted in elements. A contiguous
 *   [N, V] input is R = N, s_i = V (s_o is then unused). For logits[:, :-1]
 *   of a contiguous [B, T, V] tensor: N = B (T - 1), R = T - 1, s_o = T V,
 *   s_i = V. Inputs that need more than two strides must be copied by the
 *   caller.
 *
 * Dtypes.  VP_F32 or VP_BF16 logits. Arithmetic is fp32 throughout. Per-row
 *   outputs and saved statistics are fp32. Gradients are written contiguous,
 *   [N, V] row-major, in the dtype of the logits, rounded to nearest even
 *   [P1, second commit message: "gradients are returned contiguous"; the
 *   reviewer's note that the bf16 gradient equals the round-to-nearest-even
 *   of the fp32 one].
 *
 * Saved statistics.  Forward calls also write, per row and per input, a
 *   32-byte vp_rowstat record that the matching backward call reads back:
 *   the exact row max m, logS = log sum_j exp(z_j - m) and the centred mean c
 *   (below), the last two as unevaluated sums of two floats (hi + lo) computed
 *   in fp64 at the end of the forward. The sum lse = m + logS is never
 *   formed, so a large common offset does not round away the centred logits
 *   [P1, second commit message: "centring on the max keeps a large common
 *   offset from cancelling in fp32"]. The backward evaluates the gradients
 *   from the centred logits and c, not from the rounded fp32 output, so an
 *   element whose gradient cancels to near zero keeps its accuracy (see
 *   vp_rowstat).
 *
 * Per-row special values (the pages state the cases, not all outcomes; these
 *   are the readings the library implements):
 *   - a NaN or +inf logit in a used row: output NaN, gradient row NaN;
 *   - an all -inf row (the P row for KL): output NaN, gradient row NaN;
 *   - KL(P||Q) with some P_j > -inf where Q_j = -inf ("support mismatch",
 *     decided on the logits, even when p_j underflows) [P1, reviewer's
 *     suggested change]: +inf; the dP row is NaN and dQ = g (q - p) stays
 *     finite;
 *   - terms whose weight is exactly 0 contribute exactly 0, so a one-hot row
 *     spanning +-3e38 gives H = 0 and KL(p||p) = 0 with zero gradients [P1,
 *     Codex thread "Guard zero rescaling before applying infinite shifts"].
 *
 * Targets.  int64 global token ids, one per row (contiguous, length N). The
 *   local column is target - vocab_start. A negative target is ignored: logp
 *   0 and a zero gradient row. A target >= 0 outside [vocab_start,
 *   vocab_start + V) is a data error: that row's output (and gradient row) is
 *   NaN and bit VP_ERRBIT_TARGET is OR-ed into *err_word (a device int32,
 *   may be NULL) with an atomic; nothing is reported on the host.
 *
 * Batch invariance.  The launch shape depends on V and the dtype only, so each
 *   row's outputs and gradients are bitwise identical for any N and any other
 *   rows in the batch [P1, maintainer's remark on batch invariance for RL
 *   rollouts].
 *
 * Errors.  Every call returns a vp_status. Argument errors are found on the
 *   host before anything is queued and leave the outputs untouched. N = 0 is
 *   valid and queues nothing.
 */
#ifndef VP_H
#define VP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define VP_API __attribute__((visibility("default")))
#else
#define VP_API
#endif

struct CUstream_st;
typedef struct CUstream_st *vp_stream; /* identical to cudaStream_t */

typedef enum vp_status {
    VP_OK = 0,
    VP_ERR_NULL = 1,      /* a required pointer is NULL                              */
    VP_ERR_SHAPE = 2,     /* N < 0, V < 1, V > 2^31 - 1, R < 1, D < 1, ...              */
    VP_ERR_DTYPE = 3,     /* unknown dtype code                                      */
    VP_ERR_LAYOUT = 4,    /* a negative stride                                       */
    VP_ERR_ALIGN = 5,     /* a pointer not aligned to its element size (16 B for
                             vp_rowstat arrays)                                      */
    VP_ERR_LAUNCH = 6,    /* the CUDA launch failed                                  */
    VP_ERR_ARG = 7,       /* another invalid argument (direction, both gradients
                             requested as NULL where one is required, ...)          */
    VP_ERR_DEVICE = 8,    /* no usable device, or not an sm_103 device               */
    VP_ERR_SCRATCH = 9    /* too large for the fixed scratch of
                             vp_linear_logp_fwd_noalloc                             */
} vp_status;

typedef enum vp_dtype { VP_F32 = 0, VP_BF16 = 1 } vp_dtype;

/* KL direction [P1: "reverse KL" / "forward KL"; the pages do not define them.
 * Reading: A is the first argument (student / policy), reverse = KL(A||B),
 * forward = KL(B||A).] */
typedef enum vp_kl_direction { VP_KL_REVERSE = 0, VP_KL_FORWARD = 1 } vp_kl_direction;

#define VP_ERRBIT_TARGET 1

/* Row flags of vp_rowstat. */
#define VP_ROW_NANINF   1u  /* the row holds a NaN or a +inf                          */
#define VP_ROW_EMPTY    2u  /* no finite logit (all -inf): S = 0                      */
#define VP_ROW_MISMATCH 4u  /* KL(P||Q) record of P: some P_j > -inf has Q_j = -inf  */
#define VP_ROW_SHARDED  8u  /* written by vp_logprobs_merge: the target was checked
                               across all shards (see the sharded forms below)   */
#define VP_ROW_BADTARGET 16u /* written by vp_logprobs_merge: no shard, or more
                               than one, holds the row's target >= 0           */

/* Per-row statistics saved by a forward call for its backward call.
 * m      the exact row max; -FLT_MAX when the row has no finite logit.
 * logS   log sum_j exp(z_j - m) = logS_hi + logS_lo.
 * c      the probability-weighted mean of the centred logits, c_hi + c_lo:
 *          entropy:            c = E_p[z - m] = W / S, so H = logS - c;
 *          KL(P||Q), P record: c = E_p[(P - m_P) - (Q - m_Q)] = W / S_P,
 *                              so KL = c - logS_P + logS_Q;
 *          logprobs, and the Q record of KL: 0.
 *        Gradients use it as dH/dz_j = -p_j ((z_j - m) - c) and
 *        dKL/dP_j = p_j (((P_j - m_P) - (Q_j - m_Q)) - c).
 * flags  VP_ROW_* bits. */
typedef struct vp_rowstat {
    float m;
    float logS_hi, logS_lo;
    float c_hi, c_lo;
    uint32_t flags;
    uint32_t reserved[2];
} vp_rowstat;

/* ------------------------------------------------------------------------ */
/* Logprobs [P1, first commit message; P2, "Implementation"]                 */
/* ------------------------------------------------------------------------ */

/* logp[r] = (z_{r,t} - m_r) - logS_r for t = targets[r] - vocab_start, read in
 * one pass over each row. Outputs: logp (fp32 [N]) and stats (vp_rowstat [N],
 * 16-byte aligned), both required. err_word may be NULL. */
VP_API vp_status vp_logprobs_fwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R,
                                 int64_t s_o, int64_t s_i, int64_t vocab_start,
                                 const int64_t *targets, float *logp, vp_rowstat *stats,
                                 int32_t *err_word, vp_stream stream);

/* dx[r, j] = g[r] (onehot_{j,t} - p_{r,j}), p = exp((z - m) - logS), using
 * the stats of vp_logprobs_fwd [P2, review nitpick on the chunked backward].
 * grad_out: fp32 [N]. dx: contiguous [N, V], dtype of x. With the records of
 * vp_logprobs_merge (VP_ROW_SHARDED), x is one vocabulary shard starting at
 * vocab_start: a target outside it only drops the onehot term. */
VP_API vp_status vp_logprobs_bwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R,
                                 int64_t s_o, int64_t s_i, int64_t vocab_start,
                                 const int64_t *targets, const vp_rowstat *stats,
                                 const float *grad_out, void *dx, int32_t *err_word,
                                 vp_stream stream);

/* Several target ids per row (top-k) [P1, PR description, "Tests": duplicate
 * and ignored top-k ids and a fully ignored row]. targets: int64 [N, K]
 * row-major (global ids, each following the rules of vp_logprobs_fwd: a
 * negative id is ignored and gives 0, an id >= 0 outside the shard gives NaN
 * and VP_ERRBIT_TARGET). Outputs: logp fp32 [N, K] and stats (vp_rowstat [N],
 * the same record as vp_logprobs_fwd). K >= 1. */
VP_API vp_status vp_logprobs_topk_fwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                                      int64_t s_i, int64_t vocab_start, const int64_t *targets, int64_t K,
                                      float *logp, vp_rowstat *stats, int32_t *err_word, vp_stream stream);

/* Gradient of sum_k g[r, k] logp[r, k]: dx[r, j] = G_j - p_j Gsum, with Gsum
 * the sum of g over the row's ids that are not ignored and G_j the sum over
 * the ids equal to j (duplicate ids add up). grad_out: fp32 [N, K]. A row with
 * an id outside the shard (or without valid statistics) is NaN; a row whose
 * ids are all ignored is 0. dx: contiguous [N, V], dtype of x. */
VP_API vp_status vp_logprobs_topk_bwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                                      int64_t s_i, int64_t vocab_start, const int64_t *targets, int64_t K,
                                      const vp_rowstat *stats, const float *grad_out, void *dx, int32_t *err_word,
                                      vp_stream stream);

/* ------------------------------------------------------------------------ */
/* Entropy [P1, second commit message and reviewer's suggested change]      */
/* ------------------------------------------------------------------------ */

/* H[r] = log S - W / S from one read of the row, with the online max m,
 * S = sum e^{z-m} and W = sum e^{z-m} (z - m). Outputs: H (fp32 [N]) and
 * stats (vp_rowstat [N]). */
VP_API vp_status vp_entropy_fwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R,
                                int64_t s_o, int64_t s_i, float *H, vp_rowstat *stats,
                                vp_stream stream);

/* dx[r, j] = -g[r] p_j (log p_j + H_r) = -g[r] p_j ((z_j - m) - c), exactly 0
 * where p_j = 0. */
VP_API vp_status vp_entropy_bwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R,
                                int64_t s_o, int64_t s_i, const vp_rowstat *stats,
                                const float *grad_out, void *dx, vp_stream stream);

/* ------------------------------------------------------------------------ */
/* KL [P1, second commit message and reviewer's suggested change]           */
/* ------------------------------------------------------------------------ */

/* One read of A and B. With (P, Q) = (A, B) for VP_KL_REVERSE and (B, A) for
 * VP_KL_FORWARD: KL = W / S_P - log S_P + log S_Q, where
 * W = sum_j e^{P_j - m_P} ((P_j - m_P) - (Q_j - m_Q)), or +inf on a support
 * mismatch. A and B share one row layout (R, s_o, s_i) and dtype.
 * Outputs: kl (fp32 [N]) and the records of A and of B (vp_rowstat [N] each;
 * the record of P carries c), all required. */
VP_API vp_status vp_kl_fwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R,
                           int64_t s_o, int64_t s_i, int direction, float *kl, vp_rowstat *stats_a,
                           vp_rowstat *stats_b, vp_stream stream);

/* dP_j = g p_j (log p_j - log q_j - KL), dQ_j = g (q_j - p_j), mapped back to
 * A and B by the direction, which must be the one given to vp_kl_fwd. da and
 * db are contiguous [N, V] in the dtype of the inputs; either may be NULL
 * (that gradient is then neither computed nor written), not both. */
VP_API vp_status vp_kl_bwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R,
                           int64_t s_o, int64_t s_i, int direction, const vp_rowstat *stats_a,
                           const vp_rowstat *stats_b, const float *grad_out, void *da, void *db,
                           vp_stream stream);

/* ------------------------------------------------------------------------ */
/* Generalized Jensen-Shannon divergence [P1, the commit message that adds   */
/* vocab_parallel_jsd: "Changes", "Scope and limitations"]                   */
/* ------------------------------------------------------------------------ */

/* With p = softmax of a row of A (the student, first argument), q = softmax
 * of the row of B (the teacher) and mix = beta q + (1 - beta) p:
 *   0 < beta < 1:  JSD = beta KL(q || mix) + (1 - beta) KL(p || mix)
 *                  (the page names a GKD-style interior divergence of two
 *                  KL-to-mixture expectations; this formula is the reading
 *                  taken where it prints none);
 *   beta = 0:      KL(B || A), the same call as vp_kl_fwd with VP_KL_FORWARD;
 *   beta = 1:      KL(A || B), the same call as vp_kl_fwd with VP_KL_REVERSE
 *                  (explicit endpoint branches, as on the page).
 * Interior beta reads A and B twice: the first pass takes each row's (m,
 * logS) of A and of B, the second reduces the two KL-to-mixture expectations
 * together. beta is used in fp32. Outputs: jsd fp32 [N] and the records of A
 * and of B (vp_rowstat [N] each, required); for interior beta their c fields
 * hold KL(p || mix) and KL(q || mix). A row with a NaN or +inf, or without a
 * finite logit, in A or B gives NaN; otherwise the interior divergence is
 * finite (there is no support mismatch). beta outside [0, 1] or NaN:
 * VP_ERR_ARG. A and B share one row layout and dtype. */
VP_API vp_status vp_jsd_fwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                            int64_t s_i, double beta, float *jsd, vp_rowstat *stats_a, vp_rowstat *stats_b,
                            vp_stream stream);

/* Gradients for interior beta, from the records of vp_jsd_fwd with the same beta:
 *   dA_j = g (1 - beta) p_j ((log p_j - log mix_j) - KL(p || mix)),
 *   dB_j = g beta q_j ((log q_j - log mix_j) - KL(q || mix)),
 * exactly 0 where p_j = 0 (q_j = 0); at beta = 0 and 1, vp_kl_bwd with the
 * matching direction. da and db are contiguous [N, V] in the inputs' dtype;
 * either may be NULL (a frozen teacher or student), not both. */
VP_API vp_status vp_jsd_bwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                            int64_t s_i, double beta, const vp_rowstat *stats_a, const vp_rowstat *stats_b,
                            const float *grad_out, void *da, void *db, vp_stream stream);

/* ------------------------------------------------------------------------ */
/* Vocabulary-sharded (tensor-parallel) forms [P1, second commit message and */
/* the reviewer's suggested change: each rank reduces its own shard's max,   */
/* sum-exp and centred weighted sum, and the shards are combined by          */
/* re-centring on the row max; the pages do this with a MAX then a SUM       */
/* all-reduce]. Here one gather of fixed-size records replaces both.         */
/*                                                                           */
/* Flow for K shards of the vocabulary, shard k holding columns              */
/* [vocab_start_k, vocab_start_k + V_k) of every row (typically one shard    */
/* per GPU):                                                                 */
/*  1. each shard calls vp_*_partial on its logits: one vp_partial per row;  */
/*  2. the caller gathers the K arrays into one array of K * N records,      */
/*     shard-major (row r of shard k at index k * N + r), e.g. with an       */
/*     all-gather; the library itself makes no collective call;              */
/*  3. vp_*_merge turns the gathered records into the outputs and vp_rowstat */
/*     records that the unsharded forward would write for the whole rows;    */
/*  4. each shard calls the ordinary backward (vp_logprobs_bwd with its own  */
/*     vocab_start, vp_entropy_bwd, vp_kl_bwd) on its own logits with the    */
/*     merged records and gets its columns of the gradient.                  */
/* The merge reads a row's K records in shard order, so its result does not  */
/* depend on N or on the other rows.                                         */
/* ------------------------------------------------------------------------ */

/* Flags of vp_partial. */
#define VP_PART_NANINF     1u  /* A (P for KL) holds a NaN or +inf in this shard   */
#define VP_PART_NANINF_B   2u  /* KL: Q holds a NaN or +inf in this shard          */
#define VP_PART_MISMATCH   4u  /* KL: some P_j > -inf has Q_j = -inf in the shard  */
#define VP_PART_HAS_TARGET 8u  /* logprobs: the row's target lies in this shard    */
#define VP_PART_IGNORED   16u  /* logprobs: the row's target is negative (ignored) */

/* One row's statistics over one shard; 40 bytes, 8-byte aligned.
 * m     the exact max over the shard of A (of P for KL); -FLT_MAX when the
 *       shard has no finite logit (S is then 0).
 * S     sum over the shard of exp(z_j - m), fp64.
 * W     entropy: sum over the shard of exp(z_j - m) (z_j - m);
 *       KL(P||Q): sum of exp(P_j - m) ((P_j - m) - (Q_j - m_b)) over the terms
 *       with exp(P_j - m) > 0, meaningful only when no flag is set;
 *       logprobs: 0.
 * m_b, S_b  KL only: the max and sum-exp of Q over the shard (else 0).
 * z_t   logprobs only: the target's logit when VP_PART_HAS_TARGET (else 0).
 * flags VP_PART_* bits. */
typedef struct vp_partial {
    float m, m_b;
    double S, S_b, W;
    float z_t;
    uint32_t flags;
} vp_partial;

/* Partial records of logprobs over the shard held by x (V columns starting
 * at global id vocab_start). targets are global ids: one inside the shard
 * sets VP_PART_HAS_TARGET and z_t, a negative one VP_PART_IGNORED, one in
 * another shard neither (not an error here). parts: vp_partial [N], 8-byte
 * aligned. */
VP_API vp_status vp_logprobs_partial(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                                     int64_t s_i, int64_t vocab_start, const int64_t *targets,
                                     vp_partial *parts, vp_stream stream);

/* Partial records of entropy over the shard held by x. */
VP_API vp_status vp_entropy_partial(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                                    int64_t s_i, vp_partial *parts, vp_stream stream);

/* Partial records of KL(P||Q) over the shard held by a and b, with (P, Q) =
 * (A, B) for VP_KL_REVERSE and (B, A) for VP_KL_FORWARD. */
VP_API vp_status vp_kl_partial(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R,
                               int64_t s_o, int64_t s_i, int direction, vp_partial *parts, vp_stream stream);

/* Merges K >= 1 shards' records (K * N, shard-major) into logp (fp32 [N]) and
 * stats (vp_rowstat [N]) as vp_logprobs_fwd would write them for the whole
 * rows. A row whose target is ignored gets logp 0. A row whose target is
 * >= 0 but held by no shard or by several is a data error: logp NaN,
 * VP_ERRBIT_TARGET in *err_word (may be NULL) and VP_ROW_BADTARGET in its
 * record. Every record gets VP_ROW_SHARDED, which tells vp_logprobs_bwd that a
 * target outside the calling shard is valid (its onehot term lies in another
 * shard) and that VP_ROW_BADTARGET rows have NaN gradient rows. */
VP_API vp_status vp_logprobs_merge(const vp_partial *parts, int64_t K, int64_t N, float *logp,
                                   vp_rowstat *stats, int32_t *err_word, vp_stream stream);

/* Merges K shards' entropy records into H (fp32 [N]) and stats, as
 * vp_entropy_fwd would write them for the whole rows. */
VP_API vp_status vp_entropy_merge(const vp_partial *parts, int64_t K, int64_t N, float *H, vp_rowstat *stats,
                                  vp_stream stream);

/* Merges K shards' KL records into kl (fp32 [N]) and the records of A and of
 * B, as vp_kl_fwd would write them; direction must be the one given to
 * vp_kl_partial. */
VP_API vp_status vp_kl_merge(const vp_partial *parts, int64_t K, int64_t N, int direction, float *kl,
                             vp_rowstat *stats_a, vp_rowstat *stats_b, vp_stream stream);

/* ------------------------------------------------------------------------ */
/* Fused linear logp [P2, "Implementation"]                                  */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace vp_linear_logp_fwd needs for N rows and V
 * vocabulary rows (per-row, per-256-column (max, sum-exp) pairs and the target
 * logits). 0 for invalid sizes. */
VP_API size_t vp_linear_logp_workspace_size(int64_t N, int64_t V, int64_t D);

/* logp[r] = h_r . w_t - log sum_j exp(h_r . w_j), t = targets[r] - vocab_start,
 * over the V rows of W (a vocabulary shard starting at global id vocab_start),
 * without materialising the logits: tcgen05 tensor-core tiles (bf16 inputs,
 * fp32 accumulation in TMEM) with an online log-sum-exp epilogue, then an fp64
 * merge per row [P2, "Implementation": the forward returns (logp, lse)].
 * hidden: bf16 [N, D] row-major; weight: bf16 [V, D] row-major; both 16-byte
 * aligned; D a multiple of 64. targets: int64 [N] (negative = ignored, out of
 * the shard = data error, as for vp_logprobs_fwd). Outputs: logp fp32 [N] and
 * stats (vp_rowstat [N]: m = max logit, logS, c = 0) for the backward.
 * workspace: device memory of at least vp_linear_logp_workspace_size(N, V, D)
 * bytes, 256-byte aligned, owned by the caller; its contents are scratch.
 * Logits are rounded nowhere: each is an fp32 accumulation of bf16 products. */
VP_API vp_status vp_linear_logp_fwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                    int64_t vocab_start, const int64_t *targets, float *logp, vp_rowstat *stats,
                                    void *workspace, size_t workspace_bytes, int32_t *err_word, vp_stream stream);

/* Precision of the fused linear backwards (the `precision` argument of
 * vp_linear_logp_bwd, vp_linear_entropy_bwd, vp_linear_kl_bwd and
 * vp_linear_jsd_bwd). dz = dL/dlogits is formed in fp32 in the epilogue of
 * the recomputed logits tile, and the two gradient GEMMs (dhidden = dz . W,
 * dW = dz^T . h) run on bf16 tensor cores:
 *   VP_GRAD_EXACT  dz is carried as the pair dz_hi = bf16(dz), dz_lo =
 *                  bf16(dz - dz_hi) (about 16 significant bits), and each
 *                  gradient GEMM adds the dz_lo product into the same fp32
 *                  accumulator: the gradients then carry only the fp32
 *                  accumulation error, and the two gradient GEMMs cost twice
 *                  the work (10 N V D flops for the whole backward instead of
 *                  6 N V D);
 *   VP_GRAD_FAST   dz is rounded to bf16 once (relative error up to 2^-9 per
 *                  term of the dot products). */
#define VP_GRAD_EXACT 0
#define VP_GRAD_FAST  1

/* Bytes of device workspace vp_linear_logp_bwd needs (for either precision):
 * dz of one vocabulary chunk twice over (bf16 [N, vc] for dz_hi and for dz_lo;
 * vc = 32768 columns for N <= 8192, 16384 for N <= 16384, else 8192, at most V
 * rounded up to 256) and an fp32 accumulator of dhidden ([N, D]). 0 for
 * invalid sizes. */
VP_API size_t vp_linear_logp_bwd_workspace_size(int64_t N, int64_t V, int64_t D);

/* Gradients of sum_r g[r] logp[r] for the forward above [P2, review nitpick on
 * the chunked backward: dz = g (onehot - exp(logits - lse)), dhidden = dz . W,
 * dW = dz^T . h]. The logits are recomputed chunk by chunk (vc vocabulary
 * rows of W at a time, see above) on tcgen05 tensor cores; dz of a chunk goes
 * to the two gradient GEMMs (fp32 accumulation in TMEM) as a bf16 pair or
 * rounded once, by `precision` (VP_GRAD_EXACT or VP_GRAD_FAST, above; any other
 * value is VP_ERR_ARG); the GEMMs read dz, W and h in place (transposed
 * operands as MN-major tiles); dhidden accumulates across chunks in fp32 and
 * is rounded to bf16 at the end; dW is written chunk by chunk. dhidden: bf16 [N, D]; dW: bf16 [V, D]; either may
 * be NULL (not both). stats: the records written by vp_linear_logp_fwd, or by
 * vp_logprobs_merge for a vocabulary shard (see the sharded fused linear ops
 * below: a target outside the shard is then held by another shard).
 * Rows with an ignored target contribute nothing; rows with a data error or
 * without valid statistics make their dhidden row and all of dW NaN. */
VP_API vp_status vp_linear_logp_bwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                    int64_t vocab_start, const int64_t *targets, const vp_rowstat *stats,
                                    const float *grad_out, void *dhidden, void *dW, int precision, void *workspace,
                                    size_t workspace_bytes, int32_t *err_word, vp_stream stream);

/* The paper has no counterpart of this entry point; it exists for callers that
 * cannot allocate device memory themselves.
 *
 * Same result as vp_linear_logp_fwd (the same kernels, bitwise), but the
 * scratch lives in one fixed 24 MiB array inside the library instead of a
 * workspace passed by the caller, so the call allocates nothing. It serves
 * callers that must not call cudaMalloc or any allocating routine of their own:
 * for instance a plugin running inside a host framework that owns all device
 * memory through its own allocator, or a service that fixes its memory
 * footprint at start-up and forbids later allocations (which could fail or
 * fragment memory in the middle of a run). The caller still passes every input
 * and output.
 *
 * Limits and behaviour:
 *  - the array is 24 MiB; every GPU that loads the library holds it until the
 *    process exits;
 *  - the scratch needed is about 8 bytes per row and 256-column vocabulary
 *    tile plus 4 bytes per row (vp_linear_logp_workspace_size(N, V, D));
 *    problems needing more than 24 MiB return VP_ERR_SCRATCH before any work
 *    is queued (e.g. V = 75968 allows up to about 10,500 rows);
 *  - the first call on each device looks up the array's device address once
 *    (cudaGetSymbolAddress, with that device current) and caches it with the
 *    context it belongs to; a call from another context on that device (for
 *    instance after cudaDeviceReset) looks it up again. Make the first call
 *    on each device, and in each new context, before any stream capture;
 *  - all calls share the one array and it keeps the last call's contents;
 *    nothing in it needs clearing (every entry is written before it is read
 *    within a call), but calls that overlap on the GPU (concurrent streams)
 *    race on it and must be serialised by the caller. */
VP_API vp_status vp_linear_logp_fwd_noalloc(const void *hidden, const void *weight, int64_t N, int64_t V,
                                            int64_t D, int64_t vocab_start, const int64_t *targets, float *logp,
                                            vp_rowstat *stats, int32_t *err_word, vp_stream stream);

/* ------------------------------------------------------------------------ */
/* Fused linear entropy and KL [P1, the commit message adding               */
/* vocab_parallel_jsd, "Motivation": teacher-student divergences computed    */
/* from tiled LM-head projections without the full logits; P2,              */
/* "Implementation" and the review nitpick on the chunked backward]          */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace vp_linear_entropy_fwd needs: a 16-byte record per
 * row and 256-column vocabulary tile. 0 for invalid sizes. */
VP_API size_t vp_linear_entropy_workspace_size(int64_t N, int64_t V, int64_t D);

/* H[r] = entropy of softmax(h_r . W^T) over the V rows of W, without
 * materialising the logits: tcgen05 tiles (bf16 inputs, fp32 accumulation in
 * TMEM) whose epilogue takes, per row and tile, the max m, S = sum e^{z-m} and
 * W = sum e^{z-m} (z-m); a merge per row re-centres the tiles on the row max
 * and writes H = log S - W / S [P1, second commit message]. hidden: bf16
 * [N, D]; weight: bf16 [V, D]; row-major, 16-byte aligned, D a multiple of 64.
 * Outputs: H fp32 [N] and stats (vp_rowstat [N]: m = max logit, logS,
 * c = W / S) for the backward. workspace: at least
 * vp_linear_entropy_workspace_size(N, V, D) bytes, 256-byte aligned, caller
 * owned, scratch. A row whose logits hold NaN or +inf gives NaN. */
VP_API vp_status vp_linear_entropy_fwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                       float *H, vp_rowstat *stats, void *workspace, size_t workspace_bytes,
                                       vp_stream stream);

/* Bytes of device workspace vp_linear_entropy_bwd needs (for either
 * precision): dz of one vocabulary chunk twice over (bf16 [N, vc] each, vc as
 * for vp_linear_logp_bwd_workspace_size) and an fp32 accumulator of dhidden
 * ([N, D]). 0 for invalid sizes. */
VP_API size_t vp_linear_entropy_bwd_workspace_size(int64_t N, int64_t V, int64_t D);

/* Gradients of sum_r g[r] H[r]: per vocabulary chunk the logits tile is
 * recomputed and dz = -g p (log p + H) = -g p ((z - m) - c) formed in the
 * epilogue, then dhidden += dz . W_c and dW_c = dz^T . h (as
 * vp_linear_logp_bwd, with the same `precision`). dhidden: bf16 [N, D]; dW: bf16 [V, D]; either may
 * be NULL (not both). stats: the records of vp_linear_entropy_fwd. Rows
 * without valid statistics make their dhidden row and all of dW NaN. */
VP_API vp_status vp_linear_entropy_bwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                       const vp_rowstat *stats, const float *grad_out, void *dhidden, void *dW,
                                       int precision, void *workspace, size_t workspace_bytes, vp_stream stream);

/* Bytes of device workspace vp_linear_kl_fwd needs: a 32-byte record per row
 * and 128 columns of the vocabulary. 0 for invalid sizes. */
VP_API size_t vp_linear_kl_workspace_size(int64_t N, int64_t V);

/* KL between the next-token distributions of two models over the same V
 * vocabulary rows: model A (hidden ha bf16 [N, Da], head wa bf16 [V, Da]) and
 * model B (hb bf16 [N, Db], wb bf16 [V, Db]); each model has its own hidden
 * size (Da, Db multiples of 64). direction VP_KL_REVERSE gives KL(A||B),
 * VP_KL_FORWARD gives KL(B||A), as vp_kl_fwd. One dual tcgen05 GEMM puts the
 * same logits tile of both models in TMEM; the epilogue takes each tile's
 * maxima, sum-exps and W = sum e^{P-m_P} ((P - m_P) - (Q - m_Q)), and a merge
 * per row re-centres the tiles and writes KL = W / S_P - log S_P + log S_Q.
 * Outputs: kl fp32 [N]; stats_a, stats_b (vp_rowstat [N] each, the records of
 * vp_kl_fwd). workspace: at least vp_linear_kl_workspace_size(N, V) bytes,
 * 256-byte aligned. A row whose logits hold NaN or +inf gives NaN. */
VP_API vp_status vp_linear_kl_fwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N,
                                  int64_t V, int64_t Da, int64_t Db, int direction, float *kl, vp_rowstat *stats_a,
                                  vp_rowstat *stats_b, void *workspace, size_t workspace_bytes, vp_stream stream);

/* Bytes of device workspace vp_linear_kl_bwd needs (for either precision): dz
 * of one vocabulary chunk for each model (dz_hi and dz_lo, bf16 [N, vc] each)
 * and fp32 accumulators of both dhidden ([N, Da] and [N, Db]). 0 for invalid
 * sizes. */
VP_API size_t vp_linear_kl_bwd_workspace_size(int64_t N, int64_t V, int64_t Da, int64_t Db);

/* Gradients of sum_r g[r] KL[r] with respect to both models' hidden states
 * and heads: per vocabulary chunk the dual GEMM recomputes both logits tiles,
 * the epilogue forms dP = g p ((P - m_P) - (Q - m_Q) - c) and dQ = g (q - p),
 * and the gradient GEMMs of each model follow (`precision` as for
 * vp_linear_logp_bwd). dha bf16
 * [N, Da], dwa bf16 [V, Da], dhb bf16 [N, Db], dwb bf16 [V, Db]: any may be
 * NULL (not all); a model with neither output (a frozen teacher) costs no
 * gradient GEMMs. stats_a, stats_b: the records of vp_linear_kl_fwd with the
 * same direction. NaN rows give NaN dhidden rows and NaN heads' gradients. */
VP_API vp_status vp_linear_kl_bwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N,
                                  int64_t V, int64_t Da, int64_t Db, int direction, const vp_rowstat *stats_a,
                                  const vp_rowstat *stats_b, const float *grad_out, void *dha, void *dwa, void *dhb,
                                  void *dwb, int precision, void *workspace, size_t workspace_bytes,
                                  vp_stream stream);

/* Generalized JSD between two models' next-token distributions [P1, the
 * commit message adding vocab_parallel_jsd: "Motivation" (divergences over
 * tiled LM-head projections without the full logits) and "Changes"], with the
 * JSD of vp_jsd_fwd: p = softmax(ha . wa^T) (A, the student), q =
 * softmax(hb . wb^T) (B, the teacher), mix = beta q + (1 - beta) p,
 * JSD = beta KL(q || mix) + (1 - beta) KL(p || mix). Models and layouts as
 * vp_linear_kl_fwd. beta = 0 and beta = 1 are vp_linear_kl_fwd with
 * VP_KL_FORWARD and VP_KL_REVERSE; 0 < beta < 1 takes two passes: one GEMM
 * per model for the rows' maxima and log-sums of A and B, then the dual GEMM
 * for both KL-to-mixture expectations together. Outputs: jsd fp32 [N]; stats_a, stats_b
 * (vp_rowstat [N], the c fields holding KL(p || mix) and KL(q || mix)).
 * workspace: vp_linear_jsd_workspace_size(N, V) bytes. beta outside [0, 1]
 * or NaN: VP_ERR_ARG. */
VP_API size_t vp_linear_jsd_workspace_size(int64_t N, int64_t V);
VP_API vp_status vp_linear_jsd_fwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N,
                                   int64_t V, int64_t Da, int64_t Db, double beta, float *jsd,
                                   vp_rowstat *stats_a, vp_rowstat *stats_b, void *workspace, size_t workspace_bytes,
                                   vp_stream stream);

/* Gradients of sum_r g[r] JSD[r] from the records of vp_linear_jsd_fwd with
 * the same beta: dz_A = g (1 - beta) p ((log p - log mix) - KL(p || mix)),
 * dz_B = g beta q ((log q - log mix) - KL(q || mix)) formed in the dual GEMM's
 * epilogue, then dhidden = dz . W and dW = dz^T . h for each model asked for
 * (outputs and `precision` as vp_linear_kl_bwd; any output may be NULL, not
 * all). At beta = 0 and 1, vp_linear_kl_bwd with the matching direction. workspace:
 * vp_linear_jsd_bwd_workspace_size(N, V, Da, Db) bytes. */
VP_API size_t vp_linear_jsd_bwd_workspace_size(int64_t N, int64_t V, int64_t Da, int64_t Db);
VP_API vp_status vp_linear_jsd_bwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N,
                                   int64_t V, int64_t Da, int64_t Db, double beta, const vp_rowstat *stats_a,
                                   const vp_rowstat *stats_b, const float *grad_out, void *dha, void *dwa, void *dhb,
                                   void *dwb, int precision, void *workspace, size_t workspace_bytes,
                                   vp_stream stream);

/* ------------------------------------------------------------------------ */
/* Vocabulary-sharded fused linear ops [P2, "Implementation": tensor-parallel */
/* shards of the head's rows, each reducing its own logit tiles; P1, second   */
/* commit message: per-shard max, sum-exp and centred sum combined on the     */
/* row max]. The flow of the sharded forms above, with W's rows as the shard: */
/*  1. shard k (rows [vocab_start_k, vocab_start_k + V_k) of W, passed as    */
/*     weight + vocab_start_k * D with V = V_k) calls vp_linear_*_partial;   */
/*  2. the caller gathers the K arrays shard-major;                          */
/*  3. vp_logprobs_merge / vp_entropy_merge / vp_kl_merge write the outputs  */
/*     and records that the unsharded vp_linear_*_fwd would write;           */
/*  4. each shard calls vp_linear_*_bwd on its rows of W with the merged     */
/*     records: its dW rows are complete, and its dhidden is that shard's    */
/*     term of the sum over shards (dz_k . W_k, rounded to bf16); the caller */
/*     adds the K terms (e.g. an all-reduce). vp_linear_logp_bwd takes a     */
/*     target outside its shard as held elsewhere when the records come from */
/*     vp_logprobs_merge (VP_ROW_SHARDED), and gives VP_ROW_BADTARGET rows   */
/*     NaN gradient rows.                                                    */
/* parts: vp_partial [N], 8-byte aligned; workspace as the unsharded forward */
/* (vp_linear_logp_workspace_size / vp_linear_entropy_workspace_size /       */
/* vp_linear_kl_workspace_size with the shard's V). Argument errors as the   */
/* unsharded forwards.                                                       */
/* ------------------------------------------------------------------------ */

/* The shard's logprobs records: m and S over the shard's logits, z_t and
 * VP_PART_HAS_TARGET when the target (a global id) lies in the shard,
 * VP_PART_IGNORED for a negative target, VP_PART_NANINF for a NaN or +inf
 * logit. A target in another shard sets neither and is not an error here. */
VP_API vp_status vp_linear_logp_partial(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                        int64_t vocab_start, const int64_t *targets, vp_partial *parts,
                                        void *workspace, size_t workspace_bytes, vp_stream stream);

/* The shard's entropy records: m, S and W = sum exp(z - m) (z - m). */
VP_API vp_status vp_linear_entropy_partial(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                           vp_partial *parts, void *workspace, size_t workspace_bytes,
                                           vp_stream stream);

/* The shard's KL(P||Q) records of two models ((P, Q) = (A, B) for
 * VP_KL_REVERSE, (B, A) for VP_KL_FORWARD; wa and wb hold the same shard of
 * the vocabulary): m, S of P, m_b, S_b of Q and W as vp_kl_partial. */
VP_API vp_status vp_linear_kl_partial(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N,
                                      int64_t V, int64_t Da, int64_t Db, int direction, vp_partial *parts,
                                      void *workspace, size_t workspace_bytes, vp_stream stream);

/* ------------------------------------------------------------------------ */
/* Misc                                                                      */
/* ------------------------------------------------------------------------ */

/* Host-buffer transfers (no counterpart on the pages: they let a caller whose
 * data starts in host memory run a whole step through this library). One
 * cudaMemcpyAsync of `bytes` bytes on `stream`, host to device (vp_upload) or
 * device to host (vp_download). The host buffer should be page-locked, or the
 * copy is not asynchronous. bytes = 0 queues nothing; NULL pointers otherwise:
 * VP_ERR_NULL; a failed enqueue: VP_ERR_LAUNCH. */
VP_API vp_status vp_upload(void *dst_device, const void *src_host, size_t bytes, vp_stream stream);
VP_API vp_status vp_download(void *dst_host, const void *src_device, size_t bytes, vp_stream stream);

/* Reads the library's device fault word of the current device into *value
 * and, when `clear` is non-zero, resets it. The word is non-zero only if a
 * kernel's bounded wait on its copy pipeline gave up (bits 0-1: the forward
 * scans' producer / consumers; bits 2-4: the fused-linear GEMMs' producer / MMA /
 * epilogue); that kernel then skipped its outputs and returned instead of
 * spinning. Unlike every other call, this one synchronises with the device.
 * (No counterpart on the pages: a safety net of this implementation.) */
VP_API vp_status vp_fault_status(uint32_t *value, int clear);

/* How many CTAs share one row's vocabulary in the forward scans (logprobs,
 * top-k logprobs, entropy, KL, the generalized JSD's first pass and the
 * vocabulary-shard partials of the first three); process-wide, every device.
 * 1 (the default) streams each row through one CTA. 2 splits the aligned body
 * of every row of 64 KB or more between the two CTAs of a thread-block
 * cluster; the second CTA's partial statistics travel to the first CTA's
 * shared memory, which merges the two in a fixed order and finishes the row.
 * A row's arithmetic depends on this setting, V, the element size and the
 * row's address modulo 16, never on N, so results do not depend on the batch
 * size under either setting (they may differ by rounding between settings).
 * On GB300, 1 measured faster at every batch size tried; 2 is kept as an
 * option. Set it while no forward call is in flight. Other values:
 * VP_ERR_ARG, setting unchanged. (No counterpart on the pages: a scheduling
 * choice of this implementation.) */
VP_API vp_status vp_set_row_split(int ctas);
VP_API int vp_get_row_split(void);
VP_API const char *vp_status_string(int status);
VP_API int vp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VP_H */
