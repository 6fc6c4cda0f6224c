/*
 * vp_oracle.c -- plain fp64 CPU oracle for vocab-wide log-softmax statistics.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * cpu_baseline / reference leg load this library. The product path (the CUDA
 * library and its Python binding) never calls, links or reads it, and this
 * file shares no code, header, table or constant with that path.
 *
 * Sources (each function names the passage it follows):
 *   [P1] page "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
 *        (DeepSpeed pull request 8838): first commit message (the ops and
 *        their fused backward), second commit message and the reviewer's
 *        "Suggested change" (single-read statistics, re-centring on the max,
 *        the support-mismatch flag), the Codex review thread "Guard zero
 *        rescaling before applying infinite shifts" (zero-weight terms), and
 *        the PR description's "Tests" list (the special rows).
 *   [P2] page "[Feat][Kernel] Add TP Fused linear logp Triton" (RL-Kernel pull
 *        request 208): "Implementation" (logp = target logit - LSE of
 *        hidden.W^T, no materialised logits in the kernel) and the review
 *        nitpick on the chunked backward (dz = onehot - exp(logits - lse),
 *        scaled by the upstream gradient, then dhidden = dz.W, dW = dz^T.h).
 *
 * What this file is: the DEFINITIONS written out in fp64. Every input arrives
 * as an exact fp64 copy of the bf16 / fp32 values the GPU reads. Each row is
 * processed in two passes (max, then sums) with the softmax written out; the
 * single-read online (m, S, W) form that the GPU uses is the method under
 * test and does not appear here, except in the *_sharded functions, which
 * restate the re-centring merge of [P1] (second commit message and the
 * reviewer's suggested change) on exact per-shard sums so that the merge
 * itself can be checked against the direct definition.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *   R1 KL direction: "reverse" = KL(A||B), "forward" = KL(B||A), A being the
 *      first argument.
 *   R2 Support mismatch is decided on the logits: KL(P||Q) = +inf when some
 *      j has P_j > -inf and Q_j = -inf, even when p_j underflows.
 *   R3 Per-row precedence: a NaN or +inf in a used input row gives NaN; else
 *      an all -inf P row (S_P = 0) gives NaN; else a mismatch gives +inf;
 *      else the finite formula.
 *   R4 Gradients: NaN rows give NaN gradient rows; a flagged KL row gives a
 *      NaN dP row and the finite dQ = g (q - p); elsewhere positions with
 *      p_j = 0 get exactly 0 in the P-side terms.
 *   R5 Targets: a negative target is ignored (logp 0, zero gradient row); a
 *      target >= 0 outside [vocab_start, vocab_start + V) is a data error:
 *      NaN output and gradient row, and bit 0 of *err is set.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define VPO_ERR_TARGET 1

int vpo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (n >= 1); timing only, the results do not depend on it. */
void vpo_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int vpo_version(void) { return 1; }

/* ------------------------------------------------------------------------ */
/* Row statistics by definition: m = max_j z_j, S = sum_j exp(z_j - m).      */
/* bad = the row holds a NaN or a +inf (R3).                                 */
/* ------------------------------------------------------------------------ */
typedef struct {
    double m;     /* row max over the non-NaN entries; -inf for an all -inf row */
    double S;     /* sum_j exp(z_j - m); 0 for an all -inf row                 */
    double logS;  /* log S                                                     */
    int bad;      /* a NaN or +inf is present                                  */
} row_stats;

static row_stats scan_row(const double *z, int64_t V) {
    row_stats s;
    s.m = -INFINITY;
    s.bad = 0;
    for (int64_t j = 0; j < V; ++j) {
        double v = z[j];
        if (isnan(v) || v == INFINITY) s.bad = 1;
        else if (v > s.m) s.m = v;
    }
    s.S = 0.0;
    if (s.m > -INFINITY) {
        for (int64_t j = 0; j < V; ++j) {
            double v = z[j];
            if (isnan(v) || v == INFINITY) continue;
            s.S += exp(v - s.m);
        }
    }
    s.logS = log(s.S);
    return s;
}

/* log p_j written out: (z_j - m) - log S. -inf where z_j = -inf. */
static double log_prob(double zj, const row_stats *s) { return (zj - s->m) - s->logS; }

/* ------------------------------------------------------------------------ */
/* Logprobs [P1 first commit message: logprobs fwd+bwd; P2 "Implementation"] */
/* ------------------------------------------------------------------------ */
void vpo_logprobs_fwd(const double *x, int64_t N, int64_t V, int64_t vocab_start,
                      const int64_t *targets, double *logp, double *m_out,
                      double *logS_out, int32_t *err) {
    int32_t e = 0;
#pragma omp parallel for schedule(static) reduction(| : e)
    for (int64_t r = 0; r < N; ++r) {
        const double *z = x + r * V;
        row_stats s = scan_row(z, V);
        if (m_out) m_out[r] = s.m;
        if (logS_out) logS_out[r] = s.logS;
        int64_t t = targets[r];
        if (t < 0) { logp[r] = 0.0; continue; }                    /* R5 ignored */
        int64_t loc = t - vocab_start;
        if (loc < 0 || loc >= V) { logp[r] = NAN; e |= VPO_ERR_TARGET; continue; }
        if (s.bad || s.S == 0.0) { logp[r] = NAN; continue; }     /* R3 */
        logp[r] = log_prob(z[loc], &s);
    }
    if (err) *err |= e;
}

/* d logp_t / d z_j = onehot_j - p_j, times g [P2 review nitpick on the
 * chunked backward: dz = -exp(logits - lse), +1 at the owned target, times g]. */
void vpo_logprobs_bwd(const double *x, int64_t N, int64_t V, int64_t vocab_start,
                      const int64_t *targets, const double *g, double *dx) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *z = x + r * V;
        double *d = dx + r * V;
        int64_t t = targets[r];
        if (t < 0) { for (int64_t j = 0; j < V; ++j) d[j] = 0.0; continue; }
        int64_t loc = t - vocab_start;
        row_stats s = scan_row(z, V);
        if (loc < 0 || loc >= V || s.bad || s.S == 0.0) {
            for (int64_t j = 0; j < V; ++j) d[j] = NAN;
            continue;
        }
        for (int64_t j = 0; j < V; ++j) {
            double p = exp(log_prob(z[j], &s));
            double onehot = (j == loc) ? 1.0 : 0.0;
            d[j] = g[r] * (onehot - p);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Several target ids per row (top-k) [P1 PR description, "Tests": duplicate */
/* and ignored top-k ids and a fully ignored row]. targets and g are N x K,  */
/* row-major. Per id, R5: a negative id is ignored (logp 0, no gradient     */
/* term), an id >= 0 outside the shard is a data error (logp NaN, err bit,   */
/* and the row's gradient is NaN). The gradient is that of                   */
/* sum_k g_rk logp_rk: sum over the ids not ignored of g_rk (onehot - p),    */
/* so duplicate ids add up.                                                  */
/* ------------------------------------------------------------------------ */
void vpo_logprobs_topk_fwd(const double *x, int64_t N, int64_t V, int64_t K, int64_t vocab_start,
                           const int64_t *targets, double *logp, int32_t *err) {
    int32_t e = 0;
#pragma omp parallel for schedule(static) reduction(| : e)
    for (int64_t r = 0; r < N; ++r) {
        const double *z = x + r * V;
        row_stats s = scan_row(z, V);
        for (int64_t k = 0; k < K; ++k) {
            int64_t t = targets[r * K + k];
            double *out = logp + r * K + k;
            if (t < 0) { *out = 0.0; continue; }
            int64_t loc = t - vocab_start;
            if (loc < 0 || loc >= V) { *out = NAN; e |= VPO_ERR_TARGET; continue; }
            *out = (s.bad || s.S == 0.0) ? NAN : log_prob(z[loc], &s);
        }
    }
    if (err) *err |= e;
}

void vpo_logprobs_topk_bwd(const double *x, int64_t N, int64_t V, int64_t K, int64_t vocab_start,
                           const int64_t *targets, const double *g, double *dx) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *z = x + r * V;
        double *d = dx + r * V;
        row_stats s = scan_row(z, V);
        double gsum = 0.0;
        int used = 0, bad = 0;
        for (int64_t k = 0; k < K; ++k) {
            int64_t t = targets[r * K + k];
            if (t < 0) continue;
            int64_t loc = t - vocab_start;
            if (loc < 0 || loc >= V) bad = 1;
            used = 1;
            gsum += g[r * K + k];
        }
        if (!used) { for (int64_t j = 0; j < V; ++j) d[j] = 0.0; continue; }
        if (bad || s.bad || s.S == 0.0) { for (int64_t j = 0; j < V; ++j) d[j] = NAN; continue; }
        for (int64_t j = 0; j < V; ++j) d[j] = -gsum * exp(log_prob(z[j], &s));
        for (int64_t k = 0; k < K; ++k) {
            int64_t t = targets[r * K + k];
            if (t >= 0) d[t - vocab_start] += g[r * K + k];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Entropy H = -sum_{p_j>0} p_j log p_j  [P1 first and second commit msgs]  */
/* ------------------------------------------------------------------------ */
static double entropy_row(const double *z, int64_t V, const row_stats *s) {
    if (s->bad || s->S == 0.0) return NAN;                        /* R3 */
    double H = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        double lp = log_prob(z[j], s);
        double p = exp(lp);
        if (p > 0.0) H -= p * lp;                                 /* zero-weight terms skipped */
    }
    return H;
}

void vpo_entropy_fwd(const double *x, int64_t N, int64_t V, double *H,
                     double *m_out, double *logS_out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *z = x + r * V;
        row_stats s = scan_row(z, V);
        if (m_out) m_out[r] = s.m;
        if (logS_out) logS_out[r] = s.logS;
        H[r] = entropy_row(z, V, &s);
    }
}

/* dH/dz_j = -p_j (log p_j + H), 0 where p_j = 0 (R4), times g. */
void vpo_entropy_bwd(const double *x, int64_t N, int64_t V, const double *g, double *dx) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *z = x + r * V;
        double *d = dx + r * V;
        row_stats s = scan_row(z, V);
        double H = entropy_row(z, V, &s);
        if (isnan(H)) { for (int64_t j = 0; j < V; ++j) d[j] = NAN; continue; }
        for (int64_t j = 0; j < V; ++j) {
            double lp = log_prob(z[j], &s);
            double p = exp(lp);
            d[j] = (p > 0.0) ? -g[r] * p * (lp + H) : 0.0;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* KL(P||Q) = sum_{p_j>0} p_j (log p_j - log q_j)  [P1 commit messages,     */
/* reviewer's suggested change: the support-mismatch flag on the logits]    */
/* ------------------------------------------------------------------------ */
static int mismatch(const double *P, const double *Q, int64_t V) {   /* R2 */
    for (int64_t j = 0; j < V; ++j)
        if (P[j] > -INFINITY && Q[j] == -INFINITY) return 1;
    return 0;
}

static double kl_row(const double *P, const double *Q, int64_t V,
                     const row_stats *sp, const row_stats *sq) {
    if (sp->bad || sq->bad) return NAN;                           /* R3 */
    if (sp->S == 0.0) return NAN;
    if (mismatch(P, Q, V)) return INFINITY;
    double kl = 0.0;
    for (int64_t j = 0; j < V; ++j) {
        double lp = log_prob(P[j], sp);
        double p = exp(lp);
        if (p > 0.0) kl += p * (lp - log_prob(Q[j], sq));
    }
    return kl;
}

/* direction 0 (reverse): KL(A||B); direction 1 (forward): KL(B||A)  (R1). */
void vpo_kl_fwd(const double *a, const double *b, int64_t N, int64_t V, int direction,
                double *kl, double *ma, double *logSa, double *mb, double *logSb) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *A = a + r * V, *B = b + r * V;
        row_stats sa = scan_row(A, V), sb = scan_row(B, V);
        if (ma) ma[r] = sa.m;
        if (logSa) logSa[r] = sa.logS;
        if (mb) mb[r] = sb.m;
        if (logSb) logSb[r] = sb.logS;
        kl[r] = direction == 0 ? kl_row(A, B, V, &sa, &sb) : kl_row(B, A, V, &sb, &sa);
    }
}

/* dKL/dP_j = p_j (log p_j - log q_j - KL), dKL/dQ_j = q_j - p_j; times g (R4). */
static void kl_bwd_row(const double *P, const double *Q, int64_t V, double g,
                       double *dP, double *dQ) {
    row_stats sp = scan_row(P, V), sq = scan_row(Q, V);
    double kl = kl_row(P, Q, V, &sp, &sq);
    if (isnan(kl)) {
        for (int64_t j = 0; j < V; ++j) { if (dP) dP[j] = NAN; if (dQ) dQ[j] = NAN; }
        return;
    }
    for (int64_t j = 0; j < V; ++j) {
        double lp = log_prob(P[j], &sp), lq = log_prob(Q[j], &sq);
        double p = exp(lp), q = exp(lq);
        if (dQ) dQ[j] = g * (q - p);
        if (dP) {
            if (isinf(kl)) dP[j] = NAN;
            else dP[j] = (p > 0.0) ? g * p * (lp - lq - kl) : 0.0;
        }
    }
}

void vpo_kl_bwd(const double *a, const double *b, int64_t N, int64_t V, int direction,
                const double *g, double *da, double *db) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *A = a + r * V, *B = b + r * V;
        double *dA = da ? da + r * V : NULL, *dB = db ? db + r * V : NULL;
        if (direction == 0) kl_bwd_row(A, B, V, g[r], dA, dB);
        else kl_bwd_row(B, A, V, g[r], dB, dA);
    }
}

/* ------------------------------------------------------------------------ */
/* Generalized Jensen-Shannon divergence [P1, the commit message that adds  */
/* vocab_parallel_jsd: "Changes", "Scope and limitations"]. The page fixes  */
/* beta = 0 as forward KL and beta = 1 as reverse KL (explicit endpoint     */
/* branches) and, for 0 < beta < 1, a GKD-style divergence made of two      */
/* KL-to-mixture expectations, but prints no formula. Reading R13: with     */
/* p = softmax(A) (the student, first argument), q = softmax(B) (the        */
/* teacher) and the mixture mix = beta q + (1 - beta) p,                    */
/*   JSD = beta KL(q || mix) + (1 - beta) KL(p || mix).                      */
/* Gradients through the two softmaxes (R13):                               */
/*   dJSD/dA_j = (1 - beta) p_j ((log p_j - log mix_j) - KL(p || mix)),      */
/*   dJSD/dB_j = beta q_j ((log q_j - log mix_j) - KL(q || mix)).            */
/* A row with a NaN or +inf in A or B, or without a finite logit in A or B, */
/* gives NaN and NaN gradient rows (R3, R4); terms with p_j = 0 (q_j = 0)    */
/* contribute 0 to KL(p || mix) (KL(q || mix)).                              */
/* ------------------------------------------------------------------------ */
static double jsd_row(const double *A, const double *B, int64_t V, double beta,
                      const row_stats *sa, const row_stats *sb, double *ka, double *kb) {
    *ka = *kb = NAN;
    if (sa->bad || sb->bad || sa->S == 0.0 || sb->S == 0.0) return NAN;
    double kp = 0.0, kq = 0.0;   /* KL(p || mix), KL(q || mix) */
    for (int64_t j = 0; j < V; ++j) {
        double lp = log_prob(A[j], sa), lq = log_prob(B[j], sb);
        double p = exp(lp), q = exp(lq);
        double lmix = log(beta * q + (1.0 - beta) * p);
        if (p > 0.0) kp += p * (lp - lmix);
        if (q > 0.0) kq += q * (lq - lmix);
    }
    *ka = kp;
    *kb = kq;
    return beta * kq + (1.0 - beta) * kp;
}

void vpo_jsd_fwd(const double *a, const double *b, int64_t N, int64_t V, double beta, double *jsd) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *A = a + r * V, *B = b + r * V;
        row_stats sa = scan_row(A, V), sb = scan_row(B, V);
        double ka, kb;
        if (beta == 0.0) jsd[r] = kl_row(B, A, V, &sb, &sa);        /* forward KL(B || A) */
        else if (beta == 1.0) jsd[r] = kl_row(A, B, V, &sa, &sb);   /* reverse KL(A || B) */
        else jsd[r] = jsd_row(A, B, V, beta, &sa, &sb, &ka, &kb);
    }
}

void vpo_jsd_bwd(const double *a, const double *b, int64_t N, int64_t V, double beta,
                 const double *g, double *da, double *db) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *A = a + r * V, *B = b + r * V;
        double *dA = da ? da + r * V : NULL, *dB = db ? db + r * V : NULL;
        if (beta == 0.0) { kl_bwd_row(B, A, V, g[r], dB, dA); continue; }
        if (beta == 1.0) { kl_bwd_row(A, B, V, g[r], dA, dB); continue; }
        row_stats sa = scan_row(A, V), sb = scan_row(B, V);
        double ka, kb;
        double jsd = jsd_row(A, B, V, beta, &sa, &sb, &ka, &kb);
        for (int64_t j = 0; j < V; ++j) {
            if (isnan(jsd)) { if (dA) dA[j] = NAN; if (dB) dB[j] = NAN; continue; }
            double lp = log_prob(A[j], &sa), lq = log_prob(B[j], &sb);
            double p = exp(lp), q = exp(lq);
            double lmix = log(beta * q + (1.0 - beta) * p);
            if (dA) dA[j] = (p > 0.0) ? g[r] * (1.0 - beta) * p * ((lp - lmix) - ka) : 0.0;
            if (dB) dB[j] = (q > 0.0) ? g[r] * beta * q * ((lq - lmix) - kb) : 0.0;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Sharded forms: the re-centring merge of [P1] (second commit message and  */
/* the reviewer's suggested change), with zero-weight terms skipped as in   */
/* the Codex thread "Guard zero rescaling before applying infinite shifts". */
/* Shard s covers columns [cuts[s], cuts[s+1]); shards may be empty.        */
/* Per shard, the sums are exact fp64 sums over the shard (two passes);     */
/* only the merge is the method's.                                          */
/* ------------------------------------------------------------------------ */
typedef struct { double m, S, W; int bad; } shard_ent;

static shard_ent shard_entropy(const double *z, int64_t lo, int64_t hi) {
    shard_ent s;
    row_stats st = scan_row(z + lo, hi - lo);
    s.m = st.m; s.S = st.S; s.bad = st.bad; s.W = 0.0;
    if (st.m > -INFINITY) {
        for (int64_t j = lo; j < hi; ++j) {
            if (isnan(z[j]) || z[j] == INFINITY) continue;
            double e = exp(z[j] - s.m);
            if (e > 0.0) s.W += e * (z[j] - s.m);  /* sum e^(z-m)(z-m) */
        }
    }
    return s;
}

/* Entropy of a row from its k shard records: re-centre on the row max. */
static double merge_entropy(const shard_ent *parts, int k) {
    double m = -INFINITY;
    int bad = 0;
    for (int s = 0; s < k; ++s) {
        bad |= parts[s].bad;
        if (parts[s].m > m) m = parts[s].m;
    }
    double S = 0.0, W = 0.0;
    for (int s = 0; s < k; ++s) {
        double alpha = exp(parts[s].m - m);     /* 0 for an empty / all -inf shard */
        double w = alpha * parts[s].S;
        if (w == 0.0) continue;                  /* zero-weight shard skipped */
        S += w;
        W += alpha * (parts[s].W - (m - parts[s].m) * parts[s].S);
    }
    return (bad || S == 0.0) ? NAN : log(S) - W / S;
}

void vpo_entropy_sharded(const double *x, int64_t N, int64_t V, const int64_t *cuts,
                         int k, double *H) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *z = x + r * V;
        shard_ent parts[64];
        for (int s = 0; s < k; ++s) parts[s] = shard_entropy(z, cuts[s], cuts[s + 1]);
        H[r] = merge_entropy(parts, k);
    }
}

/* Entropy from records laid out as vpo_shard_stats writes them, K x N x 4,
 * shard-major (K <= 64). */
void vpo_merge_entropy_records(const double *recs, int64_t K, int64_t N, double *H) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        shard_ent parts[64];
        for (int64_t s = 0; s < K; ++s) {
            const double *o = recs + 4 * (s * N + r);
            parts[s].m = o[0]; parts[s].S = o[1]; parts[s].W = o[2]; parts[s].bad = o[3] != 0.0;
        }
        H[r] = merge_entropy(parts, (int)K);
    }
}

typedef struct { double mp, Sp, mq, Sq, W; int bad, flag; } shard_kl;

static shard_kl shard_kl_stats(const double *P, const double *Q, int64_t lo, int64_t hi) {
    shard_kl s;
    row_stats sp = scan_row(P + lo, hi - lo), sq = scan_row(Q + lo, hi - lo);
    s.mp = sp.m; s.Sp = sp.S; s.mq = sq.m; s.Sq = sq.S;
    s.bad = sp.bad | sq.bad;
    s.flag = mismatch(P + lo, Q + lo, hi - lo);
    s.W = 0.0;
    if (sp.m > -INFINITY && !s.flag && !s.bad) {
        for (int64_t j = lo; j < hi; ++j) {
            double e = exp(P[j] - s.mp);
            if (e > 0.0) s.W += e * ((P[j] - s.mp) - (Q[j] - s.mq));
        }
    }
    return s;
}

/* KL of a row from its k shard records: re-centre P and Q on their row maxima. */
static double merge_kl(const shard_kl *parts, int k) {
    double mp = -INFINITY, mq = -INFINITY;
    int bad = 0, flag = 0;
    for (int s = 0; s < k; ++s) {
        bad |= parts[s].bad;
        flag |= parts[s].flag;
        if (parts[s].mp > mp) mp = parts[s].mp;
        if (parts[s].mq > mq) mq = parts[s].mq;
    }
    double Sp = 0.0, Sq = 0.0, W = 0.0;
    for (int s = 0; s < k; ++s) {
        double ap = exp(parts[s].mp - mp), aq = exp(parts[s].mq - mq);
        if (aq * parts[s].Sq != 0.0) Sq += aq * parts[s].Sq;
        double w = ap * parts[s].Sp;
        if (w == 0.0) continue;
        Sp += w;
        double dp = mp - parts[s].mp, dq = mq - parts[s].mq;
        W += ap * (parts[s].W - (dp - dq) * parts[s].Sp);
    }
    if (bad || Sp == 0.0) return NAN;
    if (flag) return INFINITY;
    return W / Sp - log(Sp) + log(Sq);
}

/* Same direction convention as vpo_kl_fwd (R1). */
void vpo_kl_sharded(const double *a, const double *b, int64_t N, int64_t V, int direction,
                    const int64_t *cuts, int k, double *kl) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *P = (direction == 0 ? a : b) + r * V;
        const double *Q = (direction == 0 ? b : a) + r * V;
        shard_kl parts[64];
        for (int s = 0; s < k; ++s) parts[s] = shard_kl_stats(P, Q, cuts[s], cuts[s + 1]);
        kl[r] = merge_kl(parts, k);
    }
}

/* KL from records laid out as vpo_shard_kl_stats writes them, K x N x 7,
 * shard-major (K <= 64). */
void vpo_merge_kl_records(const double *recs, int64_t K, int64_t N, double *kl) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        shard_kl parts[64];
        for (int64_t s = 0; s < K; ++s) {
            const double *o = recs + 7 * (s * N + r);
            parts[s].mp = o[0]; parts[s].Sp = o[1]; parts[s].mq = o[2]; parts[s].Sq = o[3];
            parts[s].W = o[4]; parts[s].bad = o[5] != 0.0; parts[s].flag = o[6] != 0.0;
        }
        kl[r] = merge_kl(parts, (int)K);
    }
}

/* Per-shard records of the sharded forms: the max, sum-exp and centred     */
/* weighted sum that each vocabulary shard reduces on its own before the    */
/* merge above ([P1] second commit message). Exposed so that per-shard      */
/* records computed elsewhere can be checked against their definition.      */
/* Entropy / logprobs: out[4r + 0..3] = m, S, W, bad.                       */
void vpo_shard_stats(const double *x, int64_t N, int64_t V, int64_t lo, int64_t hi, double *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        shard_ent s = shard_entropy(x + r * V, lo, hi);
        double *o = out + 4 * r;
        o[0] = s.m; o[1] = s.S; o[2] = s.W; o[3] = s.bad;
    }
}

/* KL(P||Q), direction as in vpo_kl_fwd (R1): out[7r + 0..6] = m_P, S_P,    */
/* m_Q, S_Q, W, bad, mismatch. W is left 0 on a bad or mismatched shard.    */
void vpo_shard_kl_stats(const double *a, const double *b, int64_t N, int64_t V, int direction,
                        int64_t lo, int64_t hi, double *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        const double *P = (direction == 0 ? a : b) + r * V;
        const double *Q = (direction == 0 ? b : a) + r * V;
        shard_kl s = shard_kl_stats(P, Q, lo, hi);
        double *o = out + 7 * r;
        o[0] = s.mp; o[1] = s.Sp; o[2] = s.mq; o[3] = s.Sq; o[4] = s.W; o[5] = s.bad; o[6] = s.flag;
    }
}

/* ------------------------------------------------------------------------ */
/* Fused linear logp [P2 "Implementation"; review nitpick on the backward]   */
/* logits_rj = sum_k h_rk W_jk in fp64, never rounded.                       */
/* ------------------------------------------------------------------------ */
void vpo_linear_logits(const double *h, const double *W, int64_t N, int64_t V, int64_t D,
                       double *logits) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r)
        for (int64_t j = 0; j < V; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < D; ++k) acc += h[r * D + k] * W[j * D + k];
            logits[r * V + j] = acc;
        }
}

/* logp_r = logit_{r,t} - LSE_j logit_{r,j}; one row of logits at a time. */
void vpo_linear_logp_fwd(const double *h, const double *W, int64_t N, int64_t V, int64_t D,
                         int64_t vocab_start, const int64_t *targets, double *logp,
                         double *m_out, double *logS_out, double *row_scratch, int32_t *err) {
    /* row_scratch: caller-owned [omp threads][V] fp64 */
    int32_t e = 0;
#pragma omp parallel for schedule(static) reduction(| : e)
    for (int64_t r = 0; r < N; ++r) {
#ifdef _OPENMP
        double *z = row_scratch + (int64_t)omp_get_thread_num() * V;
#else
        double *z = row_scratch;
#endif
        vpo_linear_logits(h + r * D, W, 1, V, D, z);
        int32_t er = 0;
        vpo_logprobs_fwd(z, 1, V, vocab_start, targets + r, logp + r,
                         m_out ? m_out + r : NULL, logS_out ? logS_out + r : NULL, &er);
        e |= er;
    }
    if (err) *err |= e;
}

/* dz = g (onehot - p) per row (the logprobs backward of each logits row);
 * dhidden = dz . W; dW = dz^T . h.  dz_scratch: caller-owned [N][V] fp64.
 * dh or dW may be NULL. */
void vpo_linear_logp_bwd(const double *h, const double *W, int64_t N, int64_t V, int64_t D,
                         int64_t vocab_start, const int64_t *targets, const double *g,
                         double *dh, double *dW, double *dz_scratch) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < N; ++r) {
        double *z = dz_scratch + r * V;
        vpo_linear_logits(h + r * D, W, 1, V, D, z);
        row_stats s = scan_row(z, V);
        int64_t t = targets[r];
        int64_t loc = t - vocab_start;
        if (t < 0) { for (int64_t j = 0; j < V; ++j) z[j] = 0.0; continue; }
        if (loc < 0 || loc >= V || s.bad || s.S == 0.0) {
            for (int64_t j = 0; j < V; ++j) z[j] = NAN;
            continue;
        }
        for (int64_t j = 0; j < V; ++j) {
            double p = exp(log_prob(z[j], &s));
            z[j] = g[r] * (((j == loc) ? 1.0 : 0.0) - p);
        }
    }
    if (dh) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < N; ++r) {
            double *out = dh + r * D;
            for (int64_t k = 0; k < D; ++k) out[k] = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                double c = dz_scratch[r * V + j];
                for (int64_t k = 0; k < D; ++k) out[k] += c * W[j * D + k];
            }
        }
    }
    if (dW) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < V; ++j) {
            double *out = dW + j * D;
            for (int64_t k = 0; k < D; ++k) out[k] = 0.0;
            for (int64_t r = 0; r < N; ++r) {
                double c = dz_scratch[r * V + j];
                for (int64_t k = 0; k < D; ++k) out[k] += c * h[r * D + k];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Fused linear entropy and KL: the entropy of softmax(h . W^T), and the KL   */
/* between the next-token distributions of two models, each with its own      */
/* hidden states and LM-head weight [P1, JSD pull request "Motivation": a     */
/* teacher-student divergence computed from tiled LM-head projections         */
/* without the full logits]. The definitions are those of vpo_entropy_* and  */
/* vpo_kl_* applied to the fp64 logits rows h_r . W_j (materialised here);    */
/* the chain rule is the one of vpo_linear_logp_bwd [P2, review nitpick]:     */
/* dhidden = dz . W, dW = dz^T . h.                                           */
/* ------------------------------------------------------------------------ */

/* dh = dz . W ([N][D]) and dW = dz^T . h ([V][D]) for a materialised dz [N][V];
 * either output may be NULL. */
static void linear_chain_rule(const double *h, const double *W, int64_t N, int64_t V, int64_t D,
                              const double *dz, double *dh, double *dW) {
    if (dh) {
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < N; ++r) {
            double *out = dh + r * D;
            for (int64_t k = 0; k < D; ++k) out[k] = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                double c = dz[r * V + j];
                for (int64_t k = 0; k < D; ++k) out[k] += c * W[j * D + k];
            }
        }
    }
    if (dW) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < V; ++j) {
            double *out = dW + j * D;
            for (int64_t k = 0; k < D; ++k) out[k] = 0.0;
            for (int64_t r = 0; r < N; ++r) {
                double c = dz[r * V + j];
                for (int64_t k = 0; k < D; ++k) out[k] += c * h[r * D + k];
            }
        }
    }
}

/* H_r, m_r, logS_r of the logits h_r . W^T. logits: caller-owned [N][V]. */
void vpo_linear_entropy_fwd(const double *h, const double *W, int64_t N, int64_t V, int64_t D,
                            double *H, double *m_out, double *logS_out, double *logits) {
    vpo_linear_logits(h, W, N, V, D, logits);
    vpo_entropy_fwd(logits, N, V, H, m_out, logS_out);
}

/* dhidden and dW of sum_r g_r H_r. scratch: caller-owned [2][N][V]. */
void vpo_linear_entropy_bwd(const double *h, const double *W, int64_t N, int64_t V, int64_t D,
                            const double *g, double *dh, double *dW, double *scratch) {
    double *logits = scratch, *dz = scratch + N * V;
    vpo_linear_logits(h, W, N, V, D, logits);
    vpo_entropy_bwd(logits, N, V, g, dz);
    linear_chain_rule(h, W, N, V, D, dz, dh, dW);
}

/* KL between model A (ha [N][Da], Wa [V][Da]) and model B (hb [N][Db], Wb [V][Db])
 * in the direction of vpo_kl_fwd (R1), with both models' row max and log-sum.
 * scratch: caller-owned [2][N][V]. */
void vpo_linear_kl_fwd(const double *ha, const double *Wa, const double *hb, const double *Wb, int64_t N,
                       int64_t V, int64_t Da, int64_t Db, int direction, double *kl, double *ma, double *lsa,
                       double *mb, double *lsb, double *scratch) {
    double *za = scratch, *zb = scratch + N * V;
    vpo_linear_logits(ha, Wa, N, V, Da, za);
    vpo_linear_logits(hb, Wb, N, V, Db, zb);
    vpo_kl_fwd(za, zb, N, V, direction, kl, ma, lsa, mb, lsb);
}

/* dhidden and dW of both models for sum_r g_r KL_r; any output may be NULL.
 * scratch: caller-owned [4][N][V]. */
void vpo_linear_kl_bwd(const double *ha, const double *Wa, const double *hb, const double *Wb, int64_t N,
                       int64_t V, int64_t Da, int64_t Db, int direction, const double *g, double *dha,
                       double *dWa, double *dhb, double *dWb, double *scratch) {
    double *za = scratch, *zb = scratch + N * V, *dza = scratch + 2 * N * V, *dzb = scratch + 3 * N * V;
    vpo_linear_logits(ha, Wa, N, V, Da, za);
    vpo_linear_logits(hb, Wb, N, V, Db, zb);
    vpo_kl_bwd(za, zb, N, V, direction, g, dza, dzb);
    linear_chain_rule(ha, Wa, N, V, Da, dza, dha, dWa);
    linear_chain_rule(hb, Wb, N, V, Db, dzb, dhb, dWb);
}

/* Fused linear generalized JSD of two models [P1, the commit message adding
 * vocab_parallel_jsd: "Motivation" (TRL's trainer computes KL/JSD from tiled
 * LM-head projections without the full logits) and "Changes"]: the JSD of
 * vpo_jsd_fwd (R13, with its beta = 0 / 1 endpoints) applied to the fp64
 * logits rows of model A (ha . Wa^T, the student) and model B (hb . Wb^T, the
 * teacher). scratch: caller-owned [2][N][V]. */
void vpo_linear_jsd_fwd(const double *ha, const double *Wa, const double *hb, const double *Wb, int64_t N,
                        int64_t V, int64_t Da, int64_t Db, double beta, double *jsd, double *scratch) {
    double *za = scratch, *zb = scratch + N * V;
    vpo_linear_logits(ha, Wa, N, V, Da, za);
    vpo_linear_logits(hb, Wb, N, V, Db, zb);
    vpo_jsd_fwd(za, zb, N, V, beta, jsd);
}

/* dhidden and dW of both models for sum_r g_r JSD_r; any output may be NULL.
 * scratch: caller-owned [4][N][V]. */
void vpo_linear_jsd_bwd(const double *ha, const double *Wa, const double *hb, const double *Wb, int64_t N,
                        int64_t V, int64_t Da, int64_t Db, double beta, const double *g, double *dha, double *dWa,
                        double *dhb, double *dWb, double *scratch) {
    double *za = scratch, *zb = scratch + N * V, *dza = scratch + 2 * N * V, *dzb = scratch + 3 * N * V;
    vpo_linear_logits(ha, Wa, N, V, Da, za);
    vpo_linear_logits(hb, Wb, N, V, Db, zb);
    vpo_jsd_bwd(za, zb, N, V, beta, g, dza, dzb);
    linear_chain_rule(ha, Wa, N, V, Da, dza, dha, dWa);
    linear_chain_rule(hb, Wb, N, V, Db, dzb, dhb, dWb);
}
