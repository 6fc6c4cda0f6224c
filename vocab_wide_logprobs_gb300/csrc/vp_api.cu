// vp_api.cu -- the extern "C" entry points declared in include/vp.h.
//
// Each entry point checks its arguments on the host (no device access, no
// allocation, no synchronisation), fills a launcher argument block and queues
// the kernel on the caller's stream. The launch shape is chosen from V and the
// dtype alone.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "vp.h"
#include "vp_launch.h"

static_assert(sizeof(vp_rowstat) == 32, "vp_rowstat is 32 bytes");
static_assert(sizeof(vp_partial) == 40, "vp_partial is 40 bytes");

namespace {

constexpr int64_t kMaxV = 2147483647LL;
constexpr int64_t kMaxRowsPerLaunch = 2147483647LL;  // one CTA per row in the forward

// 0 = unknown, 1 = sm_103, 2 = other
std::atomic<int> g_dev_ok[64];

vp_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return VP_ERR_DEVICE;
    if (dev < 0 || dev >= 64) return VP_ERR_DEVICE;
    int known = g_dev_ok[dev].load(std::memory_order_relaxed);
    if (known == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return VP_ERR_DEVICE;
        known = (major == 10 && minor == 3) ? 1 : 2;
        g_dev_ok[dev].store(known, std::memory_order_relaxed);
    }
    return known == 1 ? VP_OK : VP_ERR_DEVICE;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t elem_size(int dtype) { return dtype == VP_BF16 ? 2 : 4; }

// Shared checks of the row description.
vp_status check_rows(int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o, int64_t s_i) {
    if (dtype != VP_F32 && dtype != VP_BF16) return VP_ERR_DTYPE;
    if (N < 0 || N > kMaxRowsPerLaunch || V < 1 || V > kMaxV || R < 1) return VP_ERR_SHAPE;
    if (s_o < 0 || s_i < 0) return VP_ERR_LAYOUT;
    return VP_OK;
}

vp_status launched(cudaError_t e) { return e == cudaSuccess ? VP_OK : VP_ERR_LAUNCH; }

}  // namespace

extern "C" {

vp_status vp_logprobs_fwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                          int64_t s_i, int64_t vocab_start, const int64_t *targets, float *logp,
                          vp_rowstat *stats, int32_t *err_word, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!x || !targets || !logp || !stats) return VP_ERR_NULL;
    if (!aligned(x, elem_size(dtype)) || !aligned(targets, 8) || !aligned(logp, 4) || !aligned(stats, 16) ||
        !aligned(err_word, 4))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::StatsArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, vocab_start, targets, logp, stats, err_word,
                    (cudaStream_t)stream};
    return launched(vp::launch_logprobs_fwd(a));
}

vp_status vp_logprobs_bwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                          int64_t s_i, int64_t vocab_start, const int64_t *targets, const vp_rowstat *stats,
                          const float *grad_out, void *dx, int32_t *err_word, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!x || !targets || !stats || !grad_out || !dx) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(dx, es) || !aligned(targets, 8) || !aligned(stats, 16) ||
        !aligned(grad_out, 4) || !aligned(err_word, 4))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::GradArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, vocab_start, stats, grad_out, targets, dx, err_word,
                   (cudaStream_t)stream};
    return launched(vp::launch_logprobs_bwd(a));
}

vp_status vp_logprobs_topk_fwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                               int64_t s_i, int64_t vocab_start, const int64_t *targets, int64_t K, float *logp,
                               vp_rowstat *stats, int32_t *err_word, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (K < 1 || K > kMaxRowsPerLaunch / (N > 0 ? N : 1)) return VP_ERR_SHAPE;
    if (N == 0) return VP_OK;
    if (!x || !targets || !logp || !stats) return VP_ERR_NULL;
    if (!aligned(x, elem_size(dtype)) || !aligned(targets, 8) || !aligned(logp, 4) || !aligned(stats, 16) ||
        !aligned(err_word, 4))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::StatsArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, vocab_start, targets, logp, stats, err_word,
                    (cudaStream_t)stream};
    a.K = K;
    return launched(vp::launch_logprobs_topk_fwd(a));
}

vp_status vp_logprobs_topk_bwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                               int64_t s_i, int64_t vocab_start, const int64_t *targets, int64_t K,
                               const vp_rowstat *stats, const float *grad_out, void *dx, int32_t *err_word,
                               vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (K < 1 || K > kMaxRowsPerLaunch / (N > 0 ? N : 1)) return VP_ERR_SHAPE;
    if (N == 0) return VP_OK;
    if (!x || !targets || !stats || !grad_out || !dx) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(dx, es) || !aligned(targets, 8) || !aligned(stats, 16) ||
        !aligned(grad_out, 4) || !aligned(err_word, 4))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::GradArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, vocab_start, stats, grad_out, targets, dx, err_word,
                   (cudaStream_t)stream};
    a.K = K;
    return launched(vp::launch_logprobs_topk_bwd(a));
}

vp_status vp_entropy_fwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o, int64_t s_i,
                         float *H, vp_rowstat *stats, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!x || !H || !stats) return VP_ERR_NULL;
    if (!aligned(x, elem_size(dtype)) || !aligned(H, 4) || !aligned(stats, 16)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::StatsArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, 0, nullptr, H, stats, nullptr, (cudaStream_t)stream};
    return launched(vp::launch_entropy_fwd(a));
}

vp_status vp_entropy_bwd(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o, int64_t s_i,
                         const vp_rowstat *stats, const float *grad_out, void *dx, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!x || !stats || !grad_out || !dx) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(x, es) || !aligned(dx, es) || !aligned(stats, 16) || !aligned(grad_out, 4)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::GradArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, 0, stats, grad_out, nullptr, dx, nullptr,
                   (cudaStream_t)stream};
    return launched(vp::launch_entropy_bwd(a));
}

vp_status vp_kl_fwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                    int64_t s_i, int direction, float *kl, vp_rowstat *stats_a, vp_rowstat *stats_b,
                    vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (direction != VP_KL_REVERSE && direction != VP_KL_FORWARD) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!a || !b || !kl || !stats_a || !stats_b) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(a, es) || !aligned(b, es) || !aligned(kl, 4) || !aligned(stats_a, 16) || !aligned(stats_b, 16))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    const bool rev = direction == VP_KL_REVERSE;  // reverse: P = A, Q = B
    vp::KLFwdArgs k{rev ? a : b, rev ? b : a, dtype == VP_BF16, N, V, R, s_o, s_i, kl,
                    rev ? (void *)stats_a : (void *)stats_b, rev ? (void *)stats_b : (void *)stats_a,
                    (cudaStream_t)stream};
    return launched(vp::launch_kl_fwd(k));
}

// ---------------------------------------------------------------------------
// Generalized JSD
// ---------------------------------------------------------------------------
vp_status vp_jsd_fwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                     int64_t s_i, double beta, float *jsd, vp_rowstat *stats_a, vp_rowstat *stats_b,
                     vp_stream stream) {
    if (!(beta >= 0.0 && beta <= 1.0)) return VP_ERR_ARG;
    if (beta == 0.0) return vp_kl_fwd(a, b, dtype, N, V, R, s_o, s_i, VP_KL_FORWARD, jsd, stats_a, stats_b, stream);
    if (beta == 1.0) return vp_kl_fwd(a, b, dtype, N, V, R, s_o, s_i, VP_KL_REVERSE, jsd, stats_a, stats_b, stream);
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!a || !b || !jsd || !stats_a || !stats_b) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(a, es) || !aligned(b, es) || !aligned(jsd, 4) || !aligned(stats_a, 16) || !aligned(stats_b, 16))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::JsdFwdArgs k{a, b, dtype == VP_BF16, N, V, R, s_o, s_i, beta, jsd, stats_a, stats_b, (cudaStream_t)stream};
    return launched(vp::launch_jsd_fwd(k));
}

vp_status vp_jsd_bwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                     int64_t s_i, double beta, const vp_rowstat *stats_a, const vp_rowstat *stats_b,
                     const float *grad_out, void *da, void *db, vp_stream stream) {
    if (!(beta >= 0.0 && beta <= 1.0)) return VP_ERR_ARG;
    if (beta == 0.0)
        return vp_kl_bwd(a, b, dtype, N, V, R, s_o, s_i, VP_KL_FORWARD, stats_a, stats_b, grad_out, da, db, stream);
    if (beta == 1.0)
        return vp_kl_bwd(a, b, dtype, N, V, R, s_o, s_i, VP_KL_REVERSE, stats_a, stats_b, grad_out, da, db, stream);
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!da && !db) return VP_ERR_ARG;
    if (!a || !b || !stats_a || !stats_b || !grad_out) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(a, es) || !aligned(b, es) || !aligned(da, es) || !aligned(db, es) || !aligned(stats_a, 16) ||
        !aligned(stats_b, 16) || !aligned(grad_out, 4))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::JsdBwdArgs k{a, b, dtype == VP_BF16, N, V, R, s_o, s_i, beta, stats_a, stats_b, grad_out, da, db,
                     (cudaStream_t)stream};
    return launched(vp::launch_jsd_bwd(k));
}

// ---------------------------------------------------------------------------
// Vocabulary-sharded forms
// ---------------------------------------------------------------------------
vp_status vp_logprobs_partial(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o, int64_t s_i,
                              int64_t vocab_start, const int64_t *targets, vp_partial *parts, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!x || !targets || !parts) return VP_ERR_NULL;
    if (!aligned(x, elem_size(dtype)) || !aligned(targets, 8) || !aligned(parts, 8)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::StatsArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, vocab_start, targets, nullptr, nullptr, nullptr,
                    (cudaStream_t)stream, parts};
    return launched(vp::launch_logprobs_fwd(a));
}

vp_status vp_entropy_partial(const void *x, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o, int64_t s_i,
                             vp_partial *parts, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!x || !parts) return VP_ERR_NULL;
    if (!aligned(x, elem_size(dtype)) || !aligned(parts, 8)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::StatsArgs a{x, dtype == VP_BF16, N, V, R, s_o, s_i, 0, nullptr, nullptr, nullptr, nullptr,
                    (cudaStream_t)stream, parts};
    return launched(vp::launch_entropy_fwd(a));
}

vp_status vp_kl_partial(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                        int64_t s_i, int direction, vp_partial *parts, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (direction != VP_KL_REVERSE && direction != VP_KL_FORWARD) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!a || !b || !parts) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(a, es) || !aligned(b, es) || !aligned(parts, 8)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    const bool rev = direction == VP_KL_REVERSE;  // reverse: P = A, Q = B
    vp::KLFwdArgs k{rev ? a : b, rev ? b : a, dtype == VP_BF16, N, V, R, s_o, s_i, nullptr, nullptr, nullptr,
                    (cudaStream_t)stream, parts};
    return launched(vp::launch_kl_fwd(k));
}

namespace {
vp_status check_merge(const vp_partial *parts, int64_t K, int64_t N) {
    if (K < 1 || N < 0 || N > kMaxRowsPerLaunch || K > kMaxRowsPerLaunch / (N > 0 ? N : 1)) return VP_ERR_SHAPE;
    if (N > 0 && !parts) return VP_ERR_NULL;
    if (!aligned(parts, 8)) return VP_ERR_ALIGN;
    return VP_OK;
}
}  // namespace

vp_status vp_logprobs_merge(const vp_partial *parts, int64_t K, int64_t N, float *logp, vp_rowstat *stats,
                            int32_t *err_word, vp_stream stream) {
    vp_status st = check_merge(parts, K, N);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!logp || !stats) return VP_ERR_NULL;
    if (!aligned(logp, 4) || !aligned(stats, 16) || !aligned(err_word, 4)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::MergeArgs a{parts, K, N, logp, stats, nullptr, err_word, (cudaStream_t)stream};
    return launched(vp::launch_logprobs_merge(a));
}

vp_status vp_entropy_merge(const vp_partial *parts, int64_t K, int64_t N, float *H, vp_rowstat *stats,
                           vp_stream stream) {
    vp_status st = check_merge(parts, K, N);
    if (st != VP_OK) return st;
    if (N == 0) return VP_OK;
    if (!H || !stats) return VP_ERR_NULL;
    if (!aligned(H, 4) || !aligned(stats, 16)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    vp::MergeArgs a{parts, K, N, H, stats, nullptr, nullptr, (cudaStream_t)stream};
    return launched(vp::launch_entropy_merge(a));
}

vp_status vp_kl_merge(const vp_partial *parts, int64_t K, int64_t N, int direction, float *kl,
                      vp_rowstat *stats_a, vp_rowstat *stats_b, vp_stream stream) {
    vp_status st = check_merge(parts, K, N);
    if (st != VP_OK) return st;
    if (direction != VP_KL_REVERSE && direction != VP_KL_FORWARD) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!kl || !stats_a || !stats_b) return VP_ERR_NULL;
    if (!aligned(kl, 4) || !aligned(stats_a, 16) || !aligned(stats_b, 16)) return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    const bool rev = direction == VP_KL_REVERSE;
    vp::MergeArgs a{parts, K, N, kl, rev ? (void *)stats_a : (void *)stats_b, rev ? (void *)stats_b : (void *)stats_a,
                    nullptr, (cudaStream_t)stream};
    return launched(vp::launch_kl_merge(a));
}

vp_status vp_kl_bwd(const void *a, const void *b, int dtype, int64_t N, int64_t V, int64_t R, int64_t s_o,
                    int64_t s_i, int direction, const vp_rowstat *stats_a, const vp_rowstat *stats_b,
                    const float *grad_out, void *da, void *db, vp_stream stream) {
    vp_status st = check_rows(dtype, N, V, R, s_o, s_i);
    if (st != VP_OK) return st;
    if (direction != VP_KL_REVERSE && direction != VP_KL_FORWARD) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!da && !db) return VP_ERR_ARG;
    if (!a || !b || !stats_a || !stats_b || !grad_out) return VP_ERR_NULL;
    const size_t es = elem_size(dtype);
    if (!aligned(a, es) || !aligned(b, es) || !aligned(da, es) || !aligned(db, es) || !aligned(stats_a, 16) ||
        !aligned(stats_b, 16) || !aligned(grad_out, 4))
        return VP_ERR_ALIGN;
    if ((st = check_device()) != VP_OK) return st;
    const bool rev = direction == VP_KL_REVERSE;
    vp::KLBwdArgs k{rev ? a : b, rev ? b : a, dtype == VP_BF16, N, V, R, s_o, s_i,
                    rev ? (const void *)stats_a : (const void *)stats_b,
                    rev ? (const void *)stats_b : (const void *)stats_a, grad_out, rev ? da : db, rev ? db : da,
                    (cudaStream_t)stream};
    return launched(vp::launch_kl_bwd(k));
}

size_t vp_linear_logp_workspace_size(int64_t N, int64_t V, int64_t D) {
    (void)D;
    if (N < 0 || V < 1) return 0;
    return vp::linear_workspace_bytes(N, V);
}

vp_status vp_linear_logp_fwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                             int64_t vocab_start, const int64_t *targets, float *logp, vp_rowstat *stats,
                             void *workspace, size_t workspace_bytes, int32_t *err_word, vp_stream stream) {
    if (N < 0 || N > kMaxRowsPerLaunch || V < 1 || V > kMaxV || D < 64 || D % 64 != 0 || D > (1 << 20))
        return VP_ERR_SHAPE;
    if (N == 0) return VP_OK;
    if (!hidden || !weight || !targets || !logp || !stats || !workspace) return VP_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(targets, 8) || !aligned(logp, 4) ||
        !aligned(stats, 16) || !aligned(workspace, 256) || !aligned(err_word, 4))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_workspace_bytes(N, V)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearFwdArgs a{hidden, weight, N, V, D, vocab_start, targets, logp, stats, workspace, err_word,
                        (cudaStream_t)stream};
    return launched(vp::launch_linear_logp_fwd(a));
}

vp_status vp_linear_logp_fwd_noalloc(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                     int64_t vocab_start, const int64_t *targets, float *logp, vp_rowstat *stats,
                                     int32_t *err_word, vp_stream stream) {
    if (N < 0 || N > kMaxRowsPerLaunch || V < 1 || V > kMaxV || D < 64 || D % 64 != 0 || D > (1 << 20))
        return VP_ERR_SHAPE;
    if (vp::linear_workspace_bytes(N, V) > vp::kNoAllocScratchBytes) return VP_ERR_SCRATCH;
    if (N == 0) return VP_OK;
    if (!hidden || !weight || !targets || !logp || !stats) return VP_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(targets, 8) || !aligned(logp, 4) ||
        !aligned(stats, 16) || !aligned(err_word, 4))
        return VP_ERR_ALIGN;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearFwdArgs a{hidden, weight, N, V, D, vocab_start, targets, logp, stats, nullptr, err_word,
                        (cudaStream_t)stream};
    return launched(vp::launch_linear_logp_fwd_noalloc(a));
}

static bool precision_ok(int precision) { return precision == VP_GRAD_EXACT || precision == VP_GRAD_FAST; }

size_t vp_linear_logp_bwd_workspace_size(int64_t N, int64_t V, int64_t D) {
    if (N < 0 || V < 1 || D < 64) return 0;
    return vp::linear_bwd_workspace_bytes(N, V, D);
}

vp_status vp_linear_logp_bwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                             int64_t vocab_start, const int64_t *targets, const vp_rowstat *stats,
                             const float *grad_out, void *dhidden, void *dW, int precision, void *workspace,
                             size_t workspace_bytes, int32_t *err_word, vp_stream stream) {
    if (N < 0 || N > kMaxRowsPerLaunch || V < 1 || V > kMaxV || D < 64 || D % 64 != 0 || D > (1 << 20))
        return VP_ERR_SHAPE;
    if (!dhidden && !dW) return VP_ERR_ARG;
    if (!precision_ok(precision)) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!hidden || !weight || !targets || !stats || !grad_out || !workspace) return VP_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(targets, 8) || !aligned(stats, 16) ||
        !aligned(grad_out, 4) || !aligned(dhidden, 16) || !aligned(dW, 16) || !aligned(workspace, 256) ||
        !aligned(err_word, 4))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_bwd_workspace_bytes(N, V, D)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearBwdArgs a{hidden, weight, N, V, D, vocab_start, targets, stats, grad_out, dhidden, dW, workspace,
                        err_word, (cudaStream_t)stream, precision};
    return launched(vp::launch_linear_logp_bwd(a));
}

static bool linear_dims_ok(int64_t N, int64_t V, int64_t D) {
    return N >= 0 && N <= kMaxRowsPerLaunch && V >= 1 && V <= kMaxV && D >= 64 && D % 64 == 0 && D <= (1 << 20);
}

size_t vp_linear_entropy_workspace_size(int64_t N, int64_t V, int64_t D) {
    if (!linear_dims_ok(N, V, D)) return 0;
    return vp::linear_entropy_workspace_bytes(N, V);
}

vp_status vp_linear_entropy_fwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D, float *H,
                                vp_rowstat *stats, void *workspace, size_t workspace_bytes, vp_stream stream) {
    if (!linear_dims_ok(N, V, D)) return VP_ERR_SHAPE;
    if (N == 0) return VP_OK;
    if (!hidden || !weight || !H || !stats || !workspace) return VP_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(H, 4) || !aligned(stats, 16) ||
        !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_entropy_workspace_bytes(N, V)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearEntArgs a{hidden, weight, N, V, D, H, stats, nullptr, nullptr, nullptr, workspace,
                        (cudaStream_t)stream};
    return launched(vp::launch_linear_entropy_fwd(a));
}

size_t vp_linear_entropy_bwd_workspace_size(int64_t N, int64_t V, int64_t D) {
    if (!linear_dims_ok(N, V, D)) return 0;
    return vp::linear_entropy_bwd_workspace_bytes(N, V, D);
}

vp_status vp_linear_entropy_bwd(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                const vp_rowstat *stats, const float *grad_out, void *dhidden, void *dW,
                                int precision, void *workspace, size_t workspace_bytes, vp_stream stream) {
    if (!linear_dims_ok(N, V, D)) return VP_ERR_SHAPE;
    if (!dhidden && !dW) return VP_ERR_ARG;
    if (!precision_ok(precision)) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!hidden || !weight || !stats || !grad_out || !workspace) return VP_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(stats, 16) || !aligned(grad_out, 4) ||
        !aligned(dhidden, 16) || !aligned(dW, 16) || !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_entropy_bwd_workspace_bytes(N, V, D)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearEntArgs a{hidden, weight, N, V, D, nullptr, const_cast<vp_rowstat *>(stats), grad_out, dhidden, dW,
                        workspace, (cudaStream_t)stream};
    a.precision = precision;
    return launched(vp::launch_linear_entropy_bwd(a));
}

size_t vp_linear_kl_workspace_size(int64_t N, int64_t V) {
    if (!linear_dims_ok(N, V, 64)) return 0;
    return vp::linear_kl_workspace_bytes(N, V);
}

vp_status vp_linear_kl_fwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N, int64_t V,
                           int64_t Da, int64_t Db, int direction, float *kl, vp_rowstat *stats_a,
                           vp_rowstat *stats_b, void *workspace, size_t workspace_bytes, vp_stream stream) {
    if (!linear_dims_ok(N, V, Da) || !linear_dims_ok(N, V, Db)) return VP_ERR_SHAPE;
    if (direction != VP_KL_REVERSE && direction != VP_KL_FORWARD) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!ha || !wa || !hb || !wb || !kl || !stats_a || !stats_b || !workspace) return VP_ERR_NULL;
    if (!aligned(ha, 16) || !aligned(wa, 16) || !aligned(hb, 16) || !aligned(wb, 16) || !aligned(kl, 4) ||
        !aligned(stats_a, 16) || !aligned(stats_b, 16) || !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_kl_workspace_bytes(N, V)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearKLArgs a{ha, wa, hb, wb, N, V, Da, Db, direction, kl, stats_a, stats_b, nullptr,
                       nullptr, nullptr, nullptr, nullptr, workspace, (cudaStream_t)stream};
    return launched(vp::launch_linear_kl_fwd(a));
}

size_t vp_linear_kl_bwd_workspace_size(int64_t N, int64_t V, int64_t Da, int64_t Db) {
    if (!linear_dims_ok(N, V, Da) || !linear_dims_ok(N, V, Db)) return 0;
    return vp::linear_kl_bwd_workspace_bytes(N, V, Da, Db);
}

vp_status vp_linear_kl_bwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N, int64_t V,
                           int64_t Da, int64_t Db, int direction, const vp_rowstat *stats_a,
                           const vp_rowstat *stats_b, const float *grad_out, void *dha, void *dwa, void *dhb,
                           void *dwb, int precision, void *workspace, size_t workspace_bytes, vp_stream stream) {
    if (!linear_dims_ok(N, V, Da) || !linear_dims_ok(N, V, Db)) return VP_ERR_SHAPE;
    if (direction != VP_KL_REVERSE && direction != VP_KL_FORWARD) return VP_ERR_ARG;
    if (!dha && !dwa && !dhb && !dwb) return VP_ERR_ARG;
    if (!precision_ok(precision)) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!ha || !wa || !hb || !wb || !stats_a || !stats_b || !grad_out || !workspace) return VP_ERR_NULL;
    if (!aligned(ha, 16) || !aligned(wa, 16) || !aligned(hb, 16) || !aligned(wb, 16) || !aligned(stats_a, 16) ||
        !aligned(stats_b, 16) || !aligned(grad_out, 4) || !aligned(dha, 16) || !aligned(dwa, 16) ||
        !aligned(dhb, 16) || !aligned(dwb, 16) || !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_kl_bwd_workspace_bytes(N, V, Da, Db)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearKLArgs a{ha, wa, hb, wb, N, V, Da, Db, direction, nullptr,
                       const_cast<vp_rowstat *>(stats_a), const_cast<vp_rowstat *>(stats_b), grad_out,
                       dha, dwa, dhb, dwb, workspace, (cudaStream_t)stream};
    a.precision = precision;
    return launched(vp::launch_linear_kl_bwd(a));
}

static bool beta_ok(double beta) { return beta >= 0.0 && beta <= 1.0; }   // false for NaN

size_t vp_linear_jsd_workspace_size(int64_t N, int64_t V) { return vp_linear_kl_workspace_size(N, V); }

vp_status vp_linear_jsd_fwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N, int64_t V,
                            int64_t Da, int64_t Db, double beta, float *jsd, vp_rowstat *stats_a,
                            vp_rowstat *stats_b, void *workspace, size_t workspace_bytes, vp_stream stream) {
    if (!beta_ok(beta)) return VP_ERR_ARG;
    if (beta == 0.0)
        return vp_linear_kl_fwd(ha, wa, hb, wb, N, V, Da, Db, VP_KL_FORWARD, jsd, stats_a, stats_b, workspace,
                                workspace_bytes, stream);
    if (beta == 1.0)
        return vp_linear_kl_fwd(ha, wa, hb, wb, N, V, Da, Db, VP_KL_REVERSE, jsd, stats_a, stats_b, workspace,
                                workspace_bytes, stream);
    if (!linear_dims_ok(N, V, Da) || !linear_dims_ok(N, V, Db)) return VP_ERR_SHAPE;
    if (N == 0) return VP_OK;
    if (!ha || !wa || !hb || !wb || !jsd || !stats_a || !stats_b || !workspace) return VP_ERR_NULL;
    if (!aligned(ha, 16) || !aligned(wa, 16) || !aligned(hb, 16) || !aligned(wb, 16) || !aligned(jsd, 4) ||
        !aligned(stats_a, 16) || !aligned(stats_b, 16) || !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_kl_workspace_bytes(N, V)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearKLArgs a{ha, wa, hb, wb, N, V, Da, Db, 0, jsd, stats_a, stats_b, nullptr,
                       nullptr, nullptr, nullptr, nullptr, workspace, (cudaStream_t)stream, (float)beta};
    return launched(vp::launch_linear_jsd_fwd(a));
}

size_t vp_linear_jsd_bwd_workspace_size(int64_t N, int64_t V, int64_t Da, int64_t Db) {
    return vp_linear_kl_bwd_workspace_size(N, V, Da, Db);
}

vp_status vp_linear_jsd_bwd(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N, int64_t V,
                            int64_t Da, int64_t Db, double beta, const vp_rowstat *stats_a,
                            const vp_rowstat *stats_b, const float *grad_out, void *dha, void *dwa, void *dhb,
                            void *dwb, int precision, void *workspace, size_t workspace_bytes, vp_stream stream) {
    if (!beta_ok(beta)) return VP_ERR_ARG;
    if (beta == 0.0 || beta == 1.0)
        return vp_linear_kl_bwd(ha, wa, hb, wb, N, V, Da, Db, beta == 0.0 ? VP_KL_FORWARD : VP_KL_REVERSE, stats_a,
                                stats_b, grad_out, dha, dwa, dhb, dwb, precision, workspace, workspace_bytes, stream);
    if (!linear_dims_ok(N, V, Da) || !linear_dims_ok(N, V, Db)) return VP_ERR_SHAPE;
    if (!dha && !dwa && !dhb && !dwb) return VP_ERR_ARG;
    if (!precision_ok(precision)) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!ha || !wa || !hb || !wb || !stats_a || !stats_b || !grad_out || !workspace) return VP_ERR_NULL;
    if (!aligned(ha, 16) || !aligned(wa, 16) || !aligned(hb, 16) || !aligned(wb, 16) || !aligned(stats_a, 16) ||
        !aligned(stats_b, 16) || !aligned(grad_out, 4) || !aligned(dha, 16) || !aligned(dwa, 16) ||
        !aligned(dhb, 16) || !aligned(dwb, 16) || !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_kl_bwd_workspace_bytes(N, V, Da, Db)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearKLArgs a{ha, wa, hb, wb, N, V, Da, Db, 0, nullptr,
                       const_cast<vp_rowstat *>(stats_a), const_cast<vp_rowstat *>(stats_b), grad_out,
                       dha, dwa, dhb, dwb, workspace, (cudaStream_t)stream, (float)beta};
    a.precision = precision;
    return launched(vp::launch_linear_jsd_bwd(a));
}

static vp_status copy_async(void *dst, const void *src, size_t bytes, cudaMemcpyKind kind, vp_stream stream) {
    if (bytes == 0) return VP_OK;
    if (!dst || !src) return VP_ERR_NULL;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    return cudaMemcpyAsync(dst, src, bytes, kind, (cudaStream_t)stream) == cudaSuccess ? VP_OK : VP_ERR_LAUNCH;
}

vp_status vp_upload(void *dst_device, const void *src_host, size_t bytes, vp_stream stream) {
    return copy_async(dst_device, src_host, bytes, cudaMemcpyHostToDevice, stream);
}

vp_status vp_download(void *dst_host, const void *src_device, size_t bytes, vp_stream stream) {
    return copy_async(dst_host, src_device, bytes, cudaMemcpyDeviceToHost, stream);
}

vp_status vp_fault_status(uint32_t *value, int clear) {
    if (!value) return VP_ERR_NULL;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    uint32_t a = 0, b = 0, c = 0;
    if (vp::read_fault(&a, clear != 0) != cudaSuccess || vp::read_linear_logp_fault(&b, clear != 0) != cudaSuccess ||
        vp::read_linear_ent_kl_fault(&c, clear != 0) != cudaSuccess)
        return VP_ERR_LAUNCH;
    *value = a | ((b | c) << 2);
    return VP_OK;
}

vp_status vp_set_row_split(int ctas) { return vp::set_row_split(ctas) ? VP_OK : VP_ERR_ARG; }

int vp_get_row_split(void) { return vp::row_split(); }

const char *vp_status_string(int status) {
    switch (status) {
        case VP_OK: return "ok";
        case VP_ERR_NULL: return "a required pointer is NULL";
        case VP_ERR_SHAPE: return "invalid shape (N, V, R or D)";
        case VP_ERR_DTYPE: return "unknown dtype";
        case VP_ERR_LAYOUT: return "invalid row layout (negative stride)";
        case VP_ERR_ALIGN: return "misaligned pointer";
        case VP_ERR_LAUNCH: return "CUDA launch failed";
        case VP_ERR_ARG: return "invalid argument";
        case VP_ERR_DEVICE: return "no usable sm_103 device";
        case VP_ERR_SCRATCH: return "problem too large for the fixed 24 MiB scratch of the no-allocation entry point";
        default: return "unknown status";
    }
}

int vp_version(void) { return 1; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Vocabulary-sharded fused linear ops: the shard's vp_partial records
// ---------------------------------------------------------------------------
vp_status vp_linear_logp_partial(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                 int64_t vocab_start, const int64_t *targets, vp_partial *parts, void *workspace,
                                 size_t workspace_bytes, vp_stream stream) {
    if (!linear_dims_ok(N, V, D)) return VP_ERR_SHAPE;
    if (N == 0) return VP_OK;
    if (!hidden || !weight || !targets || !parts || !workspace) return VP_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(targets, 8) || !aligned(parts, 8) ||
        !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_workspace_bytes(N, V)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearFwdArgs a{hidden, weight, N, V, D, vocab_start, targets, nullptr, nullptr, workspace, nullptr,
                        (cudaStream_t)stream, parts};
    return launched(vp::launch_linear_logp_fwd(a));
}

vp_status vp_linear_entropy_partial(const void *hidden, const void *weight, int64_t N, int64_t V, int64_t D,
                                    vp_partial *parts, void *workspace, size_t workspace_bytes, vp_stream stream) {
    if (!linear_dims_ok(N, V, D)) return VP_ERR_SHAPE;
    if (N == 0) return VP_OK;
    if (!hidden || !weight || !parts || !workspace) return VP_ERR_NULL;
    if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(parts, 8) || !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_entropy_workspace_bytes(N, V)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearEntArgs a{hidden, weight, N, V, D, nullptr, nullptr, nullptr, nullptr, nullptr, workspace,
                        (cudaStream_t)stream, parts};
    return launched(vp::launch_linear_entropy_fwd(a));
}

vp_status vp_linear_kl_partial(const void *ha, const void *wa, const void *hb, const void *wb, int64_t N, int64_t V,
                               int64_t Da, int64_t Db, int direction, vp_partial *parts, void *workspace,
                               size_t workspace_bytes, vp_stream stream) {
    if (!linear_dims_ok(N, V, Da) || !linear_dims_ok(N, V, Db)) return VP_ERR_SHAPE;
    if (direction != VP_KL_REVERSE && direction != VP_KL_FORWARD) return VP_ERR_ARG;
    if (N == 0) return VP_OK;
    if (!ha || !wa || !hb || !wb || !parts || !workspace) return VP_ERR_NULL;
    if (!aligned(ha, 16) || !aligned(wa, 16) || !aligned(hb, 16) || !aligned(wb, 16) || !aligned(parts, 8) ||
        !aligned(workspace, 256))
        return VP_ERR_ALIGN;
    if (workspace_bytes < vp::linear_kl_workspace_bytes(N, V)) return VP_ERR_ARG;
    vp_status st = check_device();
    if (st != VP_OK) return st;
    vp::LinearKLArgs a{ha, wa, hb, wb, N, V, Da, Db, direction, nullptr, nullptr, nullptr, nullptr,
                       nullptr, nullptr, nullptr, nullptr, workspace, (cudaStream_t)stream, 0.f, parts};
    return launched(vp::launch_linear_kl_fwd(a));
}
