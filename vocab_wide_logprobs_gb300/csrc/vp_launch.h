// vp_launch.h -- internal launcher interface between the C ABI and the kernels.
// Arguments here are already validated by vp_api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vp {

constexpr int VP_ERRBIT_TARGET_ = 1;  // same value as VP_ERRBIT_TARGET in include/vp.h
constexpr int VP_GRAD_EXACT_ = 0;     // same values as VP_GRAD_EXACT / VP_GRAD_FAST in include/vp.h
constexpr int VP_GRAD_FAST_ = 1;

struct StatsArgs {
    const void *x;
    bool bf16;
    int64_t N, V, R, s_o, s_i, vocab_start;
    const int64_t *targets;
    float *out;
    void *stats;  // vp_rowstat [N]
    int32_t *err;
    cudaStream_t stream;
    void *parts = nullptr;  // vp_partial [N]: per-shard records instead of out / stats
    int64_t K = 1;          // ids per row (top-k logprobs: targets [N, K], out [N, K])
};

struct KLFwdArgs {
    const void *p, *q;
    bool bf16;
    int64_t N, V, R, s_o, s_i;
    float *kl;
    void *stats_p, *stats_q;
    cudaStream_t stream;
    void *parts = nullptr;  // vp_partial [N]: per-shard records instead of kl / stats
};

// Merge of K shards' vp_partial records (K * N, shard-major) per row.
struct MergeArgs {
    const void *parts;
    int64_t K, N;
    float *out;
    void *stats_p, *stats_q;  // vp_rowstat [N]; stats_q for KL only
    int32_t *err;
    cudaStream_t stream;
};

// Generalized JSD with interior beta: A is the first argument (p), B the second (q).
struct JsdFwdArgs {
    const void *a, *b;
    bool bf16;
    int64_t N, V, R, s_o, s_i;
    double beta;
    float *jsd;
    void *stats_a, *stats_b;  // vp_rowstat [N] each; c = KL(p || mix) / KL(q || mix)
    cudaStream_t stream;
};

struct JsdBwdArgs {
    const void *a, *b;
    bool bf16;
    int64_t N, V, R, s_o, s_i;
    double beta;
    const void *stats_a, *stats_b;
    const float *g;
    void *da, *db;  // either may be NULL
    cudaStream_t stream;
};

cudaError_t launch_jsd_fwd(const JsdFwdArgs &a);
cudaError_t launch_jsd_fwd_rowwise(const JsdFwdArgs &a);
cudaError_t launch_jsd_bwd(const JsdBwdArgs &a);

cudaError_t launch_logprobs_merge(const MergeArgs &a);
cudaError_t launch_entropy_merge(const MergeArgs &a);
cudaError_t launch_kl_merge(const MergeArgs &a);

struct GradArgs {
    const void *x;
    bool bf16;
    int64_t N, V, R, s_o, s_i, vocab_start;
    const void *stats;
    const float *g;
    const int64_t *targets;
    void *dx;
    int32_t *err;
    cudaStream_t stream;
    int64_t K = 1;          // ids per row (top-k logprobs: targets and g are [N, K])
};

struct KLBwdArgs {
    const void *p, *q;
    bool bf16;
    int64_t N, V, R, s_o, s_i;
    const void *stats_p, *stats_q;
    const float *g;
    void *dp, *dq;
    cudaStream_t stream;
};

struct LinearFwdArgs {
    const void *hidden, *weight;  // bf16 [N, D], [V, D], row-major
    int64_t N, V, D, vocab_start;
    const int64_t *targets;
    float *logp;
    void *stats;      // vp_rowstat [N]
    void *workspace;  // linear_workspace_bytes(N, V)
    int32_t *err;
    cudaStream_t stream;
    void *parts = nullptr;   // vp_partial [N]: the shard's records instead of logp and stats
};

size_t linear_workspace_bytes(int64_t N, int64_t V);

struct LinearBwdArgs {
    const void *hidden, *weight;  // bf16 [N, D], [V, D], row-major
    int64_t N, V, D, vocab_start;
    const int64_t *targets;
    const void *stats;            // vp_rowstat [N] of the forward
    const float *g;               // upstream gradient of logp, fp32 [N]
    void *dhidden, *dW;           // bf16 [N, D], [V, D]; either may be NULL
    void *workspace;              // linear_bwd_workspace_bytes(N, V, D)
    int32_t *err;
    cudaStream_t stream;
    int precision = 0;            // VP_GRAD_EXACT: dz as a bf16 pair hi + lo; VP_GRAD_FAST: dz in bf16
};

size_t linear_bwd_workspace_bytes(int64_t N, int64_t V, int64_t D);
cudaError_t launch_linear_logp_bwd(const LinearBwdArgs &a);

// Fixed scratch of vp_linear_logp_fwd_noalloc (24 MiB, held by every device
// that loads the library, for the life of the process).
constexpr size_t kNoAllocScratchBytes = (size_t)24 << 20;
cudaError_t launch_linear_logp_fwd_noalloc(const LinearFwdArgs &a);
cudaError_t launch_linear_logp_fwd(const LinearFwdArgs &a);
// fault words of the GEMM kernels, one per translation unit
cudaError_t read_linear_logp_fault(uint32_t *value, bool clear);
cudaError_t read_linear_ent_kl_fault(uint32_t *value, bool clear);

// Fused linear entropy: model (hidden [N, D], weight [V, D]), bf16 row-major.
struct LinearEntArgs {
    const void *hidden, *weight;
    int64_t N, V, D;
    float *H;                     // forward output, fp32 [N]
    void *stats;                  // vp_rowstat [N]: written by the forward, read by the backward
    const float *g;               // backward: upstream gradient of H, fp32 [N]
    void *dhidden, *dW;           // backward outputs, bf16; either may be NULL
    void *workspace;
    cudaStream_t stream;
    void *parts = nullptr;        // forward: vp_partial [N], the shard's records instead of H and stats
    int precision = 0;            // backward: VP_GRAD_EXACT or VP_GRAD_FAST (as LinearBwdArgs)
};

size_t linear_entropy_workspace_bytes(int64_t N, int64_t V);
size_t linear_entropy_bwd_workspace_bytes(int64_t N, int64_t V, int64_t D);
cudaError_t launch_linear_entropy_fwd(const LinearEntArgs &a);
cudaError_t launch_linear_entropy_bwd(const LinearEntArgs &a);

// Fused linear KL between model A (ha [N, Da], wa [V, Da]) and model B (hb [N, Db],
// wb [V, Db]); reverse = KL(A||B), forward = KL(B||A).
struct LinearKLArgs {
    const void *ha, *wa, *hb, *wb;
    int64_t N, V, Da, Db;
    int direction;
    float *kl;                    // forward output, fp32 [N]
    void *stats_a, *stats_b;      // vp_rowstat [N] each
    const float *g;               // backward: upstream gradient of KL, fp32 [N]
    void *dha, *dwa, *dhb, *dwb;  // backward outputs, bf16; any may be NULL (not all)
    void *workspace;
    cudaStream_t stream;
    float beta = 0.f;             // generalized JSD: 0 < beta < 1 (the KL calls at 0 and 1)
    void *parts = nullptr;        // KL forward: vp_partial [N], the shard's records instead of KL and stats
    int precision = 0;            // backward: VP_GRAD_EXACT or VP_GRAD_FAST (as LinearBwdArgs)
};

size_t linear_kl_workspace_bytes(int64_t N, int64_t V);
size_t linear_kl_bwd_workspace_bytes(int64_t N, int64_t V, int64_t Da, int64_t Db);
cudaError_t launch_linear_kl_fwd(const LinearKLArgs &a);
cudaError_t launch_linear_kl_bwd(const LinearKLArgs &a);
// Fused linear generalized JSD, interior beta (kl = the JSD output)
cudaError_t launch_linear_jsd_fwd(const LinearKLArgs &a);
cudaError_t launch_linear_jsd_bwd(const LinearKLArgs &a);

cudaError_t launch_logprobs_fwd(const StatsArgs &a);
cudaError_t launch_entropy_fwd(const StatsArgs &a);
cudaError_t launch_logprobs_topk_fwd(const StatsArgs &a);
cudaError_t launch_logprobs_topk_bwd(const GradArgs &a);
cudaError_t launch_kl_fwd(const KLFwdArgs &a);
cudaError_t launch_kl_fwd_rowwise(const KLFwdArgs &a);
cudaError_t read_fault(uint32_t *value, bool clear);
bool set_row_split(int ctas);   // 1 or 2 CTAs per row in the forward scans; false for other values
int row_split();
cudaError_t launch_logprobs_bwd(const GradArgs &a);
cudaError_t launch_entropy_bwd(const GradArgs &a);
cudaError_t launch_kl_bwd(const KLBwdArgs &a);

}  // namespace vp
