// Internal launchers of the dgsamp kernels (host side); not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dgsamp.h"
#include "loop.cuh"

namespace dg {

int stats_cluster_size(int64_t R, int64_t V);
cudaError_t launch_row_stats(const float *logits, int64_t R, int64_t V, int64_t ldl, float *m, float *lse,
                             float *H, float *kappa, int32_t *argmax, cudaStream_t stream);

// Threads of an acceptance CTA for L_c positions: a power of two >= L_c (at least 32).
int accept_threads(int32_t L_c);
cudaError_t launch_entropy_accept(const float *H, const float *kappa, int32_t n_req, int32_t L_c,
                                  const float *budgets, int32_t min_accept, int32_t *order,
                                  uint8_t *mask, int32_t *n_accepted, cudaStream_t stream,
                                  bool overlap_previous = false, const uint8_t *eligible = nullptr);

// Denoising-loop state after a step (loop.cu): kept tokens, stable-argmax count,
// step count and convergence per request.
cudaError_t launch_loop_update(const int32_t *candidate, const int32_t *argmax, const float *H, const uint8_t *mask,
                               int32_t n_req, int32_t L_c, int32_t stable_steps, float entropy_threshold,
                               int32_t step_limit, int32_t *canvas, uint8_t *eligible, int32_t *prev_argmax,
                               int32_t *stable, int32_t *steps, uint8_t *converged, cudaStream_t stream);

constexpr int kMaxPartials = 16;
cudaError_t launch_sum_partials(const float *const *partials, int32_t T, int64_t R, int64_t d, int64_t ldp,
                                float gamma, float *out, int64_t ldo, cudaStream_t stream);
cudaError_t launch_fill_zero(float *out, int64_t R, int64_t d, int64_t ldo, cudaStream_t stream);

// The embedding table of the product: bf16 entries, or E4M3 codes with one fp32 scale per
// row (W[v, j] = scale[v] * e4m3(Q[v, j])).
enum { kTableBf16 = 0, kTableE4m3 = 1 };
struct EmbedTable {
    int fmt;              // kTableBf16 (W: uint16 bit patterns) or kTableE4m3 (W: uint8 codes)
    const void *W;        // [rows, ldw] entries; row j is vocabulary entry vocab_start + j
    int64_t ldw;          // entries per row
    const float *scale;   // kTableE4m3: [rows] row scales; else NULL
};

// Plan of the split-K soft-embed product for one shape on one device.
struct SoftEmbedPlan {
    int fmt;           // the table format it was made for
    int bn;            // output columns per tile
    int64_t k_begin;   // first vocabulary column read (vocab_start rounded down to a multiple of 4)
    int64_t nkb;       // vocabulary blocks of the product
    int m_tiles, n_tiles, splits;
    size_t workspace_bytes;    // the product and its reduce
    size_t single_pass_bytes;  // the same with the single pass's statistics (launch_soft_embed `single`)
};
struct AcceptSpec;
// Single pass: the product also folds the row statistics (no lse needed before it); they are
// written here after it.  With `accept`, the reduce kernel also runs that acceptance (in extra
// CTAs, on the statistics) and `between` is not called.
struct SinglePassOut {
    float *m, *lse, *H, *kappa;
    int32_t *argmax;
    int32_t *candidate;     // non-NULL: also draw (two-level Gumbel-max from softmax(l / T)); kappa
    uint64_t seed, offset;  // is then -ln p of the drawn token under softmax(l)
    const AcceptSpec *accept;
    // a vocabulary shard in two calls around the ranks' exchange of row summaries:
    // 0 the whole step; 1 the product and the shard's row summaries (shard_state, argmax as
    // vocab_offset + column; the split partials stay in the workspace); 2 the reduce, its scales
    // taken against the full-row lse (`lse`: read, not written)
    int phase;
    float *shard_state;
    int64_t vocab_offset;
    // non-NULL: the denoising-loop update, run by each request's acceptance CTA right after it
    const LoopSpec *loop;
    float temperature;  // T of the draw (0 is taken as 1)
};
bool plan_soft_embed(int64_t R, int64_t vocab_start, int64_t vocab_end, int64_t d, int num_sms,
                     SoftEmbedPlan *plan, int fmt = kTableBf16);
// Workspace bytes a plan needs with a given number of splits.
size_t soft_embed_workspace_bytes(const SoftEmbedPlan &plan, int splits);
// Queues the product, then `between(ctx, stream)` if given (work that may overlap the
// product: the product lets the next kernel on the stream start early, once the kernel
// before it has completed), then the split-K reduce.  overlap_previous: the product may
// start while the kernel queued before it (the row statistics) still runs; it reads lse
// only after that kernel has completed.  On failure *msg names the step.
typedef cudaError_t (*StreamHook)(void *ctx, cudaStream_t stream);
cudaError_t launch_soft_embed(const float *logits, int64_t ldl, const float *lse, int64_t R,
                              int64_t vocab_start, int64_t vocab_end, const EmbedTable &W,
                              int64_t d, float gamma, float *out, int64_t ldo, void *workspace,
                              const SoftEmbedPlan &plan, cudaStream_t stream, const char **msg,
                              StreamHook between = nullptr, void *ctx = nullptr, bool overlap_previous = false,
                              const SinglePassOut *single = nullptr);

int device_sm_count();
size_t workspace_size(int64_t R, int64_t vocab_len, int64_t d, int fmt);

// Per-row E4M3 quantisation of a bf16 table (quantize.cu).
cudaError_t launch_quantize_e4m3(const uint16_t *W, int64_t V, int64_t d, int64_t ldw, uint8_t *Q, int64_t ldq,
                                 float *scale, cudaStream_t stream);

// Gumbel-max candidates and their tempered log-probabilities (row_sample.cu).
cudaError_t launch_row_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature,
                              uint64_t seed, uint64_t offset, int32_t *candidate, float *log_p,
                              cudaStream_t stream);
// Vocabulary-sharded statistics (row_stats.cu): a shard's 16-byte summary per row, and the
// full-row statistics from the summaries of all shards, merged in shard order.
cudaError_t launch_row_stats_partial(const float *logits, int64_t R, int64_t V, int64_t ldl, int64_t vocab_offset,
                                     float *state, cudaStream_t stream);
cudaError_t launch_row_stats_combine(const float *states, int32_t T, int64_t R, float *m, float *lse, float *H,
                                     float *kappa, int32_t *argmax, cudaStream_t stream);

// The same draw fused with the row statistics (one read of the logits); kappa is
// -ln p(candidate) at temperature 1.
cudaError_t launch_row_stats_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature,
                                    uint64_t seed, uint64_t offset, float *m, float *lse, float *H, float *kappa,
                                    int32_t *argmax, int32_t *candidate, float *log_p, cudaStream_t stream);

// One thread waits on a barrier nothing completes and records a timeout after limit_us.
cudaError_t launch_wait_timeout_check(uint32_t limit_us, cudaStream_t stream);

// Shared by the C entry points: the calling thread's error text, fail() sets it and
// returns st; check_embed_args() holds the argument rules of dg_soft_embed.
extern thread_local char t_last_error[512];
dg_status fail(dg_status st, const char *fmt, ...);
dg_status cuda_fail(cudaError_t e, const char *what);
bool aligned16(const void *p);
dg_status check_embed_args(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t s, int64_t e,
                           const uint16_t *W, int64_t rows_pad, int64_t ldw, int64_t d, const float *out,
                           int64_t ldo);

}  // namespace dg
