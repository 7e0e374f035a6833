// The C ABI of libdgsamp: argument checks, status codes and launches.
// Declarations and the contract of every entry point are in include/dgsamp.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cstdint>

#include "accept.cuh"
#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

__device__ unsigned int g_device_error = 0;

thread_local char t_last_error[512] = "";

dg_status fail(dg_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return st;
}

dg_status cuda_fail(cudaError_t e, const char *what) {
    return fail(DG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

dg_status check_stats_args(const float *logits, int64_t R, int64_t V, int64_t ldl) {
    if (R < 0 || V < 1 || ldl < V) return fail(DG_ERR_INVALID_ARG, "row stats: need R >= 0, V >= 1, ldl >= V");
    if (R > 0 && !logits) return fail(DG_ERR_INVALID_ARG, "row stats: logits is NULL");
    if (V > 0x7ffffff0LL || R > (1LL << 28)) return fail(DG_ERR_UNSUPPORTED, "row stats: V or R too large");
    if (R > 0 && (!aligned16(logits) || (ldl & 3)))
        return fail(DG_ERR_UNSUPPORTED, "row stats: logits must be 16-byte aligned with ldl %% 4 == 0");
    return DG_OK;
}

dg_status check_accept_args(const float *H, const float *kappa, int32_t n_req, int32_t L_c, const float *budgets,
                            int32_t min_accept, const int32_t *order, const uint8_t *mask,
                            const int32_t *n_accepted) {
    if (n_req < 0 || L_c < 1 || min_accept < 0)
        return fail(DG_ERR_INVALID_ARG, "accept: need n_req >= 0, L_c >= 1, min_accept >= 0");
    if (L_c > 1024) return fail(DG_ERR_UNSUPPORTED, "accept: L_c = %d is above 1024", L_c);
    if (n_req > 0 && (!H || !kappa || !budgets || !order || !mask || !n_accepted))
        return fail(DG_ERR_INVALID_ARG, "accept: a pointer is NULL");
    return DG_OK;
}

}  // namespace

dg_status check_table_args(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t s, int64_t e,
                           const EmbedTable &tab, int64_t rows_pad, int64_t d, const float *out, int64_t ldo) {
    const void *W = tab.W;
    const int64_t ldw = tab.ldw;
    if (R < 0 || d < 1) return fail(DG_ERR_INVALID_ARG, "soft embed: need R >= 0 and d >= 1");
    if (s < 0 || e < s)
        return fail(DG_ERR_INVALID_ARG, "soft embed: slice [%lld, %lld) is reversed or negative", (long long)s,
                    (long long)e);
    if (e > ldl)
        return fail(DG_ERR_INVALID_ARG, "soft embed: slice end %lld is past ldl %lld", (long long)e, (long long)ldl);
    if (e - s > rows_pad)
        return fail(DG_ERR_INVALID_ARG,
                    "soft embed: the slice has %lld vocabulary entries but the shard only %lld rows",
                    (long long)(e - s), (long long)rows_pad);
    if (ldw < d || ldo < d) return fail(DG_ERR_INVALID_ARG, "soft embed: need ldw >= d and ldo >= d");
    if (R > 0 && (!logits || !lse || !out || (e > s && !W)))
        return fail(DG_ERR_INVALID_ARG, "soft embed: a pointer is NULL");
    if (R > (1LL << 30) || d > (1LL << 30) || e > 0x7fffff00LL)
        return fail(DG_ERR_UNSUPPORTED, "soft embed: a size is too large");
    if (R > 0 && e > s) {
        if (!aligned16(logits) || (ldl & 3))
            return fail(DG_ERR_UNSUPPORTED, "soft embed: logits must be 16-byte aligned with ldl %% 4 == 0");
        if (tab.fmt == kTableBf16 && (!aligned16(W) || (ldw & 7)))
            return fail(DG_ERR_UNSUPPORTED, "soft embed: W must be 16-byte aligned with ldw %% 8 == 0");
        if (tab.fmt == kTableE4m3) {
            if (!aligned16(W) || (ldw & 15))
                return fail(DG_ERR_UNSUPPORTED, "soft embed: Q must be 16-byte aligned with ldq %% 16 == 0");
            if (!tab.scale) return fail(DG_ERR_INVALID_ARG, "soft embed: scale is NULL");
            if (reinterpret_cast<uintptr_t>(tab.scale) & 3)
                return fail(DG_ERR_UNSUPPORTED, "soft embed: scale must be 4-byte aligned");
        }
    }
    return DG_OK;
}

dg_status check_embed_args(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t s, int64_t e,
                           const uint16_t *W, int64_t rows_pad, int64_t ldw, int64_t d, const float *out,
                           int64_t ldo) {
    return check_table_args(logits, ldl, lse, R, s, e, EmbedTable{kTableBf16, W, ldw, nullptr}, rows_pad, d, out, ldo);
}

namespace {

dg_status run_soft_embed(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t s, int64_t e,
                         const EmbedTable &W, int64_t d, float gamma, float *out, int64_t ldo,
                         void *ws, size_t ws_bytes, cudaStream_t stream, StreamHook between = nullptr,
                         void *ctx = nullptr, bool overlap_previous = false,
                         const SinglePassOut *single = nullptr) {
    if (R == 0) return DG_OK;
    if (e == s) {
        cudaError_t err = launch_fill_zero(out, R, d, ldo, stream);
        return err == cudaSuccess ? DG_OK : cuda_fail(err, "soft embed (empty slice)");
    }
    const int sms = device_sm_count();
    if (sms <= 0) return fail(DG_ERR_CUDA, "soft embed: no CUDA device");
    SoftEmbedPlan plan;
    if (!plan_soft_embed(R, s, e, d, sms, &plan, W.fmt))
        return fail(DG_ERR_INVALID_ARG, "soft embed: no plan for shape");
    const size_t need = single ? plan.single_pass_bytes : plan.workspace_bytes;
    if (!ws || ws_bytes < need)
        return fail(DG_ERR_INVALID_ARG, "soft embed: workspace of %zu bytes is below the %zu needed", ws_bytes, need);
    if (!aligned16(ws)) return fail(DG_ERR_UNSUPPORTED, "soft embed: workspace must be 16-byte aligned");
    const char *msg = "soft embed";
    cudaError_t err =
        launch_soft_embed(logits, ldl, lse, R, s, e, W, d, gamma, out, ldo, ws, plan, stream, &msg, between, ctx,
                          overlap_previous, single);
    return err == cudaSuccess ? DG_OK : cuda_fail(err, msg);
}

// The acceptance launch of a step, queued between the soft-embed product and its reduce
// so that it runs on a spare SM while the product streams (it reads only row statistics).
cudaError_t accept_hook(void *ctx, cudaStream_t stream) {
    const AcceptSpec *a = static_cast<const AcceptSpec *>(ctx);
    return launch_entropy_accept(a->H, a->kappa, a->n_req, a->L_c, a->budgets, a->min_accept, a->order, a->mask,
                                 a->n_accepted, stream, /*overlap_previous=*/true, a->eligible);
}

// The denoising-loop state a loop step updates after its acceptance (NULL: a plain step).
struct LoopArgs {
    int32_t stable_steps;
    float entropy_threshold;
    int32_t step_limit;
    float temperature;  // 0: the candidate is the argmax; > 0: drawn at this temperature
    uint64_t seed, offset;
    int32_t *candidate;  // the drawn tokens (temperature > 0)
    int32_t *canvas;
    uint8_t *eligible;
    int32_t *prev_argmax, *stable, *steps;
    uint8_t *converged;
};

dg_status check_loop_args(int32_t n_req, int32_t L_c, int32_t stable_steps, float entropy_threshold,
                          int32_t step_limit, const void *canvas, const void *eligible, const void *prev,
                          const void *stable, const void *steps, const void *converged) {
    if (n_req < 0 || L_c < 1) return fail(DG_ERR_INVALID_ARG, "loop: need n_req >= 0 and L_c >= 1");
    if (L_c > 1024) return fail(DG_ERR_UNSUPPORTED, "loop: L_c = %d is above 1024", L_c);
    if (stable_steps < 0 || step_limit < 1 || entropy_threshold != entropy_threshold)
        return fail(DG_ERR_INVALID_ARG, "loop: need stable_steps >= 0, step_limit >= 1 and a threshold");
    if (n_req > 0 && (!canvas || !eligible || !prev || !stable || !steps || !converged))
        return fail(DG_ERR_INVALID_ARG, "loop: a state pointer is NULL");
    return DG_OK;
}

}  // namespace

// Bytes of workspace for the product and the single-pass step over a slice of vocab_len
// entries of a table of format fmt (a slice that starts off a multiple of 4 reads up to
// one more block).
size_t workspace_size(int64_t R, int64_t vocab_len, int64_t d, int fmt) {
    if (R <= 0 || vocab_len <= 0 || d <= 0) return 0;
    const int sms = device_sm_count();
    SoftEmbedPlan plan, plan2;
    if (!plan_soft_embed(R, 0, vocab_len, d, sms, &plan, fmt)) return 0;
    size_t bytes = plan.single_pass_bytes;
    if (plan_soft_embed(R, 3, vocab_len + 3, d, sms, &plan2, fmt) && plan2.single_pass_bytes > bytes)
        bytes = plan2.single_pass_bytes;
    return bytes;
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < kMaxDevices) {
        const int c = g_sm_count[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace dg

namespace dg {
namespace {

// The two calls of a vocabulary shard's single pass (phase 1: product and row summaries; phase
// 2: the reduce against the full-row lse), over the shard's own logit columns [0, n).
dg_status run_shard_phase(int phase, const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t n,
                          int64_t vocab_offset, const EmbedTable &tab, int64_t rows_pad, int64_t d, float gamma,
                          float *state, float *out, int64_t ldo, void *ws, size_t ws_bytes, cudaStream_t stream) {
    const char *what = phase == 1 ? "shard begin" : "shard end";
    if (n < 1) return fail(DG_ERR_INVALID_ARG, "%s: the shard needs at least one vocabulary entry", what);
    // the first call writes no lse and no E: its row summaries stand in for both pointers here
    dg_status st = phase == 1 ? check_table_args(logits, ldl, state, R, 0, n, tab, rows_pad, d, state, d)
                              : check_table_args(logits, ldl, lse, R, 0, n, tab, rows_pad, d, out, ldo);
    if (st != DG_OK) return st;
    if (phase == 1) {
        if (vocab_offset < 0 || vocab_offset + n > INT32_MAX - 1)
            return fail(DG_ERR_INVALID_ARG, "shard begin: the shard must lie in [0, 2^31 - 1)");
        if (reinterpret_cast<uintptr_t>(state) % 16 != 0)
            return fail(DG_ERR_UNSUPPORTED, "shard begin: state must be 16-byte aligned");
    }
    if (R == 0) return DG_OK;
    const int sms = device_sm_count();
    if (sms <= 0) return fail(DG_ERR_CUDA, "%s: no CUDA device", what);
    SoftEmbedPlan plan;
    if (!plan_soft_embed(R, 0, n, d, sms, &plan, tab.fmt)) return fail(DG_ERR_INVALID_ARG, "%s: no plan for shape", what);
    if (!ws || ws_bytes < plan.single_pass_bytes)
        return fail(DG_ERR_INVALID_ARG, "%s: workspace of %zu bytes is below the %zu needed", what, ws_bytes,
                    plan.single_pass_bytes);
    if (!aligned16(ws)) return fail(DG_ERR_UNSUPPORTED, "%s: workspace must be 16-byte aligned", what);
    SinglePassOut so{};
    so.phase = phase;
    so.shard_state = state;
    so.vocab_offset = vocab_offset;
    so.lse = const_cast<float *>(lse);
    const char *msg = what;
    cudaError_t e = launch_soft_embed(logits, ldl, lse, R, 0, n, tab, d, gamma, out, ldo, ws, plan, stream, &msg,
                                      nullptr, nullptr, false, &so);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, msg);
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" {

int dg_version(void) { return 100; }

const char *dg_last_error(void) { return t_last_error; }

dg_status dg_row_stats(const float *logits, int64_t R, int64_t V, int64_t ldl, float *m, float *lse, float *H,
                       float *kappa, int32_t *argmax, dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_stats_args(logits, R, V, ldl);
    if (st != DG_OK || R == 0) return st;
    cudaError_t e = launch_row_stats(logits, R, V, ldl, m, lse, H, kappa, argmax, (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "row stats launch");
}

dg_status dg_row_stats_partial(const float *logits, int64_t R, int64_t n, int64_t ldl, int64_t vocab_offset,
                               float *state, dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_stats_args(logits, R, n, ldl);
    if (st != DG_OK || R == 0) return st;
    if (vocab_offset < 0 || vocab_offset + n > INT32_MAX - 1)
        return fail(DG_ERR_INVALID_ARG, "row stats partial: the shard must lie in [0, 2^31 - 1)");
    if (!state) return fail(DG_ERR_INVALID_ARG, "row stats partial: state is NULL");
    if (reinterpret_cast<uintptr_t>(state) % 16 != 0)
        return fail(DG_ERR_UNSUPPORTED, "row stats partial: state must be 16-byte aligned");
    cudaError_t e = launch_row_stats_partial(logits, R, n, ldl, vocab_offset, state, (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "row stats partial launch");
}

dg_status dg_row_stats_combine(const float *states, int32_t T, int64_t R, float *m, float *lse, float *H,
                               float *kappa, int32_t *argmax, dg_stream_t stream) {
    t_last_error[0] = 0;
    if (R < 0 || T < 1 || T > 1024) return fail(DG_ERR_INVALID_ARG, "row stats combine: need R >= 0, 1 <= T <= 1024");
    if (R == 0) return DG_OK;
    if (!states) return fail(DG_ERR_INVALID_ARG, "row stats combine: states is NULL");
    if (reinterpret_cast<uintptr_t>(states) % 16 != 0)
        return fail(DG_ERR_UNSUPPORTED, "row stats combine: states must be 16-byte aligned");
    cudaError_t e = launch_row_stats_combine(states, T, R, m, lse, H, kappa, argmax, (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "row stats combine launch");
}

dg_status dg_row_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature, uint64_t seed,
                        uint64_t offset, int32_t *candidate, float *log_p, dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_stats_args(logits, R, V, ldl);
    if (st != DG_OK || R == 0) return st;
    if (!(temperature > 0.0f) || !(temperature < INFINITY))
        return fail(DG_ERR_INVALID_ARG, "row sample: temperature must be positive and finite");
    if (!candidate || !log_p) return fail(DG_ERR_INVALID_ARG, "row sample: an output pointer is NULL");
    cudaError_t e = launch_row_sample(logits, R, V, ldl, temperature, seed, offset, candidate, log_p,
                                      (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "row sample launch");
}

dg_status dg_row_stats_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature,
                              uint64_t seed, uint64_t offset, float *m, float *lse, float *H, float *kappa,
                              int32_t *argmax, int32_t *candidate, float *log_p, dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_stats_args(logits, R, V, ldl);
    if (st != DG_OK || R == 0) return st;
    if (!(temperature > 0.0f) || !(temperature < INFINITY))
        return fail(DG_ERR_INVALID_ARG, "row stats + sample: temperature must be positive and finite");
    if (!candidate) return fail(DG_ERR_INVALID_ARG, "row stats + sample: candidate is NULL");
    cudaError_t e = launch_row_stats_sample(logits, R, V, ldl, temperature, seed, offset, m, lse, H, kappa, argmax,
                                            candidate, log_p, (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "row stats + sample launch");
}

size_t dg_soft_embed_workspace_size(int64_t R, int64_t vocab_len, int64_t d) {
    return workspace_size(R, vocab_len, d, kTableBf16);
}

size_t dg_soft_embed_workspace_size_e4m3(int64_t R, int64_t vocab_len, int64_t d) {
    return workspace_size(R, vocab_len, d, kTableE4m3);
}

dg_status dg_soft_embed(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t vocab_start,
                        int64_t vocab_end, const uint16_t *W_shard, int64_t rows_pad, int64_t ldw, int64_t d,
                        float gamma, float *out, int64_t ldo, void *workspace, size_t workspace_bytes,
                        dg_stream_t stream) {
    t_last_error[0] = 0;
    const EmbedTable tab{kTableBf16, W_shard, ldw, nullptr};
    dg_status st = check_table_args(logits, ldl, lse, R, vocab_start, vocab_end, tab, rows_pad, d, out, ldo);
    if (st != DG_OK) return st;
    return run_soft_embed(logits, ldl, lse, R, vocab_start, vocab_end, tab, d, gamma, out, ldo, workspace,
                          workspace_bytes, (cudaStream_t)stream);
}

dg_status dg_soft_embed_e4m3(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t vocab_start,
                             int64_t vocab_end, const uint8_t *Q_shard, const float *scale_shard, int64_t rows_pad,
                             int64_t ldq, int64_t d, float gamma, float *out, int64_t ldo, void *workspace,
                             size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    const EmbedTable tab{kTableE4m3, Q_shard, ldq, scale_shard};
    dg_status st = check_table_args(logits, ldl, lse, R, vocab_start, vocab_end, tab, rows_pad, d, out, ldo);
    if (st != DG_OK) return st;
    return run_soft_embed(logits, ldl, lse, R, vocab_start, vocab_end, tab, d, gamma, out, ldo, workspace,
                          workspace_bytes, (cudaStream_t)stream);
}

dg_status dg_soft_embed_shard_begin(const float *logits, int64_t ldl, int64_t R, int64_t n, int64_t vocab_offset,
                                    const uint16_t *W_shard, int64_t rows_pad, int64_t ldw, int64_t d, float *state,
                                    void *workspace, size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    return run_shard_phase(1, logits, ldl, nullptr, R, n, vocab_offset, EmbedTable{kTableBf16, W_shard, ldw, nullptr},
                           rows_pad, d, 1.0f, state, nullptr, d, workspace, workspace_bytes, (cudaStream_t)stream);
}

dg_status dg_soft_embed_shard_end(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t n,
                                  const uint16_t *W_shard, int64_t rows_pad, int64_t ldw, int64_t d, float gamma,
                                  float *out, int64_t ldo, void *workspace, size_t workspace_bytes,
                                  dg_stream_t stream) {
    t_last_error[0] = 0;
    return run_shard_phase(2, logits, ldl, lse, R, n, 0, EmbedTable{kTableBf16, W_shard, ldw, nullptr}, rows_pad, d,
                           gamma, nullptr, out, ldo, workspace, workspace_bytes, (cudaStream_t)stream);
}

dg_status dg_soft_embed_shard_begin_e4m3(const float *logits, int64_t ldl, int64_t R, int64_t n, int64_t vocab_offset,
                                         const uint8_t *Q_shard, const float *scale_shard, int64_t rows_pad,
                                         int64_t ldq, int64_t d, float *state, void *workspace,
                                         size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    return run_shard_phase(1, logits, ldl, nullptr, R, n, vocab_offset,
                           EmbedTable{kTableE4m3, Q_shard, ldq, scale_shard}, rows_pad, d, 1.0f, state, nullptr, d,
                           workspace, workspace_bytes, (cudaStream_t)stream);
}

dg_status dg_soft_embed_shard_end_e4m3(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t n,
                                       const uint8_t *Q_shard, const float *scale_shard, int64_t rows_pad,
                                       int64_t ldq, int64_t d, float gamma, float *out, int64_t ldo, void *workspace,
                                       size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    return run_shard_phase(2, logits, ldl, lse, R, n, 0, EmbedTable{kTableE4m3, Q_shard, ldq, scale_shard}, rows_pad,
                           d, gamma, nullptr, out, ldo, workspace, workspace_bytes, (cudaStream_t)stream);
}

dg_status dg_quantize_e4m3(const uint16_t *W, int64_t V, int64_t d, int64_t ldw, uint8_t *Q, int64_t ldq,
                           float *scale, dg_stream_t stream) {
    t_last_error[0] = 0;
    if (V < 0 || d < 1 || ldw < d || ldq < d) return fail(DG_ERR_INVALID_ARG, "quantize: need V >= 0, d >= 1, ldw and ldq >= d");
    if (V == 0) return DG_OK;
    if (!W || !Q || !scale) return fail(DG_ERR_INVALID_ARG, "quantize: a pointer is NULL");
    if (V > (1LL << 31) || d > (1LL << 30)) return fail(DG_ERR_UNSUPPORTED, "quantize: a size is too large");
    if ((reinterpret_cast<uintptr_t>(W) & 3) || (ldw & 1) || (reinterpret_cast<uintptr_t>(Q) & 1) || (ldq & 1))
        return fail(DG_ERR_UNSUPPORTED, "quantize: W must be 4-byte aligned and Q 2-byte aligned, ldw and ldq even");
    cudaError_t e = launch_quantize_e4m3(W, V, d, ldw, Q, ldq, scale, (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "quantize launch");
}

dg_status dg_entropy_accept(const float *H, const float *kappa, int32_t n_req, int32_t L_c, const float *budgets,
                            int32_t min_accept, int32_t *order, uint8_t *mask, int32_t *n_accepted,
                            dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_accept_args(H, kappa, n_req, L_c, budgets, min_accept, order, mask, n_accepted);
    if (st != DG_OK || n_req == 0) return st;
    cudaError_t e = launch_entropy_accept(H, kappa, n_req, L_c, budgets, min_accept, order, mask, n_accepted,
                                          (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "accept launch");
}

dg_status dg_sum_partials(const float *const *partials, int32_t T, int64_t R, int64_t d, int64_t ldp, float gamma,
                          float *out, int64_t ldo, dg_stream_t stream) {
    t_last_error[0] = 0;
    if (T < 1 || T > kMaxPartials) return fail(DG_ERR_INVALID_ARG, "sum partials: need 1 <= T <= %d", kMaxPartials);
    if (R < 0 || d < 1 || ldp < d || ldo < d) return fail(DG_ERR_INVALID_ARG, "sum partials: bad sizes");
    if (R == 0) return DG_OK;
    if (!partials || !out) return fail(DG_ERR_INVALID_ARG, "sum partials: a pointer is NULL");
    for (int t = 0; t < T; ++t)
        if (!partials[t]) return fail(DG_ERR_INVALID_ARG, "sum partials: partials[%d] is NULL", t);
    cudaError_t e = launch_sum_partials(partials, T, R, d, ldp, gamma, out, ldo, (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "sum partials launch");
}

namespace {

// The step reads the logits once (the product folds the row statistics) when the slice is
// the whole vocabulary and the workspace has room, unless the caller asks for two passes.
bool use_single_pass(int64_t R, int64_t V, int64_t vocab_start, int64_t vocab_end, int64_t d, size_t ws_bytes,
                     int fmt, uint32_t flags) {
    if (vocab_start != 0 || vocab_end != V) return false;
    if (flags & DG_STEP_TWO_PASS) return false;
    const int sms = device_sm_count();
    SoftEmbedPlan plan;
    if (sms <= 0 || !plan_soft_embed(R, vocab_start, vocab_end, d, sms, &plan, fmt)) return false;
    return ws_bytes >= plan.single_pass_bytes;
}

// The fused step, optionally restricted to eligible positions and followed by the
// loop-state update (a denoising-loop step).
dg_status run_step(const float *logits, int32_t n_req, int32_t L_c, int64_t V, int64_t ldl, const EmbedTable &W,
                   int64_t vocab_start, int64_t vocab_end, int64_t rows_pad, int64_t d, float gamma,
                   const float *budgets, int32_t min_accept, float *m, float *lse, float *H, float *kappa,
                   int32_t *argmax, int32_t *order, uint8_t *mask, int32_t *n_accepted, float *E, int64_t ldo,
                   void *workspace, size_t workspace_bytes, cudaStream_t s, const LoopArgs *loop, uint32_t flags) {
    if (n_req < 0 || L_c < 1) return fail(DG_ERR_INVALID_ARG, "step: need n_req >= 0 and L_c >= 1");
    if (flags & ~(uint32_t)DG_STEP_TWO_PASS) return fail(DG_ERR_INVALID_ARG, "step: unknown flags 0x%x", flags);
    const int64_t R = (int64_t)n_req * L_c;
    dg_status st = check_stats_args(logits, R, V, ldl);
    if (st != DG_OK) return st;
    st = check_accept_args(H, kappa, n_req, L_c, budgets, min_accept, order, mask, n_accepted);
    if (st != DG_OK) return st;
    if (vocab_end > V)
        return fail(DG_ERR_INVALID_ARG, "step: slice end %lld is past V %lld", (long long)vocab_end, (long long)V);
    st = check_table_args(logits, ldl, lse, R, vocab_start, vocab_end, W, rows_pad, d, E, ldo);
    if (st != DG_OK) return st;
    if (R > 0 && (!m || !lse || !H || !kappa || !argmax)) return fail(DG_ERR_INVALID_ARG, "step: a pointer is NULL");
    const bool sampled = loop && loop->temperature != 0.0f;
    if (loop) {
        st = check_loop_args(n_req, L_c, loop->stable_steps, loop->entropy_threshold, loop->step_limit, loop->canvas,
                             loop->eligible, loop->prev_argmax, loop->stable, loop->steps, loop->converged);
        if (st != DG_OK) return st;
        if (sampled && (!(loop->temperature > 0.0f) || !(loop->temperature < INFINITY)))
            return fail(DG_ERR_INVALID_ARG, "loop step: temperature must be 0 (argmax) or positive and finite");
        if (sampled && R > 0 && !loop->candidate) return fail(DG_ERR_INVALID_ARG, "loop step: candidate is NULL");
    }
    if (R == 0) return DG_OK;
    const uint8_t *eligible = loop ? loop->eligible : nullptr;
    if (use_single_pass(R, V, vocab_start, vocab_end, d, workspace_bytes, W.fmt, flags)) {
        // one read of the logits: the product folds the statistics (and, in a sampling loop
        // step, the draw's first level); the acceptance runs inside the reduce kernel, on the
        // statistics the product's fold gave
        // (and, in a loop step, each request's loop-state update right after its acceptance)
        AcceptSpec acc{H, kappa, budgets, n_req, L_c, min_accept, order, mask, n_accepted, eligible};
        LoopSpec ls{};
        if (loop)
            ls = LoopSpec{sampled ? loop->candidate : argmax, argmax, H, mask, L_c, loop->stable_steps,
                          loop->step_limit, loop->entropy_threshold, loop->canvas, loop->eligible,
                          loop->prev_argmax, loop->stable, loop->steps, loop->converged};
        SinglePassOut so{m, lse, H, kappa, argmax, sampled ? loop->candidate : nullptr,
                         sampled ? loop->seed : 0, sampled ? loop->offset : 0, &acc};
        so.loop = loop ? &ls : nullptr;
        so.temperature = sampled ? loop->temperature : 1.0f;
        return run_soft_embed(logits, ldl, lse, R, vocab_start, vocab_end, W, d, gamma, E, ldo, workspace,
                              workspace_bytes, s, nullptr, nullptr, false, &so);
    }
    cudaError_t e = sampled ? launch_row_stats_sample(logits, R, V, ldl, loop->temperature, loop->seed, loop->offset,
                                                      m, lse, H, kappa, argmax, loop->candidate, nullptr, s)
                            : launch_row_stats(logits, R, V, ldl, m, lse, H, kappa, argmax, s);
    if (e != cudaSuccess) return cuda_fail(e, "step: row stats launch");
    if (vocab_end == vocab_start) {
        e = launch_entropy_accept(H, kappa, n_req, L_c, budgets, min_accept, order, mask, n_accepted, s, false,
                                  eligible);
        if (e != cudaSuccess) return cuda_fail(e, "step: accept launch");
        st = run_soft_embed(logits, ldl, lse, R, vocab_start, vocab_end, W, d, gamma, E, ldo, workspace,
                            workspace_bytes, s);
    } else {
        AcceptSpec acc{H, kappa, budgets, n_req, L_c, min_accept, order, mask, n_accepted, eligible};
        // the product overlaps the tail of the statistics kernel (its W and logits loads do
        // not depend on it), the acceptance overlaps the product
        st = run_soft_embed(logits, ldl, lse, R, vocab_start, vocab_end, W, d, gamma, E, ldo, workspace,
                            workspace_bytes, s, accept_hook, &acc, /*overlap_previous=*/true);
    }
    if (st != DG_OK || !loop) return st;
    e = launch_loop_update(sampled ? loop->candidate : argmax, argmax, H, mask, n_req, L_c, loop->stable_steps,
                           loop->entropy_threshold, loop->step_limit, loop->canvas, loop->eligible,
                           loop->prev_argmax, loop->stable, loop->steps, loop->converged, s);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "step: loop update launch");
}

}  // namespace

dg_status dg_sampler_step(const float *logits, int32_t n_req, int32_t L_c, int64_t V, int64_t ldl, const uint16_t *W,
                          int64_t vocab_start, int64_t vocab_end, int64_t rows_pad, int64_t ldw, int64_t d,
                          float gamma, const float *budgets, int32_t min_accept, float *m, float *lse, float *H,
                          float *kappa, int32_t *argmax, int32_t *order, uint8_t *mask, int32_t *n_accepted, float *E,
                          int64_t ldo, uint32_t flags, void *workspace, size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    return run_step(logits, n_req, L_c, V, ldl, EmbedTable{kTableBf16, W, ldw, nullptr}, vocab_start, vocab_end,
                    rows_pad, d, gamma, budgets, min_accept, m, lse, H, kappa, argmax, order, mask, n_accepted, E,
                    ldo, workspace, workspace_bytes, (cudaStream_t)stream, nullptr, flags);
}

dg_status dg_sampler_step_e4m3(const float *logits, int32_t n_req, int32_t L_c, int64_t V, int64_t ldl,
                               const uint8_t *Q, const float *scale, int64_t vocab_start, int64_t vocab_end,
                               int64_t rows_pad, int64_t ldq, int64_t d, float gamma, const float *budgets,
                               int32_t min_accept, float *m, float *lse, float *H, float *kappa, int32_t *argmax,
                               int32_t *order, uint8_t *mask, int32_t *n_accepted, float *E, int64_t ldo,
                               uint32_t flags, void *workspace, size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    return run_step(logits, n_req, L_c, V, ldl, EmbedTable{kTableE4m3, Q, ldq, scale}, vocab_start, vocab_end,
                    rows_pad, d, gamma, budgets, min_accept, m, lse, H, kappa, argmax, order, mask, n_accepted, E,
                    ldo, workspace, workspace_bytes, (cudaStream_t)stream, nullptr, flags);
}

dg_status dg_sampler_loop_step(const float *logits, int32_t n_req, int32_t L_c, int64_t V, int64_t ldl,
                               const uint16_t *W, int64_t vocab_start, int64_t vocab_end, int64_t rows_pad,
                               int64_t ldw, int64_t d, float gamma, const float *budgets, int32_t min_accept,
                               int32_t stable_steps, float entropy_threshold, int32_t step_limit,
                               float temperature, uint64_t seed, uint64_t offset, float *m, float *lse, float *H,
                               float *kappa, int32_t *argmax, int32_t *candidate, int32_t *order, uint8_t *mask,
                               int32_t *n_accepted, float *E, int64_t ldo, int32_t *canvas, uint8_t *eligible,
                               int32_t *prev_argmax, int32_t *stable, int32_t *steps, uint8_t *converged,
                               uint32_t flags, void *workspace, size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    LoopArgs loop{stable_steps, entropy_threshold, step_limit, temperature, seed, offset, candidate, canvas,
                  eligible, prev_argmax, stable, steps, converged};
    return run_step(logits, n_req, L_c, V, ldl, EmbedTable{kTableBf16, W, ldw, nullptr}, vocab_start, vocab_end,
                    rows_pad, d, gamma, budgets, min_accept, m, lse, H, kappa, argmax, order, mask, n_accepted, E,
                    ldo, workspace, workspace_bytes, (cudaStream_t)stream, &loop, flags);
}

dg_status dg_sampler_loop_step_e4m3(const float *logits, int32_t n_req, int32_t L_c, int64_t V, int64_t ldl,
                                    const uint8_t *Q, const float *scale, int64_t vocab_start, int64_t vocab_end,
                                    int64_t rows_pad, int64_t ldq, int64_t d, float gamma, const float *budgets,
                                    int32_t min_accept, int32_t stable_steps, float entropy_threshold,
                                    int32_t step_limit, float temperature, uint64_t seed, uint64_t offset, float *m,
                                    float *lse, float *H, float *kappa, int32_t *argmax, int32_t *candidate,
                                    int32_t *order, uint8_t *mask, int32_t *n_accepted, float *E, int64_t ldo,
                                    int32_t *canvas, uint8_t *eligible, int32_t *prev_argmax, int32_t *stable,
                                    int32_t *steps, uint8_t *converged, uint32_t flags, void *workspace,
                                    size_t workspace_bytes, dg_stream_t stream) {
    t_last_error[0] = 0;
    LoopArgs loop{stable_steps, entropy_threshold, step_limit, temperature, seed, offset, candidate, canvas,
                  eligible, prev_argmax, stable, steps, converged};
    return run_step(logits, n_req, L_c, V, ldl, EmbedTable{kTableE4m3, Q, ldq, scale}, vocab_start, vocab_end,
                    rows_pad, d, gamma, budgets, min_accept, m, lse, H, kappa, argmax, order, mask, n_accepted, E,
                    ldo, workspace, workspace_bytes, (cudaStream_t)stream, &loop, flags);
}

dg_status dg_entropy_accept_eligible(const float *H, const float *kappa, const uint8_t *eligible, int32_t n_req,
                                     int32_t L_c, const float *budgets, int32_t min_accept, int32_t *order,
                                     uint8_t *mask, int32_t *n_accepted, dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_accept_args(H, kappa, n_req, L_c, budgets, min_accept, order, mask, n_accepted);
    if (st != DG_OK || n_req == 0) return st;
    if (!eligible) return fail(DG_ERR_INVALID_ARG, "accept: eligible is NULL");
    cudaError_t e = launch_entropy_accept(H, kappa, n_req, L_c, budgets, min_accept, order, mask, n_accepted,
                                          (cudaStream_t)stream, false, eligible);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "accept launch");
}

dg_status dg_loop_update(const int32_t *candidate, const int32_t *argmax, const float *H, const uint8_t *mask,
                         int32_t n_req, int32_t L_c, int32_t stable_steps, float entropy_threshold,
                         int32_t step_limit, int32_t *canvas, uint8_t *eligible, int32_t *prev_argmax,
                         int32_t *stable, int32_t *steps, uint8_t *converged, dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_loop_args(n_req, L_c, stable_steps, entropy_threshold, step_limit, canvas, eligible,
                                   prev_argmax, stable, steps, converged);
    if (st != DG_OK || n_req == 0) return st;
    if (!candidate || !argmax || !H || !mask) return fail(DG_ERR_INVALID_ARG, "loop: an input pointer is NULL");
    cudaError_t e = launch_loop_update(candidate, argmax, H, mask, n_req, L_c, stable_steps, entropy_threshold,
                                       step_limit, canvas, eligible, prev_argmax, stable, steps, converged,
                                       (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "loop update launch");
}

dg_status dg_check_wait_timeout(uint32_t limit_us, dg_stream_t stream) {
    t_last_error[0] = 0;
    if (limit_us < 1 || limit_us > 1000000u)
        return fail(DG_ERR_INVALID_ARG, "wait-timeout check: limit of %u us is outside 1 .. 1,000,000", limit_us);
    cudaError_t e = launch_wait_timeout_check(limit_us, (cudaStream_t)stream);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, "wait-timeout check launch");
}

dg_status dg_get_device_status(dg_stream_t stream) {
    t_last_error[0] = 0;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "device status: stream");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e, "device status: read");
    if (word) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e, "device status: clear");
        return fail(DG_ERR_TIMEOUT, "a kernel gave up waiting on a device barrier");
    }
    return DG_OK;
}

}  // extern "C"
