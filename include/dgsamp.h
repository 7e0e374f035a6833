/*
 * dgsamp: the DiffusionGemma denoising-sampler step on one NVIDIA GB300 (sm_103a).
 *
 * One sampler step, per canvas position (row) of logits over the full vocabulary:
 *   - softmax statistics: max, log-sum-exp, entropy, argmax candidate, confidence;
 *   - entropy-bound acceptance per request: positions ordered from most to least
 *     confident, accepted until the running entropy would pass the budget;
 *   - the self-conditioning soft embedding E = gamma * softmax(logits)[:, s:e] @ W_shard,
 *     the probability-weighted mean of the token-embedding rows over a vocabulary slice.
 *
 * Sources (the pages this library restates):
 *   [P1] calvarado04.com, post on the vLLM change that makes DiffusionGemma
 *        self-conditioning work under tensor parallelism: eq. e^sc (the expected
 *        embedding p_i W), "The fix" (the vocabulary-partition identity, the sliced
 *        product, the sum over ranks, gamma applied after it, org_vocab_start/end
 *        bounds that keep padded shard rows out), "Why not just all-gather the weights".
 *   [P2] agentlenshq.com, "DiffusionGemma: vLLMでネイティブにサポートされた初のDiffusion LLM",
 *        section "サンプリングループとエントロピー境界デノイジング" (candidates at every
 *        position, the entropy-bound acceptance rule) and "安定性のための自己条件付け"
 *        (the full softmax distribution feeds the probability-weighted mean embedding).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller unless stated otherwise.  The
 *     library never allocates device memory, never frees, and never synchronises
 *     inside a call (dg_get_device_status is the one exception and says so).
 *   - Work is queued asynchronously on `stream` (NULL = the legacy default stream);
 *     outputs are valid once the stream has reached the call.
 *   - Matrices are row-major with a leading dimension (elements between rows).
 *   - Logits are fp32; the embedding table is bfloat16, passed as its 16-bit patterns.
 *   - Arguments are checked on the host before any launch: a bad argument returns
 *     DG_ERR_INVALID_ARG or DG_ERR_UNSUPPORTED and queues nothing.  A CUDA launch
 *     error returns DG_ERR_CUDA.  dg_last_error() describes the last failure of the
 *     calling thread.
 *   - A kernel that waits on an in-kernel barrier gives up after about a second,
 *     records DG_ERR_TIMEOUT in a device word and returns; dg_get_device_status()
 *     reports and clears it.
 */
#ifndef DGSAMP_H
#define DGSAMP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st *dg_stream_t;

typedef enum dg_status {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent bounds */
    DG_ERR_UNSUPPORTED = 2,  /* well-formed but outside what the kernels handle (alignment, L_c > 1024) */
    DG_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    DG_ERR_TIMEOUT = 4       /* a device-side wait gave up (reported by dg_get_device_status) */
} dg_status;

/*
 * Options of the sampler-step calls (dg_sampler_step, dg_sampler_loop_step and their 8-bit
 * table forms), OR-ed into their `flags` argument.  Any other bit is DG_ERR_INVALID_ARG.
 *   DG_STEP_TWO_PASS  run the row-statistics pass before the product even when the slice is
 *                     the whole vocabulary (the logits are then read twice; the single pass
 *                     is the default there).  Results agree with the single pass within the
 *                     stated tolerances; the flag exists to compare the two and to keep the
 *                     two-pass workspace size.
 */
typedef enum dg_step_flags {
    DG_STEP_DEFAULT = 0,
    DG_STEP_TWO_PASS = 1
} dg_step_flags;

/* Library version, major*10000 + minor*100 + patch. */
int dg_version(void);

/* Text of the last failure on the calling thread ("" if none).  Owned by the library. */
const char *dg_last_error(void);

/*
 * Row statistics ([P1] eq. e^sc: p_i is a softmax over all V entries; [P2] sampling loop:
 * a candidate and an entropy at every position).
 *
 *   logits  [R, ldl] fp32, ldl >= V.  Row i holds l_{i,0..V-1}.
 *   m       [R] fp32   m_i = max_v l_{i,v}
 *   lse     [R] fp32   lse_i = m_i + ln Z_i,  Z_i = sum_v exp(l_{i,v} - m_i)
 *   H       [R] fp32   entropy -sum_v p ln p in nats, p_{i,v} = exp(l_{i,v} - lse_i)
 *   kappa   [R] fp32   -ln(confidence) = ln Z_i, where confidence = p_{i,argmax};
 *                      computed as log1p of the sum over the non-argmax entries, so
 *                      rows near one-hot keep distinct values (small kappa = confident)
 *   argmax  [R] int32  the smallest index attaining m_i (the candidate token)
 * Any output pointer may be NULL to skip it.
 * -inf logits are allowed (masked vocabulary: probability 0).  A row that is all
 * -inf gives NaN statistics and argmax 0.  NaN logits are undefined.
 * Requires: logits 16-byte aligned, ldl % 4 == 0 (else DG_ERR_UNSUPPORTED); V >= 1.
 * R == 0 queues nothing.
 */
dg_status dg_row_stats(const float *logits, int64_t R, int64_t V, int64_t ldl,
                       float *m, float *lse, float *H, float *kappa, int32_t *argmax,
                       dg_stream_t stream);

/*
 * Bytes of device workspace dg_soft_embed (and dg_sampler_step) needs for R rows, a
 * vocabulary slice of vocab_len entries and hidden size d on the current device.
 * Returns 0 for an invalid shape or when no device is present.
 */
size_t dg_soft_embed_workspace_size(int64_t R, int64_t vocab_len, int64_t d);

/*
 * Self-conditioning soft embedding over the vocabulary slice [vocab_start, vocab_end)
 * ([P1] eq. e^sc and "The fix": S = P[:, s:e] W_shard[0:e-s], E = gamma * S).
 *
 *   logits     [R, ldl] fp32, the FULL-width logits (columns [vocab_start, vocab_end) are read)
 *   lse        [R] fp32, the full-vocabulary log-sum-exp from dg_row_stats.  The
 *              probabilities are exp(l - lse): never renormalised inside the slice.
 *   W_shard    [rows_pad, ldw] bf16 bit patterns; row j is vocabulary entry vocab_start + j.
 *              Only rows [0, vocab_end - vocab_start) are read: padding rows after
 *              them are never touched (they may hold anything, NaN included).
 *   gamma      the normaliser, applied once after the sum (pass 1 for a partial that
 *              will be summed with other slices first)
 *   out        [R, ldo] fp32 result E
 *   workspace  device scratch of at least dg_soft_embed_workspace_size(R, e - s, d)
 *              bytes, 16-byte aligned, owned by the caller; its contents on entry do
 *              not matter.
 * The probabilities are rounded to bfloat16 before the product (the pages cast them
 * to the embedding dtype); the product accumulates in fp32 and the split-K partial
 * sums are added in a fixed order, so the result is bitwise reproducible.
 * Errors: vocab_end - vocab_start > rows_pad, a negative or reversed slice, or a
 * slice past ldl are DG_ERR_INVALID_ARG (the contraction-length mismatch the pages
 * report becomes an error instead of a crash).  logits/W_shard not 16-byte aligned,
 * ldl % 4 != 0 or ldw % 8 != 0 are DG_ERR_UNSUPPORTED.  An empty slice writes zeros.
 */
dg_status dg_soft_embed(const float *logits, int64_t ldl, const float *lse, int64_t R,
                        int64_t vocab_start, int64_t vocab_end,
                        const uint16_t *W_shard, int64_t rows_pad, int64_t ldw, int64_t d,
                        float gamma, float *out, int64_t ldo,
                        void *workspace, size_t workspace_bytes, dg_stream_t stream);

/*
 * dg_soft_embed for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call: it exists for code that is handed only its input and
 * output buffers (a plugin inside another framework's memory pool, a server under
 * a fixed memory budget that must not allocate once it is running) and so cannot
 * supply the workspace dg_soft_embed asks for.
 *
 * Same arguments, results and errors as dg_soft_embed, without the workspace: the
 * split-K partial tiles go to a 16 MiB array compiled into the library, which every
 * GPU that loads the library holds until the process exits.  The call allocates
 * and frees nothing.  One vocabulary split's partial tiles take
 *     ceil(R / 256) * 256  x  ceil(d / 1024) * 1024  x  4 bytes
 * (rows in whole 256-row tiles, columns in whole pairs of 512-column tiles); a shape for which
 * that exceeds 16 MiB (16,777,216 bytes) returns DG_ERR_UNSUPPORTED: R = 1024 at d = 2816
 * (12 MiB) fits, R = 1100 (padded to 1280 rows, 15 MiB) fits, R = 1400 does not.  When
 * several splits do not fit, the call uses as many as fit.  Results match dg_soft_embed
 * within the soft-embedding tolerance; the number of splits (hence the order of the
 * additions) may differ.
 * The array is shared by every call on a device and keeps the last call's data;
 * calls whose kernels may overlap on the GPU race on it, so order them on one
 * stream.  The first call on each device, and the first after the device's context
 * was created anew (a device reset), looks up the array's device address with that
 * device current: make those calls before any stream capture.
 */
dg_status dg_soft_embed_no_alloc(const float *logits, int64_t ldl, const float *lse, int64_t R,
                                 int64_t vocab_start, int64_t vocab_end,
                                 const uint16_t *W_shard, int64_t rows_pad, int64_t ldw, int64_t d,
                                 float gamma, float *out, int64_t ldo, dg_stream_t stream);

/*
 * Entropy-bound acceptance ([P2] sampling loop: tokens are kept from most to least
 * confident until the cumulative entropy would exceed a fixed budget).
 *
 *   H, kappa    [n_req * L_c] fp32 from dg_row_stats; rows q*L_c .. q*L_c+L_c-1 are request q
 *   budgets     [n_req] fp32, nats
 *   min_accept  accept at least min(min_accept, L_c) positions per request (0 = the literal rule)
 *   order       [n_req * L_c] int32: order[q*L_c + j] = the position (0..L_c-1) that is
 *               j-th most confident (kappa ascending; equal kappa: lower position first)
 *   mask        [n_req * L_c] uint8: 1 where the position is accepted
 *   n_accepted  [n_req] int32: n = max{k : H[order_1] + ... + H[order_k] <= B_q}, taken
 *               as a prefix (the first position that would pass the budget stops it),
 *               then raised to min_accept.  The running sum is kept in fp64.
 * Requires 1 <= L_c <= 1024 (else DG_ERR_UNSUPPORTED), n_req >= 0, min_accept >= 0.
 * A position with NaN statistics (an all -inf row) sorts last and stops the running sum.
 */
dg_status dg_entropy_accept(const float *H, const float *kappa, int32_t n_req, int32_t L_c,
                            const float *budgets, int32_t min_accept,
                            int32_t *order, uint8_t *mask, int32_t *n_accepted,
                            dg_stream_t stream);

/*
 * Sum of per-slice partial products on one device: out = gamma * (S_0 + ... + S_{T-1}),
 * added in index order in fp32 ([P1] "The fix": E = gamma * sum_r S^(r); here the T
 * partials sit on one GPU, so the sum is a kernel, not a collective).
 *
 *   partials  HOST array of T device pointers, each [R, ldp] fp32
 *   out       [R, ldo] fp32 (may alias partials[0] only if ldo == ldp)
 * Requires 1 <= T <= 16.
 */
dg_status dg_sum_partials(const float *const *partials, int32_t T, int64_t R, int64_t d,
                          int64_t ldp, float gamma, float *out, int64_t ldo,
                          dg_stream_t stream);

/*
 * One fused sampler step on one stream: row statistics, then acceptance and the soft
 * embedding over the slice [vocab_start, vocab_end) (pass 0 and V for the whole
 * vocabulary, W then being the full table with rows_pad >= V).
 *
 *   logits [n_req*L_c, ldl] fp32; W [rows_pad, ldw] bf16 bits; budgets [n_req] fp32
 *   outputs: m, lse, H, kappa [R] fp32; argmax [R] int32; order [R] int32; mask [R] uint8;
 *            n_accepted [n_req] int32; E [R, ldo] fp32
 *   workspace  >= dg_soft_embed_workspace_size(R, vocab_end - vocab_start, d) bytes
 * All output pointers are required.  The argument rules of the three calls above apply.
 *
 * When the slice is the whole vocabulary (vocab_start == 0, vocab_end == V) and the
 * workspace is that size, the step reads the logits once: each vocabulary split of the
 * product takes its probabilities against a per-row reference c (the largest of the
 * split's first 32 entries), exp(l - c), while it folds the row statistics; the split
 * summaries then give the statistics (as dg_row_stats, up to the order of the fp32
 * additions) and each split's partial is scaled by exp(c - lse) in the reduce.  A
 * (split, row) whose probabilities against c could overflow (their sum above e^82, or the
 * split's maximum 64 nats below c) is recomputed against lse on the CUDA cores (exact,
 * slow, rare: one-hot rows).  E then equals the two-pass result up
 * to the bf16 rounding of different probabilities.  flags = DG_STEP_TWO_PASS runs the
 * statistics pass before the product instead (a workspace of the two-pass size is enough
 * then).
 */
dg_status dg_sampler_step(const float *logits, int32_t n_req, int32_t L_c, int64_t V, int64_t ldl,
                          const uint16_t *W, int64_t vocab_start, int64_t vocab_end,
                          int64_t rows_pad, int64_t ldw, int64_t d, float gamma,
                          const float *budgets, int32_t min_accept,
                          float *m, float *lse, float *H, float *kappa, int32_t *argmax,
                          int32_t *order, uint8_t *mask, int32_t *n_accepted,
                          float *E, int64_t ldo, uint32_t flags,
                          void *workspace, size_t workspace_bytes, dg_stream_t stream);

/*
 * Synchronises `stream`, then reports (and clears) the device-side error word:
 * DG_ERR_TIMEOUT if a kernel gave up waiting since the last call, DG_ERR_CUDA if
 * the stream reports a CUDA error, else DG_OK.  This call blocks the host.
 */
dg_status dg_get_device_status(dg_stream_t stream);

/*
 * Vocabulary-sharded row statistics ([P1] "The fix": the vocabulary is split into
 * contiguous ranges, one per rank, while the softmax stays over all V entries).  A rank
 * holding the logit columns [vocab_offset, vocab_offset + n) summarises each row in 16
 * bytes; the summaries of all shards, gathered in shard order, give dg_row_stats'
 * statistics of the whole row.
 *
 * dg_row_stats_partial:
 *   logits  [R, ldl] fp32, the shard's n columns (layout rules of dg_row_stats with V = n)
 *   state   [R] x 16 bytes, 16-byte aligned: per row {m fp32, a int32, rest fp32, t fp32}
 *           m = max over the shard, a = vocab_offset + the first column attaining it
 *           (2^31 - 1 if the shard row has no finite logit), rest = sum over the shard's
 *           other entries of exp(l - m), t = sum over the shard of exp(l - m)(l - m)
 *   Requires 0 <= vocab_offset and vocab_offset + n < 2^31 - 1.
 * dg_row_stats_combine:
 *   states  [T][R] summaries (the shards' arrays one after another, shard order =
 *           vocabulary order), 1 <= T <= 1024, 16-byte aligned
 *   m, lse, H, kappa [R] fp32, argmax [R] int32: as dg_row_stats (each may be NULL);
 *   the maxima are merged in shard order, so a maximum tied across shards takes the
 *   lowest index.  The result equals dg_row_stats of the whole row up to the order of
 *   the fp32 additions.
 * Both asynchronous; R == 0 queues nothing.
 */
dg_status dg_row_stats_partial(const float *logits, int64_t R, int64_t n, int64_t ldl,
                               int64_t vocab_offset, float *state, dg_stream_t stream);
dg_status dg_row_stats_combine(const float *states, int32_t T, int64_t R, float *m, float *lse,
                               float *H, float *kappa, int32_t *argmax, dg_stream_t stream);

/*
 * A vocabulary shard's soft embedding in one read of its logits ([P1] "The fix": each rank
 * holds the logit columns and the W rows of one contiguous vocabulary range; the softmax is
 * over all V entries).  Two calls around the ranks' exchange of row summaries:
 *
 *   1. dg_soft_embed_shard_begin: the product over the shard's columns [0, n) with
 *      exp(l - c) against a per-row, per-split reference c, folding the row statistics on
 *      the way; writes the shard's 16-byte row summaries `state` in dg_row_stats_partial's
 *      format (argmax = vocab_offset + column) and keeps the split partials and references
 *      in `workspace`.
 *   2. (the caller gathers every shard's `state` in shard order and runs
 *      dg_row_stats_combine: the full-row m, lse, H, kappa, argmax)
 *   3. dg_soft_embed_shard_end: with that full-row `lse`, scales each split's partial by
 *      exp(c - lse), recomputes on the CUDA cores the rare (split, row) pairs whose
 *      probabilities against c could overflow (as dg_sampler_step's single pass does), adds
 *      the splits in a fixed order and writes out = gamma * E_shard.
 *
 * The shard's E then equals dg_soft_embed over the same columns with the full-row lse, up
 * to the bf16 rounding of different probabilities (exp(l - c) scaled afterwards instead of
 * exp(l - lse)).  Both calls take the same logits, W_shard, R, n and d, and the same
 * workspace of at least dg_soft_embed_workspace_size(R, n, d) bytes (the _e4m3 forms:
 * dg_soft_embed_workspace_size_e4m3), which must not be used for anything else in between.
 *   logits   [R, ldl] fp32, the shard's n columns (the layout rules of dg_soft_embed)
 *   W_shard  [rows_pad >= n, ldw] bf16 bits; the _e4m3 forms: Q_shard [rows_pad, ldq] E4M3
 *            codes and scale_shard [rows_pad] fp32 row scales (as dg_soft_embed_e4m3)
 *   state    [R] x 16 bytes, 16-byte aligned (begin)
 *   lse      [R] fp32, the full-row log-sum-exp (end; NaN for a row without a distribution,
 *            whose E is then NaN)
 * Errors: n < 1, or the argument rules of dg_soft_embed and dg_row_stats_partial.
 * Asynchronous; R == 0 queues nothing.
 */
dg_status dg_soft_embed_shard_begin(const float *logits, int64_t ldl, int64_t R, int64_t n,
                                    int64_t vocab_offset, const uint16_t *W_shard, int64_t rows_pad,
                                    int64_t ldw, int64_t d, float *state, void *workspace,
                                    size_t workspace_bytes, dg_stream_t stream);
dg_status dg_soft_embed_shard_end(const float *logits, int64_t ldl, const float *lse, int64_t R,
                                  int64_t n, const uint16_t *W_shard, int64_t rows_pad, int64_t ldw,
                                  int64_t d, float gamma, float *out, int64_t ldo, void *workspace,
                                  size_t workspace_bytes, dg_stream_t stream);
dg_status dg_soft_embed_shard_begin_e4m3(const float *logits, int64_t ldl, int64_t R, int64_t n,
                                         int64_t vocab_offset, const uint8_t *Q_shard,
                                         const float *scale_shard, int64_t rows_pad, int64_t ldq,
                                         int64_t d, float *state, void *workspace,
                                         size_t workspace_bytes, dg_stream_t stream);
dg_status dg_soft_embed_shard_end_e4m3(const float *logits, int64_t ldl, const float *lse, int64_t R,
                                       int64_t n, const uint8_t *Q_shard, const float *scale_shard,
                                       int64_t rows_pad, int64_t ldq, int64_t d, float gamma,
                                       float *out, int64_t ldo, void *workspace,
                                       size_t workspace_bytes, dg_stream_t stream);

/*
 * Stochastic candidates ([P2] sampling loop: candidate tokens are sampled at every
 * position).  For each row i, a categorical draw from softmax(l_i / temperature), taken
 * as a two-level Gumbel-max (an exact categorical sampler): with z = l_i / temperature,
 * groups of 16 consecutive entries g = v / 16 and G(u) = -ln(-ln u),
 *   g* = argmax_g (logsumexp_{v in g} z_v + G(u_{i,g}))          (lowest g on ties),
 *   candidate_i = argmax_{v in g*} (z_v + G(u_{i,v}))           (lowest v on ties),
 * with uniforms from Philox4x32-10 (Salmon et al., SC 2011), key (seed mod 2^32,
 * seed / 2^32): entry v of row i uses word v % 4 of the block with counter
 * (v / 4, i, offset mod 2^32, offset / 2^32), group g word g % 4 of the block with counter
 * (2^31 + g / 4, i, offset mod 2^32, offset / 2^32), and u = ((word >> 9) + 1/2) * 2^-23.
 * The same (seed, offset) gives the same draws; a sampling loop advances `offset` once
 * per step.
 *
 *   logits     [R, ldl] fp32, ldl >= V (as dg_row_stats; the padding columns up to the next
 *              multiple of 4 are read and ignored)
 *   candidate  [R] int32  the drawn token
 *   log_p      [R] fp32   ln of its probability under softmax(l_i / temperature)
 * -inf entries are never drawn; a row that is all -inf gives candidate 0 and NaN log_p.
 * Requires: temperature > 0 and finite (else DG_ERR_INVALID_ARG); the layout rules of
 * dg_row_stats.  R == 0 queues nothing.
 */
dg_status dg_row_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature,
                        uint64_t seed, uint64_t offset, int32_t *candidate, float *log_p,
                        dg_stream_t stream);

/*
 * Diagnostic of the timeout path (no counterpart on the pages): queues on `stream` one
 * thread that waits on a device barrier nothing ever completes, gives up after
 * `limit_us` microseconds (1 .. 1,000,000) and records the timeout exactly as the
 * product's bounded waits do.  The next dg_get_device_status() then returns
 * DG_ERR_TIMEOUT, and the CUDA context stays usable.  DG_ERR_INVALID_ARG for a limit
 * outside the range; DG_ERR_CUDA if the launch fails.  Asynchronous.
 */
dg_status dg_check_wait_timeout(uint32_t limit_us, dg_stream_t stream);

/*
 * Entropy-bound acceptance over the positions still open ([P2] sampling loop: kept
 * tokens stay kept while the rest of the canvas is resampled).  As dg_entropy_accept,
 * restricted to the positions with eligible[q*L_c + j] != 0:
 *   order  the eligible positions from most to least confident (kappa ascending, equal
 *          kappa: lower position first, NaN statistics last among them), then the
 *          ineligible positions in position order;
 *   the running entropy sum runs over the eligible positions only; min_accept is
 *          capped at the number eligible; an ineligible position is never accepted.
 *   eligible  [n_req * L_c] uint8, required when n_req > 0.
 * Argument rules and errors as dg_entropy_accept.
 */
dg_status dg_entropy_accept_eligible(const float *H, const float *kappa, const uint8_t *eligible,
                                     int32_t n_req, int32_t L_c, const float *budgets,
                                     int32_t min_accept, int32_t *order, uint8_t *mask,
                                     int32_t *n_accepted, dg_stream_t stream);

/*
 * Row statistics and a stochastic candidate in one read of the logits ([P2] sampling
 * loop: candidates are sampled at every position, and kept from most to least
 * confident).  m and argmax are those of dg_row_stats, lse and H too up to the order of
 * the fp32 additions; candidate and log_p are those of dg_row_sample with the same
 * (temperature, seed, offset), bit for bit; and
 *   kappa[i] = -ln p_i(candidate_i) under the untempered softmax: ln Z_i (dg_row_stats'
 *              kappa) when the candidate is the argmax, (m_i - l_{i,c}) + ln Z_i otherwise,
 * the confidence by which a sampling loop orders its positions.
 *   candidate  required; m, lse, H, kappa, argmax, log_p may each be NULL (not written).
 * Requires: temperature > 0 and finite (else DG_ERR_INVALID_ARG); the layout rules of
 * dg_row_stats.  R == 0 queues nothing.
 */
dg_status dg_row_stats_sample(const float *logits, int64_t R, int64_t V, int64_t ldl,
                              float temperature, uint64_t seed, uint64_t offset,
                              float *m, float *lse, float *H, float *kappa, int32_t *argmax,
                              int32_t *candidate, float *log_p, dg_stream_t stream);

/*
 * Denoising-loop state after one step ([P2] sampling loop: accepted tokens are kept; a
 * canvas has converged when its argmax predictions have been stable for several steps
 * and the mean entropy per token is below a threshold, or when the step limit is
 * reached).  Per request q, one CTA:
 *   canvas[p] = candidate[p] and eligible[p] = 0 where mask[p] != 0;
 *   stable[q] = stable[q] + 1 if argmax[p] == prev_argmax[p] at every position of the
 *               request, else 0;
 *   prev_argmax[p] = argmax[p];  steps[q] += 1;
 *   converged[q] = (stable[q] >= stable_steps && mean_H < entropy_threshold)
 *                  || steps[q] >= step_limit,
 *   mean_H = (sum of H over the request's L_c positions, in fp64) / L_c, compared with
 *   the threshold widened to fp64.
 *
 *   candidate [R] int32: the tokens the step puts on the canvas (drawn, or the argmax)
 *   argmax [R] int32: the step's argmax predictions; H [R] fp32; mask [R] uint8
 *   canvas [R] int32, eligible [R] uint8, prev_argmax [R] int32: read and written
 *   stable, steps [n_req] int32, converged [n_req] uint8: read and written
 * The caller owns the state and starts it as: prev_argmax = -1 (every byte 0xFF),
 * stable = steps = 0, eligible = 1, canvas = the starting canvas.  The flag is
 * recomputed at every step; the caller retires a converged canvas.
 * Requires n_req >= 0, 1 <= L_c <= 1024 (above: DG_ERR_UNSUPPORTED), stable_steps >= 0,
 * step_limit >= 1, a threshold that is not NaN, non-NULL pointers when n_req > 0
 * (else DG_ERR_INVALID_ARG).  n_req == 0 queues nothing.  Asynchronous.
 */
dg_status dg_loop_update(const int32_t *candidate, const int32_t *argmax, const float *H,
                         const uint8_t *mask, int32_t n_req, int32_t L_c, int32_t stable_steps,
                         float entropy_threshold, int32_t step_limit,
                         int32_t *canvas, uint8_t *eligible, int32_t *prev_argmax,
                         int32_t *stable, int32_t *steps, uint8_t *converged,
                         dg_stream_t stream);

/*
 * One step of the denoising loop on one stream: the fused step with its acceptance
 * restricted to the eligible positions (dg_entropy_accept_eligible), followed by
 * dg_loop_update.
 *   temperature == 0: the candidate is the argmax and kappa is dg_row_stats' (ln Z);
 *                     `candidate` may be NULL.
 *   temperature > 0:  the candidates are drawn as dg_row_stats_sample draws them (seed,
 *                     offset; advance the offset every step) into `candidate`, kappa is
 *                     -ln p of the drawn token, and the canvas takes the drawn tokens;
 *                     stability is still judged on the argmax.  Over the whole vocabulary
 *                     (one read of the logits) the draw is folded into the product, with
 *                     the same distribution and Philox stream; over a slice, or with
 *                     DG_STEP_TWO_PASS, dg_row_stats_sample itself runs first.
 * Other arguments as dg_sampler_step, dg_entropy_accept_eligible and dg_loop_update;
 * the loop state (canvas, eligible, prev_argmax, stable, steps, converged) is read and
 * written in place, so successive calls on one stream (or one captured graph,
 * replayed) run successive steps.  A negative, infinite or NaN temperature is
 * DG_ERR_INVALID_ARG.  flags as dg_sampler_step.
 */
dg_status dg_sampler_loop_step(const float *logits, int32_t n_req, int32_t L_c, int64_t V,
                               int64_t ldl, const uint16_t *W, int64_t vocab_start,
                               int64_t vocab_end, int64_t rows_pad, int64_t ldw, int64_t d,
                               float gamma, const float *budgets, int32_t min_accept,
                               int32_t stable_steps, float entropy_threshold, int32_t step_limit,
                               float temperature, uint64_t seed, uint64_t offset,
                               float *m, float *lse, float *H, float *kappa, int32_t *argmax,
                               int32_t *candidate, int32_t *order, uint8_t *mask,
                               int32_t *n_accepted, float *E, int64_t ldo,
                               int32_t *canvas, uint8_t *eligible, int32_t *prev_argmax,
                               int32_t *stable, int32_t *steps, uint8_t *converged, uint32_t flags,
                               void *workspace, size_t workspace_bytes, dg_stream_t stream);

/*
 * ---- 8-bit embedding table (E4M3 codes with per-row scales) ----
 *
 * The pages run quantised checkpoints ([P2] "量子化チェックポイント": FP8 weights; [P1]
 * "Running it": INT8) but do not say the embedding table is quantised or how.  These calls
 * take the table as E4M3 codes Q [rows, ldq] uint8 (the OCP 8-bit format: 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits, subnormals, no infinity, 0x7F/0xFF NaN, 448
 * the largest finite magnitude) and one fp32 scale per row: W[v, j] = scale[v] e4m3(Q[v, j]).
 * The table is half the bytes of bf16, and the product streams it.
 */

/*
 * Per-row quantisation of a bf16 table W [V, ldw] (bit patterns) into Q [V, ldq] and
 * scale [V]: scale[v] = amax_v / 448 (fp32, correctly rounded) with amax_v the largest
 * |W[v, j]|; Q[v, j] = the E4M3 code nearest to W[v, j] / scale[v] (correctly rounded fp32
 * quotient), ties to the even code, magnitudes past 448 saturated.  A zero row gets scale 0
 * and codes 0.  Entries must be finite.  W 4-byte aligned, Q 2-byte aligned, ldw and ldq
 * even (else DG_ERR_UNSUPPORTED); the caller owns all three buffers.
 */
dg_status dg_quantize_e4m3(const uint16_t *W, int64_t V, int64_t d, int64_t ldw, uint8_t *Q,
                           int64_t ldq, float *scale, dg_stream_t stream);

/*
 * Bytes of device workspace dg_soft_embed_e4m3 and dg_sampler_step_e4m3 need (the tile
 * width differs from the bf16 product's).  0 for an invalid shape or without a device.
 */
size_t dg_soft_embed_workspace_size_e4m3(int64_t R, int64_t vocab_len, int64_t d);

/*
 * dg_soft_embed with the 8-bit table: E = gamma * sum over the slice of
 * exp(l - lse) scale[v] e4m3(Q[v - s, :]).
 *   Q_shard      [rows_pad, ldq] E4M3 codes, row j = vocabulary entry vocab_start + j
 *   scale_shard  [rows_pad] fp32 row scales (rows past the slice are never read)
 * The probabilities are not cast to 8 bits: each p scale[v] is held as two E4M3 parts
 * (high and low, about eight significant bits together, as bf16) with a power-of-two scale
 * per row and 32-entry block, and the product runs as block-scaled E4M3 MMAs with fp32
 * accumulation and the same fixed-order split-K reduce.  Requires Q 16-byte aligned with
 * ldq % 16 == 0 and scale 4-byte aligned (else DG_ERR_UNSUPPORTED); other rules as
 * dg_soft_embed, with the workspace from dg_soft_embed_workspace_size_e4m3.
 */
dg_status dg_soft_embed_e4m3(const float *logits, int64_t ldl, const float *lse, int64_t R,
                             int64_t vocab_start, int64_t vocab_end, const uint8_t *Q_shard,
                             const float *scale_shard, int64_t rows_pad, int64_t ldq, int64_t d,
                             float gamma, float *out, int64_t ldo, void *workspace,
                             size_t workspace_bytes, dg_stream_t stream);

/*
 * dg_sampler_step with the 8-bit table (Q, scale, ldq as dg_soft_embed_e4m3).  With the
 * whole vocabulary and a workspace of dg_soft_embed_workspace_size_e4m3 bytes it is the
 * single-pass step (the same references, redo rule and statistics as dg_sampler_step);
 * flags as dg_sampler_step.
 */
dg_status dg_sampler_step_e4m3(const float *logits, int32_t n_req, int32_t L_c, int64_t V,
                               int64_t ldl, const uint8_t *Q, const float *scale,
                               int64_t vocab_start, int64_t vocab_end, int64_t rows_pad,
                               int64_t ldq, int64_t d, float gamma, const float *budgets,
                               int32_t min_accept, float *m, float *lse, float *H, float *kappa,
                               int32_t *argmax, int32_t *order, uint8_t *mask,
                               int32_t *n_accepted, float *E, int64_t ldo, uint32_t flags,
                               void *workspace, size_t workspace_bytes, dg_stream_t stream);

/*
 * dg_sampler_loop_step with the 8-bit table (Q, scale, ldq as dg_soft_embed_e4m3; the loop
 * state and the other arguments as dg_sampler_loop_step).  The loop's decisions depend on
 * the statistics only, so a loop over the 8-bit table keeps the same canvas and state as one
 * over the bf16 table it was quantised from; E differs by the table's quantisation.
 */
dg_status dg_sampler_loop_step_e4m3(const float *logits, int32_t n_req, int32_t L_c, int64_t V,
                                    int64_t ldl, const uint8_t *Q, const float *scale,
                                    int64_t vocab_start, int64_t vocab_end, int64_t rows_pad,
                                    int64_t ldq, int64_t d, float gamma, const float *budgets,
                                    int32_t min_accept, int32_t stable_steps,
                                    float entropy_threshold, int32_t step_limit, float temperature,
                                    uint64_t seed, uint64_t offset, float *m, float *lse, float *H,
                                    float *kappa, int32_t *argmax, int32_t *candidate,
                                    int32_t *order, uint8_t *mask, int32_t *n_accepted, float *E,
                                    int64_t ldo, int32_t *canvas, uint8_t *eligible,
                                    int32_t *prev_argmax, int32_t *stable, int32_t *steps,
                                    uint8_t *converged, uint32_t flags, void *workspace,
                                    size_t workspace_bytes, dg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DGSAMP_H */
