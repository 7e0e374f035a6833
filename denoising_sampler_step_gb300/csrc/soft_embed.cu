// Self-conditioning soft embedding E = gamma * P[:, s:e] W_shard[0:e-s], with
// P = bf16(exp(logits - lse)) formed on the fly in shared memory.
//
// What it computes: calvarado04.com, eq. e^sc (the expected embedding p_i W) and
// "The fix" (the product over a vocabulary slice [s, e) with the shard's first e-s
// rows, the probabilities cast to the embedding dtype, gamma applied after the sum;
// padded shard rows are never part of the product).
//
// Kernel design (the one dense contraction of the step, on the tcgen05 tensor cores):
//   - a cluster of four CTAs, two tcgen05 CTA pairs, owns 256 output rows x two adjacent
//     512-column tiles and one contiguous range of 32-entry vocabulary blocks (split-K over
//     the vocabulary): each pair (M = 256, 128 rows per CTA) computes one column tile into
//     its CTAs' 512 TMEM columns;
//   - per block, each CTA loads its 128 of every 256 W columns of its pair's tile — four
//     64-column atoms of 32 rows in one 4-D TMA load (the pair form, counted on the even
//     CTA's barrier): every W byte leaves L2 once, and W and A share a six-deep ring;
//   - the CTAs of one column parity form a block's A operand: they load its logits tile
//     [128 x 32] fp32 by TMA, and eight producer warps (two groups of four taking alternate
//     blocks, 32 rows each) turn it into bf16 exp2(l*log2e - lse*log2e) (rounded to nearest
//     even) in the K-major 64-byte-swizzled layout, hand the logits slot back at once and
//     copy their rows to the CTA with the same rows in the other pair; the probabilities
//     never go to global memory;
//   - one thread of each pair's even CTA issues tcgen05.mma.cta_group::2 (M = 256, N = 256,
//     K = 16, bf16 x bf16 -> fp32) for the two 256-column halves once the A tile is in place
//     in both CTAs (its producers' arrivals, the odd CTA's 16-byte signal copies, or the
//     copied tile and the odd CTA's relayed signal) and both CTAs' W bytes have landed; one
//     tcgen05.commit frees the W and A slots in all four CTAs once the MMAs have read them;
//   - every warp then reads the accumulator with tcgen05.ld and stores the partial tile;
//     splitk_reduce_kernel adds the split partials in split order, multiplies by gamma
//     and writes E (bitwise reproducible).
//   A column tail of 256 or fewer (d = 2816 = 5 x 512 + 256) is a half-width tile.  bf16 W
//   loads mark their lines evict-first, which keeps the logits in L2.  Every barrier wait is
//   bounded (about a second); a wait that gives up records DG_ERR_TIMEOUT, drains what is in
//   flight and leaves the kernel.
//
// Single pass (no lse yet): the producers form exp(l - c) against a per-(split, row)
// reference c, and the CTAs of one column pair fold each block's row statistics (and, in a
// sampling loop step, the draw's first level) from the same values; single_pass_stats_kernel
// merges the split summaries into the row statistics and the scales exp(c - lse), and the
// reduce applies them (recomputing the rare (split, row) whose probabilities against c
// could overflow), with each request's acceptance (and loop update) in its first CTAs.
//
// The same kernel, instantiated for an 8-bit table (E4M3 codes with one fp32 scale per
// vocabulary row), runs block-scaled E4M3 MMAs (kind::mxf8f6f4) on the same four-CTA layout:
// the producers take each block's exponentials against its own maximum, fold in the
// (normalised, staged) row scales and split each value into two E4M3 parts under a
// power-of-two scale per (row, block); each CTA keeps the scales of its rows with its A tile
// (and copies them with it), and per block the pair's MMA thread copies them into both CTAs'
// TMEM ahead of four M = 256 MMAs (two column halves, high and low parts).  Column tiles are
// 480 wide (256 + 224), so that the scale factors fit beside the accumulator in TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "accept.cuh"
#include "dg_common.cuh"
#include "dg_internal.h"
#include "philox.cuh"
#include "row_state.cuh"

namespace dg {

namespace {

constexpr int BM = 128;          // rows per CTA (TMEM lanes)
constexpr int BK = 32;           // vocabulary entries per block
#ifndef DG_SE_LSTAGES
#define DG_SE_LSTAGES 4
#endif
constexpr int LSTAGES = DG_SE_LSTAGES;  // logits ring, released by the producers once read
constexpr int PRODUCER_WARPS = 8;
#ifndef DG_SE_PGROUPS
#define DG_SE_PGROUPS 2
#endif
constexpr int PGROUPS = DG_SE_PGROUPS;           // producer groups, taking the blocks in turn
constexpr int GROUP_WARPS = PRODUCER_WARPS / PGROUPS;
constexpr int ROWS_PER_LANE = 128 / (32 * GROUP_WARPS);
// Warp roles.  A thread blocked in a barrier wait or in a full MMA/TMA queue slows the
// shared-memory work of the other warps on its scheduler (warp % 4), so: warp 4 issues the
// MMAs and warp 8 the logits TMA (scheduler 0, no producers); warp 11 issues the W TMA
// (scheduler 3, two producers); warps 1-3, 5-7, 9 and 10 produce A.  Every warp takes part
// in the epilogue.  The 8-bit table has the same roles; its warp 0 stages the row scales.
constexpr int THREADS = 384;
constexpr int TMEM_COLS = 512;
constexpr uint16_t kPairMask = 0x3;
// A cluster of CTAs.
// bf16 table: four CTAs, two tcgen05 CTA pairs (ranks 0-1 and 2-3) over the same 256 rows and
//   two adjacent column tiles: rank r holds rows 128 (r & 1) ... of the 256 and column tile
//   2 cp + (r >> 1).  In each pair the even CTA issues M = 256 MMAs over both CTAs' rows
//   (cta_group::2); each CTA loads 128 of every 256 W columns, so each W byte leaves L2 once
//   and a W slot is half a block's tile.  The odd CTA's W bytes complete on the even CTA's
//   barrier (the pair form of the TMA load).  The A operand is shared between the pairs: for
//   block i the CTAs with (r >> 1) == i % 2 load its logits and form its A tile, keep it and
//   copy it to the CTA with the same rows in the other pair (r ^ 2); a pair's odd CTA tells
//   its even CTA that its rows are in place with a 16-byte bulk copy onto the even CTA's
//   barrier (directly when it formed them, relayed when they were copied in).
// 8-bit table: the same four CTAs, with 480-column tiles; a CTA's A tile carries the (row,
//   block) scale factors, which travel with it.
constexpr int kQuadCtas = 4;  // the product's cluster
// ring depth of the pair (W and A slots, one index): half-size W slots leave room for six
// (and the 8-bit table's TMEM holds the scale factors of six slots)
constexpr int kPairStages = 6;

constexpr int L_BYTES = BM * BK * 4;      // logits tile, rows of 128 B (128-byte swizzle)
constexpr int W_BOX_BYTES = BK * 128;     // one TMA box: 32 rows x 128 bytes (64 bf16 or 128 e4m3 columns)
// A operand, rows of 64 B (64-byte swizzle): 32 bf16 probabilities, or for the 8-bit table
// the 32 e4m3 high parts then the 32 low parts
constexpr int A_BYTES = BM * 64;
constexpr int L_RING = LSTAGES * L_BYTES;

// The embedding table's format.  kBf16: bf16 entries, kind::f16 MMAs (bf16 x bf16).
// kE4m3: E4M3 codes with one fp32 scale per vocabulary row; the producers fold the row scale
// into the probabilities and split each into two E4M3 parts with a power-of-two scale per
// (row, block), and the MMAs are block-scaled kind::mxf8f6f4 (e4m3 x e4m3).
enum { kBf16 = kTableBf16, kE4m3 = kTableE4m3 };
template <int F>
struct Fmt;
template <>
struct Fmt<kBf16> {
    static constexpr int BN = 512;                // output columns per cluster tile: halves of 256 + 256
    static constexpr int WST = kPairStages;       // W ring depth (the A ring's: one index for both)
    static constexpr int AST = kPairStages;       // A ring depth
    static constexpr int W_SLOT = BK * BN;        // this CTA's 128 of every 256 columns of a block's W tile
    static constexpr int SF_BYTES = 0;
};
template <>
struct Fmt<kE4m3> {
    // 24 TMEM columns hold the per-slot A scales and 8 the B scales, so the accumulator keeps
    // 480: halves of 256 + 224
    static constexpr int BN = 480;
    static constexpr int N1 = 224;                // N of the second half
    static constexpr int WST = kPairStages;
    static constexpr int AST = kPairStages;
    // this CTA's N/2 columns of each half: one 128-column atom of 32 rows per half (of the
    // second half's atom 112 columns are used)
    static constexpr int W_SLOT = 2 * W_BOX_BYTES;
    // per-slot A scale matrices (128 rows x 16 bytes), the B scale chunk, then the staged
    // row scales (one slot per logits stage: 32 normalised scales and their exponent)
    static constexpr int SF_STAGE = 2048;
    static constexpr int SF_BYTES = AST * SF_STAGE + 512 + LSTAGES * 160;
};
constexpr int S_SLOT = 160;
// TMEM columns of the scale factors (8-bit table): four per A slot (lane m's word in column
// m / 32), then eight for the B scales
constexpr uint32_t kSfaCol = 480, kSfbCol = 504;
template <int F>
constexpr int smem_bytes() {
    return L_RING + Fmt<F>::WST * Fmt<F>::W_SLOT + Fmt<F>::AST * A_BYTES + Fmt<F>::SF_BYTES + 1024 /*align*/ +
           512 /*barriers*/;
}

static_assert(L_BYTES % 1024 == 0 && Fmt<kBf16>::W_SLOT % 1024 == 0 && Fmt<kE4m3>::W_SLOT % 1024 == 0 &&
                  A_BYTES % 1024 == 0,
              "1 KiB alignment");
static_assert(smem_bytes<kBf16>() <= 232448 && smem_bytes<kE4m3>() <= 232448, "shared memory per CTA");
static_assert(kSfaCol + 4 * Fmt<kE4m3>::AST <= kSfbCol && kSfbCol + 8 <= TMEM_COLS,
              "scale-factor columns");
// each producer group keeps to every other slot of the logits and A rings
// a group waits only for phases its own blocks need, and no slot can run two phases ahead
// of its waiter, so the depths need not be multiples of the group count
static_assert(LSTAGES >= PGROUPS && kPairStages >= PGROUPS, "a slot per producer group at least");
// the bf16 pair's A-ready signals: 16 bytes per producer warp in the even CTA, after the barriers
constexpr int kSigOffset = 256;
static_assert(kSigOffset + 16 * (PRODUCER_WARPS + 2) <= 512, "signal area inside the barrier region");

struct Params {
    const float *lse;
    float *ws;           // partial tiles [split][m_tile][n_tile][BN/4][BM][4]
    int64_t k_begin;     // first vocabulary column of block 0 (multiple of 4)
    int64_t vocab_start;
    int64_t vocab_end;
    int64_t nkb;
    int R;
    int m_tiles, n_tiles;
    int n_full;          // n-tiles of full width (two halves)
    int tail_halves;     // 1 if the last n-tile is 256 wide or less, else 0
    int splits, tail_splits;
    int w3d;             // 1: the W map is 3-D (atom columns x rows x atoms), one load per CTA and half
    int w4d_atoms;       // > 0: the 4-D W map (both halves in one load) holds this many atoms per row
    // 8-bit table: the fp32 scale of vocabulary entry v is w_scale[v - vocab_start]
    const float *w_scale;
    // single pass (no lse yet): each split's probabilities are taken against a reference
    // c per row, exp(l - c), and the column-tile-0 clusters also fold the row statistics
    int fused;
    const float *logits; // the reference's source (the split's first kRefEntries entries)
    int64_t ldl;
    float *ref;          // [splits][R] c, then (after the statistics) exp(c - lse), or -1 where the
                         // (split, row) must be recomputed (kRedo)
    float4 *state;       // [splits][n_tiles][R] row summaries (m, argmax bits, rest, t) of the blocks
                         // of the split the column tile folds (`fold` in the producers)
    // single pass with the draw at temperature 1 / inv_tau: the folded blocks also take the
    // draw's first level (a group of 16 entries by the log-mass of l / T + Gumbel), the
    // statistics kernel the second
    int draw;
    float inv_tau;
    uint32_t k0, k1, o0, o1;  // Philox key (seed) and counter offset words
    float2 *draws;            // [splits][n_tiles][R] best group score, group (int bits)
    int32_t *candidate;       // [R] the drawn tokens
};

// A (split, row) is redone when its probabilities against c could overflow: when the sum
// of exp(l - c) over the split passes e^kRefSumLog (about 4e35, so that with |W| <= 100 the
// fp32 partial stays below 4e37), or when the split's maximum lies more than kRefBelow nats
// below c (everything would underflow).
// Vocabulary blocks [kb0, kb1) of split j of S.
__host__ __device__ inline void split_range(const Params &p, int j, int S, int64_t *kb0, int64_t *kb1) {
    *kb0 = (int64_t)j * p.nkb / S;
    *kb1 = (int64_t)(j + 1) * p.nkb / S;
}

constexpr float kRefSumLog = 82.0f;
constexpr float kRefBelow = 64.0f;
// The scale the statistics kernel leaves for a (split, row) the reduce recomputes.
constexpr float kRedo = -1.0f;
// The reference is the largest of a split's first kRefEntries logits.
constexpr int kRefEntries = 32;

// The largest of 32 values (NaN ignored), as a tree of three-input maxima: 16 instructions
// and five levels of dependency.
__device__ __forceinline__ float max32(const float (&v)[32]) {
    float a[11];
#pragma unroll
    for (int t = 0; t < 10; ++t) a[t] = max3f(v[3 * t], v[3 * t + 1], v[3 * t + 2]);
    a[10] = fmaxf(v[30], v[31]);
    const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]), b2 = max3f(a[6], a[7], a[8]);
    const float b3 = fmaxf(a[9], a[10]);
    return fmaxf(max3f(b0, b1, b2), b3);
}

// Sum of 16 values as a tree (15 additions, depth 4).
__device__ __forceinline__ float sum16(const float *v) {
    float a[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) a[t] = v[2 * t] + v[2 * t + 1];
#pragma unroll
    for (int t = 0; t < 4; ++t) a[t] = a[2 * t] + a[2 * t + 1];
    return (a[0] + a[1]) + (a[2] + a[3]);
}

// The single pass's statistics fold of the bf16 product, kept relative to the split's
// reference c (the exponentials e = exp(l - c) the producers already formed): the running
// maximum M of the lane's row over the folded blocks, A the index of its first occurrence,
// E = exp(M - c), R = the sum of e over the other entries, T = the sum of e (l - c) over all
// entries; R and T in two levels (R16, T16 over up to 16 blocks) so that no fp32 sum runs
// over more than a few dozen terms.  No exponential per block: a block whose maximum does
// not pass M adds all its e to R, and only a block that raises M takes the exact sum of its
// other entries (keeping the argmax's own term out of R keeps kappa = log1p(rest) exact for
// rows near one-hot).  Blocks more than 60 nats above c (e could overflow) take the
// statistics kernel's fold instead.
struct RefState {
    float M;
    int A;
    float E;
    float R, T, R16, T16;
};

// The RowState (m, a, rest, t relative to m) of a RefState: rest = R exp(c - M),
// t = exp(c - M) (T - (M - c)(R + E)).
__device__ __forceinline__ rowstate::RowState ref_to_row_state(const RefState &r, float c) {
    if (r.M == -INFINITY) return rowstate::empty_row_state();
    const float R = r.R + r.R16, T = r.T + r.T16;
    const float inv = ex2_approx((c - r.M) * kLog2e);
    return rowstate::RowState{r.M, r.A, R * inv, inv * fmaf(-(r.M - c), R + r.E, T)};
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int F>
__global__ void __launch_bounds__(THREADS, 1)
    soft_embed_kernel(const __grid_constant__ CUtensorMap tm_logits, const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_w4,
                      const Params p) {
    constexpr int BN = Fmt<F>::BN;
    constexpr int W_SLOT = Fmt<F>::W_SLOT;
    constexpr int WST = Fmt<F>::WST;
    constexpr int AST = Fmt<F>::AST;
    constexpr int W_RING = WST * W_SLOT;
    constexpr int A_SLOT = A_BYTES;
    constexpr int A_RING = AST * A_SLOT;
    static_assert(ROWS_PER_LANE == 1, "a warp copies 32 whole rows");
    static_assert(AST >= PGROUPS, "an A slot per producer group at least");
    // a block's W bytes complete on its A slot's barrier (one index for both rings), so the
    // MMA thread waits on one barrier per block
    static_assert(WST == AST, "one ring index");
    // the scale rows that travel with an 8-bit A tile
    constexpr uint32_t kSfRows = F == kE4m3 ? (uint32_t)Fmt<kE4m3>::SF_STAGE : 0u;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *l_ring = smem;
    uint8_t *w_ring = smem + L_RING;
    uint8_t *a_ring = smem + L_RING + W_RING;
    uint8_t *sf_ring = smem + L_RING + W_RING + A_RING;  // 8-bit table: per-stage A scale chunks, B scale chunk
    uint8_t *sfb_chunk = sf_ring + (F == kE4m3 ? AST * Fmt<kE4m3>::SF_STAGE : 0);  // 8-bit table: the B scale chunk
    uint8_t *s_ring = sfb_chunk + 512;                   // 8-bit table: staged row scales
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L_RING + W_RING + A_RING + Fmt<F>::SF_BYTES);
    uint64_t *full_l = bars;                   // logits tile landed
    uint64_t *empty_l = full_l + LSTAGES;      // the producer warps have read it
    uint64_t *full_a = empty_l + LSTAGES;      // A operand written and the W tile landed
    uint64_t *empty = full_a + AST;            // MMAs done with the A slot (and, one ring, the W slot: both CTAs')
    uint64_t *acc_full = empty + AST;          // accumulator complete
    uint64_t *full_s = acc_full + 1;           // 8-bit table: a block's row scales staged
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(full_s + LSTAGES);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // bf16 pair: 16-byte landing places of the odd CTA's A-ready signals (one per producer
    // warp, in the even CTA; never read) and the source of those copies
    uint8_t *sig_area = reinterpret_cast<uint8_t *>(bars) + kSigOffset;

    // Overlap with the neighbours on the stream (programmatic dependent launch): this grid
    // may start while the row-statistics grid before it runs, so every thread calls
    // grid_dependency_wait() before it touches lse (or before it lets the next grid start);
    // the W and logits loads of the first ring round do not depend on it and go first.
    // The kernel queued next (the acceptance) reads only the row statistics, so each thread
    // lets it start once its own wait has returned.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();

    // work of this cluster: (column pair cp, row pair mp, split j); n_tiles is even (a last
    // odd tile's partner lies past d and reads zeros); tiles from n_full on are half width
    const int pair = blockIdx.x / kQuadCtas;
    const int m_pairs = p.m_tiles / 2;
    const int ntp_count = p.n_tiles / 2;
    const int ntp = pair % ntp_count;
    const int mp = (pair / ntp_count) % m_pairs;
    const int j = pair / (ntp_count * m_pairs);
    const int S = p.splits;
    const int nt = 2 * ntp + (int)(rank >> 1);
    const int halves = nt < p.n_full ? 2 : 1;
    const int mt = 2 * mp + (int)(rank & 1);
    // the column parity of this CTA in its cluster: it produces (loads the logits of, stages
    // the scales of, computes the A operand of) the blocks i with i % 2 == cpar and copies each
    // A operand to the CTA with the same rows in the other column tile
    const int cpar = (int)(rank >> 1);
    const int i0 = cpar, di = 2;
    int64_t kb0, kb1;
    split_range(p, j, S, &kb0, &kb1);
    const int nkb = (int)(kb1 - kb0);
    const int row0 = mt * BM;
    const int col0 = nt * BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < LSTAGES; ++s) {
            mbar_init(smem_u32(&full_l[s]), 1);
            mbar_init(smem_u32(&empty_l[s]), GROUP_WARPS);
            mbar_init(smem_u32(&full_s[s]), 1);
        }
        for (int s = 0; s < AST; ++s) {
            // full_a, a pair's even CTA: a slot of its own parity, the producer group's warps and
            // the W TMA's arrival (with both CTAs' W bytes and the odd CTA's four signals); a slot
            // of the other parity, the W TMA's arrival alone (with the W bytes, the copied A tile
            // (8-bit table: and its scale rows) and the odd CTA's relayed signal).  Odd CTA: the
            // relay's arrival (with the copied A tile; slots of the other parity only).
            // empty: the commits of both CTA pairs (the pair that reads the slot and the one that
            // copies into it)
            const int fa = (rank & 1) == 0 && (s & 1) == cpar ? GROUP_WARPS + 1 : 1;
            mbar_init(smem_u32(&full_a[s]), fa);
            mbar_init(smem_u32(&empty[s]), 2);
        }
        mbar_init(smem_u32(acc_full), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_logits);
        prefetch_tmap(&tm_w);
        if (p.w4d_atoms > 0) prefetch_tmap(&tm_w4);
    }
    if constexpr (F == kE4m3) {
        // the B scale chunk: every byte 127, a factor of 1 (the table's row scales go into A)
        if (threadIdx.x < 128) reinterpret_cast<uint32_t *>(sfb_chunk)[threadIdx.x] = 0x7F7F7F7Fu;
        fence_proxy_async_smem();
    }
    __syncwarp();
    if (warp == 0) tmem_alloc_pair<TMEM_COLS>(smem_u32(tmem_slot));  // a joint allocation in both CTAs
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the peer's barriers exist before any copy or commit reaches them
    cluster_sync_all();
    const uint32_t tmem_base = *tmem_slot;
    bool ok = true;  // false once this thread gave up on a wait
    // single pass: the producers' reference per row and their row statistics; each block of
    // the split is folded by one column tile (`fold` below), evenly by the producer groups,
    // after handing the block's A tile over, so that the fold stays off the product's
    // critical path; in levels (a block, 16 blocks, all) so that no fp32 sum runs over more
    // than a few dozen terms: rest keeps kappa = log1p(rest) accurate near one-hot
    int my_grp = -1;
    int my_rows[ROWS_PER_LANE];
    float my_ref[ROWS_PER_LANE];
    rowstate::RowState my_st[ROWS_PER_LANE], my_st16[ROWS_PER_LANE];
    RefState my_rs[ROWS_PER_LANE];  // bf16 table: the fold relative to the reference c
    int my_folded = 0;
    float my_gbest[ROWS_PER_LANE];  // the draw's first level: best group score and group
    int my_gidx[ROWS_PER_LANE];
#pragma unroll
    for (int q = 0; q < ROWS_PER_LANE; ++q) {
        my_rows[q] = 0;
        my_ref[q] = 0.0f;
        my_st[q] = rowstate::empty_row_state();
        my_st16[q] = rowstate::empty_row_state();
        my_rs[q] = RefState{-INFINITY, 0x7fffffff, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        my_gbest[q] = -INFINITY;
        my_gidx[q] = 0x7fffffff;
    }

    constexpr int kWarpW = 11, kWarpL = 8, kWarpMma = 4, kWarpStage = 0;
    const bool producer = (warp & 3) != 0 && warp < 11;
    if (warp == kWarpW) {
        // ------------------------------------------------------------ W TMA
        // each CTA loads its N/2 columns of each half (bf16: atoms 4h + 2 (rank & 1) and + 1 of
        // 64 columns; 8-bit table: one 128-column atom at 256 h + (rank & 1) N_h / 2), the bytes
        // counted on its pair's even CTA's A slot barrier, which that CTA arms for both CTAs'
        // bytes and the odd CTA's A-ready signals (or, for a block the other pair forms, the
        // copied A tile, its scale rows and the relayed signal)
        if (lane == 0) {
            int issued[WST];
            for (int s = 0; s < WST; ++s) issued[s] = 0;
            // bf16 over one 256-row block: every W byte leaves L2 once (evict first).  Over
            // several row blocks (or the 8-bit table's two row-block clusters) the clusters of a
            // column pair read each W tile close together: ordinary priority keeps it in L2 for
            // them (at 2,048 rows evict-first made the product read W about five times from DRAM)
            const uint64_t w_policy =
                (F == kE4m3 || p.m_tiles > 2) ? l2_policy_evict_normal() : l2_policy_evict_first();
            // bf16: a 4-D map fetches a CTA's four atoms of a full-width tile in one load, a 3-D
            // map its two atoms of a half (the TMA unit's cost is per load, not per byte: two
            // 64-column boxes per half in place of one 3-D load made the product 8 % slower,
            // and one load per block in place of two made it 4 % faster)
            const bool w3d = p.w3d;
            const uint32_t lead_a = map_to_cta(smem_u32(&full_a[0]), rank & ~1u);  // the pair's even CTA's full_a[0]
            for (int i = 0; i < nkb; ++i) {  // one block per ring slot
                const int s = i % WST;
                const uint32_t u = (uint32_t)(i / WST);
                if (i == WST) {  // the first round of W loads is out
                    grid_dependency_wait();
                    grid_launch_dependents();
                }
                if (u > 0 && !mbar_wait(smem_u32(&empty[s]), (u - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int64_t k = p.k_begin + (kb0 + (int64_t)i) * BK;
                const uint32_t bw = smem_u32(&full_a[s]);
                const int wy = (int)(k - p.vocab_start);
                // both CTAs' W bytes of the slot, and the odd CTA's four A-ready signals (a block
                // this pair forms) or the A tile (and scale rows) copied in and the odd CTA's
                // relayed signal
                if ((rank & 1) == 0)
                    mbar_arrive_expect_tx(bw, (uint32_t)halves * W_SLOT +
                                                  ((i & 1) == cpar ? 16u * GROUP_WARPS
                                                                   : (uint32_t)A_BYTES + kSfRows + 16u));
                const uint32_t bl = lead_a + 8u * (uint32_t)s;
                if constexpr (F == kE4m3) {
                    for (int h = 0; h < halves; ++h) {
                        const int xh = col0 + 256 * h + (int)(rank & 1) * (h == 0 ? 128 : Fmt<kE4m3>::N1 / 2);
                        tma_load_2d_pair_hint(smem_u32(w_ring + s * W_SLOT + h * W_BOX_BYTES), &tm_w, bl, xh, wy,
                                              w_policy);
                    }
                } else if (halves == 2 && col0 / 64 + 2 * (int)(rank & 1) + 6 <= p.w4d_atoms) {
                    // both halves' atoms (4h + 2 (rank & 1) and + 1) in one load
                    tma_load_4d_pair_hint(smem_u32(w_ring + s * W_SLOT), &tm_w4, bl, 0, wy,
                                          col0 / 64 + 2 * (int)(rank & 1), 0, w_policy);
                } else {
                    for (int h = 0; h < halves; ++h) {
                        const uint32_t dst = smem_u32(w_ring + s * W_SLOT + h * 2 * W_BOX_BYTES);
                        const int atom = col0 / 64 + 4 * h + 2 * (int)(rank & 1);  // this CTA's half of the pair
                        if (w3d) {
                            tma_load_3d_pair_hint(dst, &tm_w, bl, 0, wy, atom, w_policy);
                        } else {
                            tma_load_2d_pair_hint(dst, &tm_w, bl, 64 * atom, wy, w_policy);
                            tma_load_2d_pair_hint(dst + W_BOX_BYTES, &tm_w, bl, 64 * (atom + 1), wy, w_policy);
                        }
                    }
                }
                issued[s] = (int)u + 1;
            }
            if (nkb <= WST) {
                grid_dependency_wait();
                grid_launch_dependents();
            }
            // loads in flight finish before the CTA may leave (bf16 pair: the even CTA's barriers
            // count both CTAs' loads, and the odd CTA leaves only after the final cluster
            // barrier, which the even CTA reaches after this drain)
            if (!ok && (rank & 1) == 0)
                for (int s = 0; s < WST; ++s)
                    if (issued[s] > 0) drain_wait(smem_u32(&full_a[s]), (issued[s] - 1) & 1);
        }
    } else if (warp == kWarpL) {
        // ------------------------------------------------------------ logits TMA
        if (lane == 0) {
            int issued[LSTAGES];
            for (int s = 0; s < LSTAGES; ++s) issued[s] = 0;
            int nl = 0;  // logits tiles this CTA loads
            for (int li = 0, i = i0; i < nkb; ++li, i += di, ++nl) {
                const int s = li % LSTAGES;
                const uint32_t u = (uint32_t)(li / LSTAGES);
                if (li == LSTAGES) {  // the first round of logits loads is out
                    grid_dependency_wait();
                    grid_launch_dependents();
                }
                if (u > 0 && !mbar_wait(smem_u32(&empty_l[s]), (u - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const int64_t k = p.k_begin + (kb0 + i) * BK;
                const uint32_t bl = smem_u32(&full_l[s]);
                mbar_arrive_expect_tx(bl, L_BYTES);
                tma_load_2d(smem_u32(l_ring + s * L_BYTES), &tm_logits, bl, (int)k, row0);
                issued[s] = (int)u + 1;
            }
            if (nl <= LSTAGES) {
                grid_dependency_wait();
                grid_launch_dependents();
            }
            if (!ok)
                for (int s = 0; s < LSTAGES; ++s)
                    if (issued[s] > 0) drain_wait(smem_u32(&full_l[s]), (issued[s] - 1) & 1);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        // (a pair's even CTA's thread issues for both CTAs; the odd CTA's relays)
        if (lane == 0 && (rank & 1) != 0) {
            // relay: the A tiles (8-bit table: with their scale rows) of the blocks the other pair
            // forms arrive here by copy; once one has landed, a 16-byte copy onto the even CTA's
            // barrier tells its MMA thread
            const uint32_t lead = rank & ~1u;
            for (int i = 1 - cpar; i < nkb; i += 2) {
                const int s = i % AST;
                const uint32_t u = (uint32_t)(i / AST);
                mbar_arrive_expect_tx(smem_u32(&full_a[s]), (uint32_t)A_BYTES + kSfRows);
                if (!mbar_wait(smem_u32(&full_a[s]), u & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                bulk_copy_to_cluster(map_to_cta(smem_u32(sig_area + 16 * (PRODUCER_WARPS + 1)), lead),
                                     smem_u32(sig_area), 16u, map_to_cta(smem_u32(&full_a[s]), lead));
            }
        } else if (lane == 0) {
            grid_dependency_wait();  // nothing to issue before the producers' first tile anyway
            grid_launch_dependents();
            constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, 256, /*A K-major*/ 0, /*B N-major*/ 1);
            // operand descriptors of slot 0; a slot, a K = 16 step or a half is a constant added
            // to the start-address field (addresses stay below 2^18 bytes)
            // A: K-major, 64-byte rows, 8-row groups 512 B apart; +32 B per K = 16 step (bf16) or
            // from the high to the low E4M3 parts (8-bit table)
            const uint64_t a_desc0 = smem_desc(smem_u32(a_ring), 16, 512, 4);
            // B: N-major, atoms of 128-byte rows 4 KiB apart (LBO), 8-row groups 1 KiB apart
            // (SBO); bf16: +2 KiB per K = 16 step, a half is 2 atoms; 8-bit table: one K = 32 step
            // per block, a half is 1 atom
            const uint64_t b_desc0 = smem_desc(smem_u32(w_ring), W_BOX_BYTES, 1024, 2);
            constexpr uint64_t kA_K16 = 32 >> 4, kB_K16 = 2048 >> 4, kB_HALF = (W_SLOT / 2) >> 4;
            // 8-bit table: the B scale factors (all 1) go into their columns once; per block the
            // slot's A scale chunk goes into its four columns ahead of the block's MMAs (the copy
            // and the MMAs run in issue order; the commit covers both); each copy fills both CTAs
            // of the pair, each from its own shared memory
            if constexpr (F == kE4m3) {
                const uint64_t sfb_desc = smem_desc(smem_u32(sfb_chunk), 16, 128, 0);
                for (int q = 0; q < 8; q += 4) tmem_cp_32x128b_warpx4_pair(tmem_base + kSfbCol + q, sfb_desc);
            }
            bool issued_any = false;
            // a block's tiles are tested right after the previous block's MMAs are issued, ahead
            // of its commit; the bounded waits run only when a tile is not there yet.  The odd
            // CTA's loads and signals complete from the other CTA, so the tests acquire at
            // cluster scope
            bool a_in = nkb > 0 && mbar_try_wait_cluster(smem_u32(&full_a[0]), 0);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % AST;
                const uint32_t ph = (uint32_t)(i / AST) & 1;
                if (!a_in && !mbar_wait_cluster(smem_u32(&full_a[s]), ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = a_desc0 + (uint64_t)((s * A_SLOT) >> 4);
                const uint64_t bd = b_desc0 + (uint64_t)((s * W_SLOT) >> 4);
                const uint32_t acc = i > 0 ? 1u : 0u;
                if constexpr (F == kE4m3) {
                    // high parts, then low parts (the word's four bytes are the same scale)
                    constexpr uint32_t id_h0 = idesc_mxf8_e4m3(2 * BM, 256, 0, 1, 0, 0);
                    constexpr uint32_t id_h1 = idesc_mxf8_e4m3(2 * BM, Fmt<F>::N1, 0, 1, 0, 0);
                    constexpr uint32_t id_l0 = idesc_mxf8_e4m3(2 * BM, 256, 0, 1, 1, 0);
                    constexpr uint32_t id_l1 = idesc_mxf8_e4m3(2 * BM, Fmt<F>::N1, 0, 1, 1, 0);
                    constexpr uint64_t kB_ATOM = W_BOX_BYTES >> 4;
                    const uint32_t sfb = tmem_base + kSfbCol;
                    // the slot's TMEM scale columns: free, as the A slot is, once the MMAs of the
                    // slot's previous block are done (its producers waited for that)
                    const uint32_t sfa = tmem_base + kSfaCol + 4 * (uint32_t)s;
                    tmem_cp_128x128b_pair(sfa, smem_desc(smem_u32(sf_ring + s * Fmt<kE4m3>::SF_STAGE), 16, 128, 0));
                    umma_mxf8_pair(tmem_base, ad, bd, id_h0, sfa, sfb, acc);
                    if (halves == 2) umma_mxf8_pair(tmem_base + 256, ad, bd + kB_ATOM, id_h1, sfa, sfb, acc);
                    umma_mxf8_pair(tmem_base, ad + kA_K16, bd, id_l0, sfa, sfb, 1u);
                    if (halves == 2) umma_mxf8_pair(tmem_base + 256, ad + kA_K16, bd + kB_ATOM, id_l1, sfa, sfb, 1u);
                } else {
                    umma_bf16_pair(tmem_base, ad, bd, idesc, acc);
                    if (halves == 2) umma_bf16_pair(tmem_base + 256, ad, bd + kB_HALF, idesc, acc);
                    umma_bf16_pair(tmem_base, ad + kA_K16, bd + kB_K16, idesc, 1u);
                    if (halves == 2) umma_bf16_pair(tmem_base + 256, ad + kA_K16, bd + kB_HALF + kB_K16, idesc, 1u);
                }
                if (i + 1 < nkb) a_in = mbar_try_wait_cluster(smem_u32(&full_a[(i + 1) % AST]), (uint32_t)((i + 1) / AST) & 1);
                // one commit releases the W and A slots, in all four CTAs, once the MMAs have read
                // them (the pair's MMAs read both its CTAs' slots, and the other pair's CTAs copy
                // A tiles into them)
                umma_commit_pair(smem_u32(&empty[s]), 0xF);
                issued_any = true;
            }
            umma_commit_pair(smem_u32(acc_full), (uint16_t)(kPairMask << (rank & 2u)));  // this pair
            if (*abort_flag && issued_any) drain_wait(smem_u32(acc_full), 0);
        }
    } else if (F == kE4m3 && warp == kWarpStage) {
        // ------------------------------------------------------------ row-scale staging
        // (8-bit table) per block: lane t holds the row scale of entry k + t (0 outside the
        // slice); the warp writes u = scale 2^-E with E chosen so that the largest u lies in
        // [0.5, 1), and E.  A block whose scales are all zero (or below 2^-126) stages zeros.
        // The loads run kScalePrefetch blocks ahead of the stores, so that their latency
        // overlaps (the slots themselves follow the logits ring).
        constexpr int kScalePrefetch = 8;
        const int nl = nkb > i0 ? (nkb - i0 + di - 1) / di : 0;  // this CTA's blocks
        auto load_scale = [&](int li) {
            const int64_t v = p.k_begin + (kb0 + i0 + (int64_t)di * li) * BK + lane;
            return (li < nl && v >= p.vocab_start && v < p.vocab_end) ? __ldg(p.w_scale + (v - p.vocab_start)) : 0.0f;
        };
        float pre[kScalePrefetch];
#pragma unroll
        for (int jj = 0; jj < kScalePrefetch; ++jj) pre[jj] = load_scale(jj);
        for (int l0 = 0; l0 < nl && ok; l0 += kScalePrefetch) {
#pragma unroll
            for (int jj = 0; jj < kScalePrefetch; ++jj) {
                const int li = l0 + jj;
                if (li >= nl) break;
                const float sv = pre[jj];
                pre[jj] = load_scale(li + kScalePrefetch);
                const int sl = li % LSTAGES;
                const uint32_t ul = (uint32_t)(li / LSTAGES);
                // the slot is free once the producers of this CTA's block li - LSTAGES have read it
                if (ul > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_l[sl]), (ul - 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                float mx = sv;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const uint32_t eb = __float_as_uint(mx) >> 23;  // biased exponent of the largest scale (>= 0)
                float uu = 0.0f;
                int E = 0;
                if (eb >= 1u && eb <= 252u) {
                    uu = sv * __uint_as_float((253u - eb) << 23);  // times 2^(126 - eb)
                    E = (int)eb - 126;
                }
                float *slot = reinterpret_cast<float *>(s_ring + sl * S_SLOT);
                slot[lane] = uu;
                if (lane == 0) reinterpret_cast<int *>(slot)[32] = E;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&full_s[sl]));
            }
        }
    } else if (producer) {
        // ------------------------------------------------------------ A producers
        // PGROUPS groups take the blocks in turn, so a warp has PGROUPS block times for the
        // dependent chain of one block (barrier waits, stores, proxy fence, arrival); a
        // warp converts ROWS_PER_LANE * 32 rows x all 32 entries of its group's block
        // producer 0..7 (warps 1-3, 5-7, 9, 10)
        const int pw = 3 * (warp >> 2) + (warp & 3) - 1;
        const int grp = pw / GROUP_WARPS;
        const int wig = pw % GROUP_WARPS;
        my_grp = grp;
        int rr[ROWS_PER_LANE];
        float neg_lse2[ROWS_PER_LANE];
        if (p.fused) {
            // reference c: the largest of the split's first 32 entries inside the slice (0 if
            // none is finite); every column tile takes the same c.  A float4 that starts below
            // vocab_end ends inside the row (ldl is a multiple of 4).
            const int64_t k0 = p.k_begin + kb0 * BK;
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q) {
                rr[q] = (wig * ROWS_PER_LANE + q) * 32 + lane;
                const int row = row0 + rr[q];
                float c = -INFINITY;
                if (row < p.R && nkb > 0) {
                    const float *lr = p.logits + (int64_t)row * p.ldl;
#pragma unroll 8
                    for (int c4 = 0; c4 < kRefEntries / 4; ++c4) {
                        const int64_t kk = k0 + 4 * c4;
                        if (kk >= p.vocab_end) break;
                        const float4 f = __ldg(reinterpret_cast<const float4 *>(lr + kk));
                        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            if (kk + t >= p.vocab_start && kk + t < p.vocab_end) c = fmaxf(c, fv[t]);
                    }
                }
                if (!(c > -INFINITY)) c = 0.0f;
                my_rows[q] = rr[q];
                my_ref[q] = c;
                neg_lse2[q] = row < p.R ? -c * kLog2e : -INFINITY;
            }
        } else {
            grid_dependency_wait();  // lse comes from the grid queued before this one
            grid_launch_dependents();
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q) {
                rr[q] = (wig * ROWS_PER_LANE + q) * 32 + lane;  // row of the tile
                const int row = row0 + rr[q];
                // rows past R are zero-filled by the TMA: an offset of -inf makes their entries 0
                neg_lse2[q] = row < p.R ? -p.lse[row] * kLog2e : -INFINITY;
            }
        }
        // the group's blocks: this CTA's li-th block is i = i0 + di li (all blocks, or for the
        // 8-bit table every other); logits and staged scales by li, the A ring by i (8-bit
        // table: by li)
        for (int li = grp, i = i0 + di * grp; i < nkb; li += PGROUPS, i += di * PGROUPS) {
            const int sl = li % LSTAGES;
            // the A ring: slot of block i
            const int s = i % AST;
            const uint32_t ul = (uint32_t)(li / LSTAGES);
            const uint32_t u = (uint32_t)(i / AST);
            // every lane waits (acquire), the warp decides together; the 8-bit table's staged
            // row scales share the logits slot's index and phase
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full_l[sl]), ul & 1, abort_flag) &&
                                             (F != kE4m3 || mbar_wait(smem_u32(&full_s[sl]), ul & 1, abort_flag)))) {
                ok = false;
                break;
            }
            const uint8_t *lt = l_ring + sl * L_BYTES;
            const int64_t k = p.k_begin + (kb0 + i) * BK;
            const bool edge = (k < p.vocab_start) || (k + BK > p.vocab_end);
            uint32_t packed[ROWS_PER_LANE][16];
            uint32_t sf_word[ROWS_PER_LANE];  // 8-bit table: the (row, block) scale bytes
            // every block is folded once per row block, by the producers of a CTA that forms it:
            // the one in column pair (i / 2) % (n_tiles / 2); a CTA's folds alternate between its
            // producer groups
            const bool fold = p.fused && (i >> 1) % ntp_count == ntp;
            // 8-bit table: the block's normalised row scales u (0 outside the slice) and their
            // exponent E (row scale = u 2^E), staged by warp 0
            float us[F == kE4m3 ? 32 : 1];
            int ue = 0;
            if constexpr (F == kE4m3) {
                const float *slot = reinterpret_cast<const float *>(s_ring + sl * S_SLOT);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 f = *reinterpret_cast<const float4 *>(slot + 4 * c);
                    us[4 * c + 0] = f.x;
                    us[4 * c + 1] = f.y;
                    us[4 * c + 2] = f.z;
                    us[4 * c + 3] = f.w;
                }
                ue = reinterpret_cast<const int *>(slot)[32];
            }
            float4 vk[ROWS_PER_LANE][8];  // the logits and their exponentials, kept for the fold
            float ek[ROWS_PER_LANE][32];
            float bmq[ROWS_PER_LANE], kfq[ROWS_PER_LANE];  // 8-bit table: block maximum and k (below)
            // every 16-byte load of the block's rows first; the logits slot (and the staged scales)
            // go back to the TMA at once, so that the next tile's load overlaps this block's work
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q)
#pragma unroll
                for (int c = 0; c < 8; ++c)  // 16-byte chunk of the 128-byte row
                    vk[q][c] = *reinterpret_cast<const float4 *>(lt + rr[q] * 128 + ((c ^ (rr[q] & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_l[sl]));
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q) {
                // the exponentials, then the packing
                float4 v[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) v[c] = vk[q][c];
                float e[32];
                if constexpr (F == kE4m3) {
                    // Each block's exponentials are taken against its own maximum bm: with
                    // k = floor((bm - c) log2 e), e'' = 2^((l - c) log2 e - k + 7) =
                    // exp(l - c) 2^(7 - k) lies in (0, 256), its maximum in [128, 256).  With the
                    // staged scales x = e'' u < 256, and p(l) scale = x 2^(k - 7 + E): the
                    // block's power-of-two scale 2^S, S = k - 7 + E, goes to the MMA (scale byte
                    // 127 + S).  x is split as x = h + l (h = x rounded to E4M3 through fp16, l =
                    // the rest, exact in fp16, rounded to E4M3 too): both MMAs take 2^S, and
                    // together h and l carry about eight significant bits, as bf16 does (a rest
                    // below E4M3's normal range, 2^-6, only occurs for x < 2^-2, under 2^-9 of
                    // the block maximum, and keeps an absolute error under 2^-10).
                    float xb[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        xb[4 * c + 0] = v[c].x;
                        xb[4 * c + 1] = v[c].y;
                        xb[4 * c + 2] = v[c].z;
                        xb[4 * c + 3] = v[c].w;
                    }
                    if (edge) {
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (k + t < p.vocab_start || k + t >= p.vocab_end) xb[t] = -INFINITY;
                    }
                    const float bm = max32(xb);
                    // a block with nothing finite keeps k = 0: its exponentials are all 0
                    // (rows past R have no reference: k = 0 and exponentials of 0)
                    const float kf =
                        (bm > -INFINITY && neg_lse2[q] > -INFINITY) ? floorf(fmaf(bm, kLog2e, neg_lse2[q])) : 0.0f;
                    const float off = neg_lse2[q] - kf + 7.0f;
#pragma unroll
                    for (int t = 0; t < 32; ++t) e[t] = ex2_approx(fmaf(xb[t], kLog2e, off));
                    bmq[q] = bm;
                    kfq[q] = kf;
                    int S = (int)kf - 7 + ue;
                    // the largest x: when the largest exponential and the largest scale sit on
                    // different entries it can fall far below 128; then x goes up by 2^j (and
                    // S down) so that it lies in [128, 256) again
                    float x[32];
#pragma unroll
                    for (int t = 0; t < 32; ++t) x[t] = e[t] * us[t];
                    const float xm = max32(x);
                    bool live = bm > -INFINITY && xm > 0.0f;
                    if (live && xm < 32.0f) {
                        const int eb = (int)(__float_as_uint(xm) >> 23);  // xm > 0
                        const int j = 134 - eb;                           // 2^j xm in [128, 256)
                        if (eb >= 7) {
                            const float up = __uint_as_float((uint32_t)(127 + j) << 23);
#pragma unroll
                            for (int t = 0; t < 32; ++t) x[t] *= up;
                            S -= j;
                        } else {
                            live = false;  // below 2^-120 of the reference
                        }
                    }
                    if (live && S >= -127 && S <= 127) {
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            uint32_t hw = 0, lw = 0;
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const float x0 = x[4 * w + 2 * h2];
                                const float x1 = x[4 * w + 2 * h2 + 1];
                                uint32_t xh, hh, rh;
                                uint16_t h8, l8;
                                asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(xh) : "f"(x1), "f"(x0));
                                asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h8) : "r"(xh));
                                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(h8));
                                // the rest, exact in fp16 (under half a spacing of h)
                                asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(rh) : "r"(xh), "r"(hh));
                                asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l8) : "r"(rh));
                                hw |= (uint32_t)h8 << (16 * h2);
                                lw |= (uint32_t)l8 << (16 * h2);
                            }
                            packed[q][w] = hw;
                            packed[q][8 + w] = lw;
                        }
                        sf_word[q] = (uint32_t)(127 + S) * 0x01010101u;
                    } else {
                        // nothing in the slice, or a block far under the reference: zero
#pragma unroll
                        for (int w = 0; w < 16; ++w) packed[q][w] = 0u;
                        sf_word[q] = 0x7F7F7F7Fu;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        e[4 * c + 0] = ex2_approx(fmaf(v[c].x, kLog2e, neg_lse2[q]));
                        e[4 * c + 1] = ex2_approx(fmaf(v[c].y, kLog2e, neg_lse2[q]));
                        e[4 * c + 2] = ex2_approx(fmaf(v[c].z, kLog2e, neg_lse2[q]));
                        e[4 * c + 3] = ex2_approx(fmaf(v[c].w, kLog2e, neg_lse2[q]));
                    }
                    if (edge) {  // a block that straddles an end of the slice (warp-uniform, rare)
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (k + t < p.vocab_start || k + t >= p.vocab_end) e[t] = 0.f;
                    }
#pragma unroll
                    for (int t = 0; t < 16; ++t) packed[q][t] = pack_bf16x2(e[2 * t], e[2 * t + 1]);
                    sf_word[q] = 0u;
                    bmq[q] = 0.0f;
                    kfq[q] = 0.0f;
                }
#pragma unroll
                for (int t = 0; t < 32; ++t) ek[q][t] = e[t];
            }
            // the A slot is free once the MMAs of its previous round are done
            if (u > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[s]), (u - 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            uint8_t *at = a_ring + s * A_SLOT;
            uint8_t *sft = sf_ring + s * Fmt<kE4m3>::SF_STAGE;  // 8-bit table
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q) {
                const int r = rr[q];
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {  // 16-byte chunk of the 64-byte A row
                    const uint4 w = make_uint4(packed[q][4 * c8], packed[q][4 * c8 + 1], packed[q][4 * c8 + 2],
                                               packed[q][4 * c8 + 3]);
                    *reinterpret_cast<uint4 *>(at + r * 64 + ((c8 ^ ((r >> 1) & 3)) << 4)) = w;
                }
                // the scale word of row r: word r / 32 of 16-byte row r, which the MMA thread
                // copies into TMEM lane r (the MMA reads lane r's scale from column r / 32)
                if constexpr (F == kE4m3) reinterpret_cast<uint32_t *>(sft)[4 * r + (r >> 5)] = sf_word[q];
            }
            fence_proxy_async_smem();
            __syncwarp();  // every lane's A stores (and proxy fence) before the arrival
            if (lane == 0) {
                if (rank & 1) {
                    // the pair's even CTA's MMA thread reads this CTA's rows (and scale rows) too:
                    // a 16-byte copy that completes on its barrier tells it this warp's rows are
                    // in place (issued after the rows' stores and proxy fence; never read)
                    const uint32_t lead = rank & ~1u;
                    bulk_copy_to_cluster(map_to_cta(smem_u32(sig_area + 16 * (1 + pw)), lead), smem_u32(sig_area),
                                         16u, map_to_cta(smem_u32(&full_a[s]), lead));
                } else {
                    mbar_arrive(smem_u32(&full_a[s]));
                }
                // the warp's 32 A rows (2 KiB; 8-bit table: and its 32 scale rows, 512 B) to the
                // same slot of the CTA with the same rows in the other column tile, completing on
                // its full_a
                const uint32_t twin = rank ^ 2u;
                const uint32_t tbar = map_to_cta(smem_u32(&full_a[s]), twin);
                const uint32_t a_src = smem_u32(at + wig * 2048);
                bulk_copy_to_cluster(map_to_cta(a_src, twin), a_src, 2048u, tbar);
                if constexpr (F == kE4m3) {
                    const uint32_t f_src = smem_u32(sft + wig * 512);
                    bulk_copy_to_cluster(map_to_cta(f_src, twin), f_src, 512u, tbar);
                }
            }
            if (fold) {
#pragma unroll
                for (int q = 0; q < ROWS_PER_LANE; ++q) {
                    // the block's statistics from the probabilities' own exponentials e = exp(l - c)
                    // (bf16 table: sums against c, RefState; 8-bit table: a block summary relative
                    // to the block max bm, exp(l - bm) = e exp(c - bm)).  A block whose max lies
                    // more than 60 nats above c (e may overflow) takes the statistics kernel's fold
                    // instead.  Entries that underflow in e lie more than 87 nats below c, so below
                    // every row maximum by as much: they add nothing the fp32 statistics could hold.
                    float xb[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        xb[4 * c + 0] = vk[q][c].x;
                        xb[4 * c + 1] = vk[q][c].y;
                        xb[4 * c + 2] = vk[q][c].z;
                        xb[4 * c + 3] = vk[q][c].w;
                    }
                    if (edge) {
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (k + t < p.vocab_start || k + t >= p.vocab_end) xb[t] = -INFINITY;
                    }
                    float bm = bmq[q];  // the 8-bit path's block maximum
                    if constexpr (F == kBf16) bm = max32(xb);
                    rowstate::RowState blk = rowstate::empty_row_state();
                    float glm[2] = {-INFINITY, -INFINITY};  // the two groups' log-masses
                    if (F == kE4m3 && bm > -INFINITY) {
                        // the 8-bit path's exponentials e'' = exp(l - bm) 2^(7 + f), f the
                        // fraction (bm - c) log2 e - k: the summary takes them times 2^-(7 + f)
                        int ja = 31;
#pragma unroll
                        for (int t = 31; t >= 0; --t)
                            if (xb[t] == bm) ja = t;
                        float se = 0.0f, sd = 0.0f;
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            se += t == ja ? 0.0f : ek[q][t];
                            sd = fmaf(ek[q][t], fmaxf(xb[t] - bm, -FLT_MAX), sd);
                        }
                        const float f = fmaf(bm, kLog2e, neg_lse2[q]) - kfq[q];
                        const float inv = ex2_approx(-7.0f - f);
                        blk = rowstate::RowState{bm, (int)(k + ja), se * inv, sd * inv};
                        if (p.draw && p.inv_tau == 1.0f) {  // c + ln(sum of exp(l - c)) = c + ln 2 (log2(sum e'') + k - 7)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                float gsum = 0.0f;
#pragma unroll
                                for (int t = 0; t < 16; ++t) gsum += ek[q][16 * h + t];
                                glm[h] = my_ref[q] + philox::kLn2 * (__log2f(gsum) + kfq[q] - 7.0f);
                            }
                        }
                    } else if (F == kBf16 && bm > -INFINITY && bm - my_ref[q] <= 60.0f) {
                        // the block's sums against c (see RefState); a block with a masked (-inf)
                        // entry gets NaN from 0 * -inf in the first sum of e (l - c) and takes the
                        // guarded one
                        const float *ev = ek[q];
                        const float s_lo = sum16(ev), s_hi = sum16(ev + 16);
                        const float S = s_lo + s_hi;
                        float tx[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int t = 0; t < 32; ++t) tx[t & 3] = fmaf(ev[t], xb[t], tx[t & 3]);
                        float Tx = (tx[0] + tx[1]) + (tx[2] + tx[3]);
                        if (Tx != Tx) {
                            Tx = 0.0f;
#pragma unroll
                            for (int t = 0; t < 32; ++t) Tx = fmaf(ev[t], fmaxf(xb[t], -FLT_MAX), Tx);
                        }
                        RefState &rs = my_rs[q];
                        if (bm > rs.M) {
                            // a new maximum: its first occurrence leaves the sum, the old one enters it
                            int ja = 31;
#pragma unroll
                            for (int t = 31; t >= 0; --t)
                                if (xb[t] == bm) ja = t;
                            float se = 0.0f;
#pragma unroll
                            for (int t = 0; t < 32; ++t) se += t == ja ? 0.0f : ev[t];
                            rs.R16 += rs.E + se;
                            // e of the new maximum, formed exactly as the producers formed ev[ja]
                            rs.E = ex2_approx(fmaf(bm, kLog2e, neg_lse2[q]));
                            rs.M = bm;
                            rs.A = (int)(k + ja);
                        } else {
                            rs.R16 += S;  // equal maxima keep the earlier index
                        }
                        rs.T16 += fmaf(-my_ref[q], S, Tx);
                        if (p.draw && p.inv_tau == 1.0f) {  // the two groups' log-masses, c + ln(sum of e)
                            glm[0] = my_ref[q] + philox::kLn2 * __log2f(s_lo);
                            glm[1] = my_ref[q] + philox::kLn2 * __log2f(s_hi);
                        }
                    } else if (F == kBf16 && bm > -INFINITY) {
                    // far above c: the statistics kernel's fold over this row's 32 entries, in two halves
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float xs[16];
                        int bs[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float4 w = vk[q][4 * h + c];
                            bs[c] = (int)((k >> 2) + 4 * h + c);
                            xs[4 * c + 0] = w.x;
                            xs[4 * c + 1] = w.y;
                            xs[4 * c + 2] = w.z;
                            xs[4 * c + 3] = w.w;
                        }
                        if (edge) {
#pragma unroll
                            for (int t = 0; t < 16; ++t)
                                if (k + 16 * h + t < p.vocab_start || k + 16 * h + t >= p.vocab_end) xs[t] = -INFINITY;
                        }
                        rowstate::absorb<16>(blk, xs, bs);
                    }
                    if (p.draw && p.inv_tau == 1.0f) {  // far from c: the log-masses against the block max
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float gsum = 0.0f;
#pragma unroll
                            for (int t = 0; t < 16; ++t) gsum += ex2_approx((xb[16 * h + t] - bm) * kLog2e);
                            glm[h] = bm + philox::kLn2 * __log2f(gsum);
                        }
                    }
                    }
                    if (p.draw && p.inv_tau != 1.0f && bm > -INFINITY) {
                        // another temperature: the two groups' log-masses of l / T, against the
                        // block maximum (entries at -inf add nothing)
                        const float sl = kLog2e * p.inv_tau;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float gsum = 0.0f;
#pragma unroll
                            for (int t = 0; t < 16; ++t) gsum += ex2_approx((xb[16 * h + t] - bm) * sl);
                            glm[h] = bm * p.inv_tau + philox::kLn2 * __log2f(gsum);
                        }
                    }
                    rowstate::merge(my_st16[q], blk);
                    if (p.draw && bm > -INFINITY) {
                        // groups k/16 and k/16 + 1 (k is a multiple of 32): words of one Philox block
                        const int g0 = (int)(k >> 4);
                        const philox::Philox w = philox::philox4x32_10(philox::kGroupCounter + (uint32_t)(g0 >> 2),
                                                                       (uint32_t)(row0 + rr[q]), p.o0, p.o1, p.k0,
                                                                       p.k1);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const float sc =
                                glm[h] - philox::kLn2 * __log2f(philox::neg_log_uniform(philox::philox_word(w, (g0 + h) & 3)));
                            if (sc > my_gbest[q]) {  // groups arrive in increasing order: ties keep the lower
                                my_gbest[q] = sc;
                                my_gidx[q] = g0 + h;
                            }
                        }
                    }
                }
                if (++my_folded % 16 == 0) {
#pragma unroll
                    for (int q = 0; q < ROWS_PER_LANE; ++q) {
                        rowstate::merge(my_st[q], my_st16[q]);
                        my_st16[q] = rowstate::empty_row_state();
                        my_rs[q].R += my_rs[q].R16;
                        my_rs[q].T += my_rs[q].T16;
                        my_rs[q].R16 = 0.0f;
                        my_rs[q].T16 = 0.0f;
                    }
                }
            }
        }
        if (p.fused)
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q) {
                rowstate::merge(my_st[q], my_st16[q]);
                if constexpr (F == kBf16) rowstate::merge(my_st[q], ref_to_row_state(my_rs[q], my_ref[q]));
            }
    }

    // threads without a role in the main loop (lanes 1-31 of the single-thread roles, and
    // the bf16 kernel's warp 0) and roles whose wait came last
    grid_dependency_wait();
    grid_launch_dependents();
    // ---------------------------------------------------------------- epilogue (all warps)
    // accumulator -> partial tile, layout [BN/4 column groups][128 rows][4]; a warp reads the
    // TMEM lane quarter of its scheduler, the three warps of a quarter one third of the columns each
    __syncwarp();
    {
        const int quarter = warp & 3;
        const int third = warp >> 2;
        const int r = quarter * 32 + lane;
        float4 *dst = reinterpret_cast<float4 *>(p.ws) +
                      ((int64_t)(j * p.m_tiles + mt) * p.n_tiles + nt) * (BN / 4) * BM;
        const int nch = halves == 2 ? BN / 32 : 8;  // 32-column chunks of this tile
        const int c_lo = third * nch / 3, c_hi = (third + 1) * nch / 3;
        // tcgen05.ld is warp-collective: the warp goes on only if every lane got here cleanly
        bool have_acc = false;
        if (nkb > 0 && __all_sync(0xffffffffu, ok)) {
            const bool got = mbar_wait(smem_u32(acc_full), 0, abort_flag);
            have_acc = __all_sync(0xffffffffu, got);
        }
        if (have_acc) {
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int jc = c_lo; jc < c_hi; ++jc) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(trow + jc * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 o = make_float4(__uint_as_float(v[4 * c4]), __uint_as_float(v[4 * c4 + 1]),
                                                 __uint_as_float(v[4 * c4 + 2]), __uint_as_float(v[4 * c4 + 3]));
                    dst[(jc * 8 + c4) * BM + r] = o;
                }
            }
        } else if (nkb == 0) {
            for (int cg4 = c_lo * 8; cg4 < c_hi * 8; ++cg4) dst[cg4 * BM + r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (p.fused) {
        // single pass: merge the producer groups' row states in group order (the A ring is
        // idle: every MMA has completed or been drained), write the summary of this tile's
        // share of the split's blocks per row, and (column tile 0) the reference
        rowstate::RowState *scratch = reinterpret_cast<rowstate::RowState *>(a_ring);
        float2 *dscratch = reinterpret_cast<float2 *>(a_ring + 8192);  // after (PGROUPS - 1) x 2 KiB of states
        if (my_grp > 0)
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q) {
                scratch[(my_grp - 1) * BM + my_rows[q]] = my_st[q];
                dscratch[(my_grp - 1) * BM + my_rows[q]] = make_float2(my_gbest[q], __int_as_float(my_gidx[q]));
            }
        __syncthreads();
        if (my_grp == 0 && !*abort_flag) {
#pragma unroll
            for (int q = 0; q < ROWS_PER_LANE; ++q) {
                const int row = row0 + my_rows[q];
                if (row >= p.R) continue;
                rowstate::RowState st = my_st[q];
                for (int g = 1; g < PGROUPS; ++g) rowstate::merge(st, scratch[(g - 1) * BM + my_rows[q]]);
                const int a = st.m == -INFINITY ? 0x7fffffff : st.a;
                p.state[((int64_t)j * p.n_tiles + nt) * p.R + row] = make_float4(st.m, __int_as_float(a), st.rest, st.t);
                if (nt == 0) p.ref[(int64_t)j * p.R + row] = my_ref[q];
                if (p.draw) {
                    float best = my_gbest[q];
                    int gi = my_gidx[q];
                    for (int g = 1; g < PGROUPS; ++g) {
                        const float2 o = dscratch[(g - 1) * BM + my_rows[q]];
                        const int oi = __float_as_int(o.y);
                        if (o.x > best || (o.x == best && oi < gi)) {
                            best = o.x;
                            gi = oi;
                        }
                    }
                    p.draws[((int64_t)j * p.n_tiles + nt) * p.R + row] = make_float2(best, __int_as_float(gi));
                }
            }
        }
    }
    // neither CTA leaves while the other may still copy into it or commit to it
    cluster_sync_all();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair<TMEM_COLS>(tmem_base);
    }
}

// Single pass, the rare (split, row) pairs whose reference was too far from their maximum
// (scale kRedo): the split's partial for row i and columns c .. c + 3, recomputed on the CUDA
// cores against lse (fp32, vocabulary in order).
template <int F>
__device__ float4 redo_partial(const Params &p, const void *__restrict__ Wv, int64_t ldw, int d, float lse_i,
                               int j, int i, int c) {
    int64_t kb0, kb1;
    split_range(p, j, p.splits, &kb0, &kb1);
    int64_t v0 = p.k_begin + kb0 * BK, v1 = p.k_begin + kb1 * BK;
    if (v0 < p.vocab_start) v0 = p.vocab_start;
    if (v1 > p.vocab_end) v1 = p.vocab_end;
    const float l2 = lse_i * kLog2e;
    const float *lrow = p.logits + (int64_t)i * p.ldl;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t v = v0; v < v1; ++v) {
        const float pv = ex2_approx(fmaf(lrow[v], kLog2e, -l2));
        if constexpr (F == kE4m3) {
            const uint8_t *wr = static_cast<const uint8_t *>(Wv) + (v - p.vocab_start) * ldw + c;
            const float ps = pv * p.w_scale[v - p.vocab_start];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (c + t < d) acc[t] = fmaf(ps, e4m3_to_f32(wr[t]), acc[t]);
        } else {
            const uint16_t *wr = static_cast<const uint16_t *>(Wv) + (v - p.vocab_start) * ldw + c;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (c + t < d) acc[t] = fmaf(pv, __uint_as_float((uint32_t)wr[t] << 16), acc[t]);
        }
    }
    return make_float4(acc[0], acc[1], acc[2], acc[3]);
}

// E[i, c] = gamma * sum over the splits of column c's tile, in split order.
// Single pass (scale given): each split's partial is scaled by f[split][row] = exp(c - lse)
// first, and a pair marked kRedo is recomputed (redo_partial) and taken with scale 1; the
// first n_acc CTAs run the acceptance of request blockIdx.x on the statistics instead (they
// need blockDim.x >= the acceptance's threads and its keys in dynamic shared memory).
template <int F>
__global__ void __launch_bounds__(1024) splitk_reduce_kernel(const float4 *__restrict__ ws, const Params p, int d, float gamma,
                                     float *__restrict__ out, int64_t ldo, int vec_out,
                                     const float *__restrict__ scale, const void *__restrict__ Wv, int64_t ldw,
                                     const float *__restrict__ lse, const AcceptSpec acc, int n_acc,
                                     const LoopSpec loop) {
    constexpr int BN = Fmt<F>::BN;
    // the kernel queued next reads nothing this one writes; this one reads the partials and
    // the statistics only after the kernel before it (the single pass's statistics) completed
    grid_launch_dependents();
    grid_dependency_wait();
    if ((int)blockIdx.x < n_acc) {
        extern __shared__ unsigned long long keys[];
        __shared__ float H_s[1024];
        __shared__ double warp_tot[32];
        __shared__ int first_fail;
        accept_request(acc, (int)blockIdx.x, blockDim.x, AcceptSmem{keys, H_s, warp_tot, &first_fail});
        if (loop.canvas) {
            __syncthreads();  // the request's mask written, warp_tot free again
            loop_update_request(loop, (int)blockIdx.x, warp_tot);
        }
        return;
    }
    const int64_t groups = ((int64_t)d + 3) / 4;  // column groups of 4
    const int64_t total = (int64_t)p.R * groups;
    const int64_t tile_elems = (int64_t)(BN / 4) * BM;  // float4 per partial tile
    const int64_t nthreads = (int64_t)(gridDim.x - n_acc) * blockDim.x;
    for (int64_t t = (blockIdx.x - n_acc) * (int64_t)blockDim.x + threadIdx.x; t < total; t += nthreads) {
        // consecutive threads take consecutive rows of one column group: coalesced reads
        const int64_t g = t / p.R;
        const int i = (int)(t - g * p.R);
        const int c = (int)(g * 4);
        const int mt = i / BM, r = i % BM;
        const int nt = c / BN, cg = (c % BN) / 4;
        const int S = nt < p.n_full ? p.splits : p.tail_splits;
        const int64_t split_stride = (int64_t)p.m_tiles * p.n_tiles * tile_elems;
        const float4 *src = ws + ((int64_t)mt * p.n_tiles + nt) * tile_elems + (int64_t)cg * BM + r;
        // the partials (and scales) of kRedBatch splits loaded together, clamped to the last
        // split so that every load is unconditional, then added strictly in split order
        constexpr int kRedBatch = 6;
        float4 acc4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int s0 = 0; s0 < S; s0 += kRedBatch) {
            float4 v[kRedBatch];
            float f[kRedBatch];
#pragma unroll
            for (int q = 0; q < kRedBatch; ++q) {
                const int sq = min(s0 + q, S - 1);
                v[q] = src[sq * split_stride];
                f[q] = scale ? scale[(int64_t)sq * p.R + i] : 1.0f;
            }
            bool redo = false;
#pragma unroll
            for (int q = 0; q < kRedBatch; ++q) redo |= f[q] < 0.0f;
            if (!redo) {
#pragma unroll
                for (int q = 0; q < kRedBatch; ++q) {
                    if (s0 + q >= S) break;
                    acc4.x = fmaf(f[q], v[q].x, acc4.x);
                    acc4.y = fmaf(f[q], v[q].y, acc4.y);
                    acc4.z = fmaf(f[q], v[q].z, acc4.z);
                    acc4.w = fmaf(f[q], v[q].w, acc4.w);
                }
            } else {
                // a (split, row) to recompute (rare): the batch again, one split at a time
#pragma unroll 1
                for (int sq = s0; sq < S && sq < s0 + kRedBatch; ++sq) {
                    float4 vq = src[sq * split_stride];
                    float fq = scale[(int64_t)sq * p.R + i];
                    if (fq < 0.0f) {
                        vq = redo_partial<F>(p, Wv, ldw, d, lse[i], sq, i, c);
                        fq = 1.0f;
                    }
                    acc4.x = fmaf(fq, vq.x, acc4.x);
                    acc4.y = fmaf(fq, vq.y, acc4.y);
                    acc4.z = fmaf(fq, vq.z, acc4.z);
                    acc4.w = fmaf(fq, vq.w, acc4.w);
                }
            }
        }
        float *o = out + (int64_t)i * ldo + c;
        if (vec_out && c + 4 <= d) {
            *reinterpret_cast<float4 *>(o) =
                make_float4(gamma * acc4.x, gamma * acc4.y, gamma * acc4.z, gamma * acc4.w);
        } else {
            const float a4[4] = {acc4.x, acc4.y, acc4.z, acc4.w};
            for (int e = 0; e < 4 && c + e < d; ++e) o[e] = gamma * a4[e];
        }
    }
}

// Single pass, after the product: per row (one warp), lane l merges the tile summaries of
// splits l, l + 32, ... (tile order), checks each split's maximum against its reference
// (a pair whose probabilities could overflow gets the scale kRedo, and the reduce recomputes
// it), the lanes' states merge in a fixed shuffle tree, lane 0 writes the statistics, and
// each split's reference becomes its scale exp(c - lse).
__global__ void __launch_bounds__(256)
    single_pass_stats_kernel(const Params p, float *__restrict__ out_m, float *__restrict__ out_lse,
                             float *__restrict__ out_H, float *__restrict__ out_kappa,
                             int32_t *__restrict__ out_argmax) {
    // launched to overlap the product's tail: the summaries are read after it completes
    grid_dependency_wait();
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= p.R) return;  // warp-uniform
    rowstate::RowState st = rowstate::empty_row_state();
    float dbest = -INFINITY;  // the draw's first level: best group score and group
    int dgrp = 0x7fffffff;
    uint32_t redo_bits = 0;  // bit k: split lane + 32 k is recomputed by the reduce
    for (int s = lane, kk = 0; s < p.splits; s += 32, ++kk) {
        rowstate::RowState sp = rowstate::empty_row_state();
        const float c = p.ref[(int64_t)s * p.R + row];
        // eight tiles' summaries in flight at once (unconditional loads: past the last tile
        // they repeat it), then merged in tile order
        for (int t0 = 0; t0 < p.n_tiles; t0 += 8) {
            float4 v[8];
            float2 dv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t at = ((int64_t)s * p.n_tiles + min(t0 + u, p.n_tiles - 1)) * p.R + row;
                v[u] = p.state[at];
                dv[u] = p.draw ? p.draws[at] : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (t0 + u < p.n_tiles) {
                    rowstate::merge(sp, rowstate::RowState{v[u].x, __float_as_int(v[u].y), v[u].z, v[u].w});
                    if (p.draw) {
                        const int gi = __float_as_int(dv[u].y);
                        if (dv[u].x > dbest || (dv[u].x == dbest && gi < dgrp)) {
                            dbest = dv[u].x;
                            dgrp = gi;
                        }
                    }
                }
        }
        // the split's probabilities against its reference: ln of their sum is
        // (m - c) + ln Z_split; list the pair for the redo pass if they could overflow
        const float gap = sp.m - c;
        if (sp.m > -INFINITY && !(gap + log1pf(sp.rest) <= kRefSumLog && gap >= -kRefBelow))
            redo_bits |= 1u << kk;
        rowstate::merge(st, sp);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        rowstate::merge(st, rowstate::shfl_down(st, off));
        const float ob = __shfl_down_sync(0xffffffffu, dbest, off);
        const int og = __shfl_down_sync(0xffffffffu, dgrp, off);
        if (ob > dbest || (ob == dbest && og < dgrp)) {
            dbest = ob;
            dgrp = og;
        }
    }
    float lse = __int_as_float(0x7fc00000), H = lse, kappa = lse;
    int a = 0;
    if (lane == 0 && st.m != -INFINITY) {
        const float lnZ = log1pf(st.rest);
        lse = st.m + lnZ;
        H = lnZ - st.t / (1.0f + st.rest);
        kappa = lnZ;
        a = st.a;
    }
    lse = __shfl_sync(0xffffffffu, lse, 0);
    const float m = __shfl_sync(0xffffffffu, st.m, 0);
    for (int s = lane, kk = 0; s < p.splits; s += 32, ++kk) {
        float *r = p.ref + (int64_t)s * p.R + row;
        // c <= m <= lse: at most 1; a row without a distribution gets NaN, as in the two-pass step
        *r = m == -INFINITY          ? __int_as_float(0x7fc00000)
             : (redo_bits >> kk) & 1u ? kRedo
                                      : ex2_approx((*r - lse) * kLog2e);
    }
    if (p.draw) {
        // the second level: lanes 0-15 draw inside the chosen group (temperature 1); kappa
        // becomes -ln p of the drawn token
        const int gs = __shfl_sync(0xffffffffu, dgrp, 0);
        const int64_t v = (int64_t)16 * gs + lane;
        const bool valid = gs != 0x7fffffff && lane < 16 && v < p.vocab_end;
        const float l = valid ? p.logits[row * p.ldl + v] : -INFINITY;
        float sc = -INFINITY;
        if (valid && l != -INFINITY) {
            const philox::Philox w = philox::philox4x32_10((uint32_t)(v >> 2), (uint32_t)row, p.o0, p.o1, p.k0, p.k1);
            sc = l * p.inv_tau - philox::kLn2 * __log2f(philox::neg_log_uniform(philox::philox_word(w, (int)(v & 3))));
        }
        int bi = valid ? (int)v : 0x7fffffff;
        float bl = l;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float os = __shfl_down_sync(0xffffffffu, sc, off);
            const int oi = __shfl_down_sync(0xffffffffu, bi, off);
            const float ol = __shfl_down_sync(0xffffffffu, bl, off);
            if (os > sc || (os == sc && oi < bi)) {
                sc = os;
                bi = oi;
                bl = ol;
            }
        }
        if (lane == 0) {
            const bool drawn = st.m != -INFINITY && sc > -INFINITY;
            p.candidate[row] = drawn ? bi : 0;
            const float lnZ = kappa;  // ln Z (NaN without a distribution)
            kappa = !drawn ? __int_as_float(0x7fc00000) : (bi == a ? lnZ : (st.m - bl) + lnZ);
        }
    }
    if (lane == 0) {
        if (out_m) out_m[row] = st.m;
        if (out_lse) out_lse[row] = lse;
        if (out_H) out_H[row] = H;
        if (out_kappa) out_kappa[row] = kappa;
        if (out_argmax) out_argmax[row] = a;
    }
}

// A vocabulary shard's first call, after the single pass's product: per row (one warp) the
// splits' tile summaries merged as single_pass_stats_kernel merges them, written as the
// shard's 16-byte row summary (m, argmax as vocab_offset + column, rest, t: the format of
// dg_row_stats_partial), and each split whose probabilities against its reference could
// overflow marked for the second call (its reference becomes +inf).
__global__ void __launch_bounds__(256)
    shard_summary_kernel(const Params p, float4 *__restrict__ out_state, int64_t vocab_offset) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= p.R) return;  // warp-uniform
    rowstate::RowState st = rowstate::empty_row_state();
    for (int s = lane; s < p.splits; s += 32) {
        rowstate::RowState sp = rowstate::empty_row_state();
        float *ref = p.ref + (int64_t)s * p.R + row;
        const float c = *ref;
        for (int t0 = 0; t0 < p.n_tiles; t0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = p.state[((int64_t)s * p.n_tiles + min(t0 + u, p.n_tiles - 1)) * p.R + row];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (t0 + u < p.n_tiles)
                    rowstate::merge(sp, rowstate::RowState{v[u].x, __float_as_int(v[u].y), v[u].z, v[u].w});
        }
        const float gap = sp.m - c;
        if (sp.m > -INFINITY && !(gap + log1pf(sp.rest) <= kRefSumLog && gap >= -kRefBelow)) *ref = INFINITY;
        rowstate::merge(st, sp);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) rowstate::merge(st, rowstate::shfl_down(st, off));
    if (lane == 0) {
        const int a = st.m == -INFINITY ? 0x7fffffff : (int)(st.a + vocab_offset);
        out_state[row] = make_float4(st.m, __int_as_float(a), st.rest, st.t);
    }
}

// A vocabulary shard's second call: each split's reference becomes its scale exp(c - lse) against
// the full-row lse (NaN for a row without a distribution), or kRedo where the first call marked it.
__global__ void __launch_bounds__(256) shard_scale_kernel(const Params p, const float *__restrict__ lse) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)p.splits * p.R) return;
    const int64_t row = idx % p.R;
    const float c = p.ref[idx];
    p.ref[idx] = c == INFINITY ? kRedo : ex2_approx((c - lse[row]) * kLog2e);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

constexpr int kMaxAttrDevices = 64;

int tile_width(int fmt) { return fmt == kE4m3 ? Fmt<kE4m3>::BN : Fmt<kBf16>::BN; }

// Column tiling of d: n_full tiles of bn columns (two MMA halves), then (if tail) one of
// <= 256 (the first half alone).
void column_tiles(int64_t d, int bn, int *n_tiles, int *n_full, int *tail) {
    const int nt = (int)((d + bn - 1) / bn);
    const int64_t last = d - (int64_t)(nt - 1) * bn;
    *n_tiles = nt;
    *tail = last <= 256 ? 1 : 0;
    *n_full = nt - *tail;
}

// A block costs about the same time whatever its width (the stage round trip, not the
// bytes, sets the pace), so the half-width tail gets as many splits as the full tiles.
int tail_splits_of(int splits, int tail) { return tail ? splits : 0; }

}  // namespace

size_t soft_embed_workspace_bytes(const SoftEmbedPlan &plan, int splits) {
    return (size_t)splits * (size_t)plan.m_tiles * (size_t)plan.n_tiles * BM * (size_t)plan.bn * sizeof(float);
}

// The single pass's extra workspace, after the partial tiles: references / scales
// [splits][R] fp32, summaries [splits][n_tiles][R] x 16 B, the draw's first level
// [splits][n_tiles][R] x 8 B.
static size_t align16(size_t b) { return (b + 15) & ~size_t(15); }
size_t single_pass_extra_bytes(const SoftEmbedPlan &plan, int64_t R) {
    const size_t n = (size_t)plan.splits * (size_t)R;
    return align16(n * 4) + n * (size_t)plan.n_tiles * 16 + n * (size_t)plan.n_tiles * 8;
}

// The product kernels' shared-memory limit, raised once per device (a function attribute
// belongs to the device's context; setting it twice from racing threads is harmless).
static cudaError_t ensure_kernel_attributes() {
    static std::atomic<int> attr_set[kMaxAttrDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < kMaxAttrDevices && attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(soft_embed_kernel<kBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<kBf16>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(soft_embed_kernel<kE4m3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes<kE4m3>());
    if (e == cudaSuccess && dev < kMaxAttrDevices) attr_set[dev].store(1, std::memory_order_release);
    return e;
}

// Clusters of the product (four CTAs) for a table format that fit on the current device at
// once (36 on a 152-SM GB300: whole clusters must sit in one GPC), looked up once per device.
static int quad_clusters_per_wave(int fmt, int num_sms) {
    static std::atomic<int> cached[2][kMaxAttrDevices];
    const int f = fmt == kE4m3 ? 1 : 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return num_sms / kQuadCtas;
    if (dev < kMaxAttrDevices) {
        const int c = cached[f][dev].load(std::memory_order_acquire);
        if (c > 0) return c;
    }
    int n = 0;
    if (ensure_kernel_attributes() == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kQuadCtas * 64, 1, 1);
        cfg.blockDim = dim3(THREADS, 1, 1);
        cfg.dynamicSmemBytes = f ? smem_bytes<kE4m3>() : smem_bytes<kBf16>();
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = kQuadCtas;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        const void *fn = f ? (const void *)soft_embed_kernel<kE4m3> : (const void *)soft_embed_kernel<kBf16>;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    }
    if (n <= 0) n = num_sms / kQuadCtas;
    if (dev < kMaxAttrDevices) cached[f][dev].store(n, std::memory_order_release);
    return n;
}

bool plan_soft_embed(int64_t R, int64_t vocab_start, int64_t vocab_end, int64_t d, int num_sms,
                     SoftEmbedPlan *plan, int fmt) {
    if (R <= 0 || d <= 0 || vocab_end <= vocab_start || vocab_start < 0 || num_sms < 2) return false;
    if (fmt != kBf16 && fmt != kE4m3) return false;
    SoftEmbedPlan pl;
    pl.fmt = fmt;
    pl.bn = tile_width(fmt);
    pl.k_begin = vocab_start & ~int64_t(3);
    pl.nkb = (vocab_end - pl.k_begin + BK - 1) / BK;
    int64_t m_pairs = (R + 2 * BM - 1) / (2 * BM);  // 256-row blocks
    pl.m_tiles = (int)(2 * m_pairs);
    int n_full, tail;
    column_tiles(d, pl.bn, &pl.n_tiles, &n_full, &tail);
    // clusters of two column tiles and both 128-row halves of a 256-row block: an even tile
    // count, a last odd tile's partner past d
    pl.n_tiles += pl.n_tiles & 1;
    const int64_t clusters = quad_clusters_per_wave(fmt, num_sms);
    n_full = pl.n_tiles / 2;  // units per split and row block: column pairs
    tail = 0;
    // choose the vocabulary splits that finish soonest: whole waves of clusters times
    // the largest per-cluster work (vocabulary blocks)
    int best = 1;
    double best_t = 1e300;
    // at least 16 blocks (four rounds of the stage ring) per split, at most 64 splits
    int64_t max_s = pl.nkb / 16;
    if (max_s > 64) max_s = 64;
    if (max_s < 1) max_s = 1;
    for (int64_t S = 1; S <= max_s; ++S) {
        const int64_t St = tail_splits_of((int)S, tail);
        const int64_t pairs = m_pairs * (n_full * S + St);
        const double waves = (double)((pairs + clusters - 1) / clusters);
        // every cluster costs its number of vocabulary blocks
        double work = (double)((pl.nkb + S - 1) / S);
        if (St) work = fmax(work, (double)((pl.nkb + St - 1) / St));
        const double t = waves * (work + 32.0);  // a wave also pays its pipeline fill and epilogue
        if (t < best_t * 0.98) {
            best_t = t;
            best = (int)S;
        }
    }
    pl.splits = best;
    pl.workspace_bytes = soft_embed_workspace_bytes(pl, pl.splits);
    pl.single_pass_bytes = pl.workspace_bytes + single_pass_extra_bytes(pl, R);
    *plan = pl;
    return true;
}

cudaError_t launch_soft_embed(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t vocab_start,
                              int64_t vocab_end, const EmbedTable &tab, int64_t d, float gamma, float *out,
                              int64_t ldo, void *workspace, const SoftEmbedPlan &plan, cudaStream_t stream,
                              const char **msg, StreamHook between, void *ctx, bool overlap_previous,
                              const SinglePassOut *single) {
    if (tab.fmt != plan.fmt) {
        *msg = "soft embed: the plan was made for another table format";
        return cudaErrorInvalidValue;
    }
    const bool e4 = tab.fmt == kE4m3;
    const int64_t ldw = tab.ldw;
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode) {
        *msg = "cuTensorMapEncodeTiled is not available from the driver";
        return cudaErrorNotSupported;
    }
    CUtensorMap tm_l, tm_w, tm_w4;
    memset(&tm_w4, 0, sizeof(tm_w4));
    int w4d_atoms = 0;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)vocab_end, (cuuint64_t)R};
        const cuuint64_t strides[1] = {(cuuint64_t)ldl * 4};
        const cuuint32_t box[2] = {BK, BM};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_l, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(logits), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *msg = "tensor map of the logits could not be encoded";
            return cudaErrorInvalidValue;
        }
    }
    // W (bf16): a 3-D view (64 columns of an atom, rows, atoms 128 bytes apart) when every
    // atom's 64 columns lie inside the row pitch, else 2-D boxes of 64 columns.
    // W (E4M3): 2-D boxes of 128 columns.
    int w3d = 0;
    const int64_t atoms = (d + 63) / 64;
    const uint16_t *W = static_cast<const uint16_t *>(tab.W);
    if (e4) {
        const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)(vocab_end - vocab_start)};
        const cuuint64_t strides[1] = {(cuuint64_t)ldw};
        const cuuint32_t box[2] = {128, (cuuint32_t)BK};  // one 128-column atom of a block
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(tab.W), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *msg = "tensor map of the 8-bit embedding shard could not be encoded";
            return cudaErrorInvalidValue;
        }
    } else if (atoms * 64 <= ldw) {
        const cuuint64_t dims[3] = {64, (cuuint64_t)(vocab_end - vocab_start), (cuuint64_t)atoms};
        const cuuint64_t strides[2] = {(cuuint64_t)ldw * 2, 128};
        const cuuint32_t box[3] = {64, BK, 2u};  // one CTA's 2 atoms of a 256-column half
        const cuuint32_t estr[3] = {1, 1, 1};
        w3d = encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(W), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    if (!e4 && !w3d) {
        const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)(vocab_end - vocab_start)};
        const cuuint64_t strides[1] = {(cuuint64_t)ldw * 2};
        const cuuint32_t box[2] = {64, BK};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(W), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *msg = "tensor map of the embedding shard could not be encoded";
            return cudaErrorInvalidValue;
        }
    }
    if (!e4) {
        // a 4-D view (64 columns, rows, atoms 128 bytes apart, halves 512 bytes apart) over the
        // atoms that lie wholly inside the row pitch: a CTA's four atoms of a full-width tile
        // in one load, used where the last of them lies inside the pitch too (the kernel checks)
        const int64_t pitch_atoms = ldw / 64;
        const cuuint64_t dims4[4] = {64, (cuuint64_t)(vocab_end - vocab_start), (cuuint64_t)pitch_atoms, 2};
        const cuuint64_t strides4[3] = {(cuuint64_t)ldw * 2, 128, 512};
        const cuuint32_t box4[4] = {64, BK, 2u, 2u};
        const cuuint32_t estr4[4] = {1, 1, 1, 1};
        if (pitch_atoms >= 6 &&
            encode(&tm_w4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(W), dims4, strides4, box4,
                   estr4, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
            w4d_atoms = (int)pitch_atoms;
    }
    const cudaError_t attr_err = ensure_kernel_attributes();
    if (attr_err != cudaSuccess) {
        *msg = "could not raise the shared-memory limit of the soft-embed kernel";
        return attr_err;
    }
    int n_tiles, n_full, tail;
    column_tiles(d, plan.bn, &n_tiles, &n_full, &tail);
    n_tiles = plan.n_tiles;  // rounded up to pairs of column tiles
    Params p;
    p.lse = lse;
    p.ws = static_cast<float *>(workspace);
    p.k_begin = plan.k_begin;
    p.vocab_start = vocab_start;
    p.vocab_end = vocab_end;
    p.nkb = plan.nkb;
    p.R = (int)R;
    p.m_tiles = plan.m_tiles;
    p.n_tiles = n_tiles;
    p.n_full = n_full;
    p.tail_halves = tail;
    p.splits = plan.splits;
    p.tail_splits = tail_splits_of(plan.splits, tail);
    p.w3d = w3d;
    p.w4d_atoms = w4d_atoms;
    p.w_scale = e4 ? tab.scale : nullptr;
    p.fused = single ? 1 : 0;
    p.logits = logits;
    p.ldl = ldl;
    p.ref = nullptr;
    p.state = nullptr;
    p.draw = 0;
    p.inv_tau = 1.0f;
    p.k0 = p.k1 = p.o0 = p.o1 = 0;
    p.draws = nullptr;
    p.candidate = nullptr;
    if (single) {
        const size_t n = (size_t)plan.splits * (size_t)R;
        uint8_t *x = static_cast<uint8_t *>(workspace) + soft_embed_workspace_bytes(plan, plan.splits);
        p.ref = reinterpret_cast<float *>(x);
        x += align16(n * 4);
        p.state = reinterpret_cast<float4 *>(x);
        x += n * (size_t)plan.n_tiles * 16;
        if (single->candidate) {
            p.draw = 1;
            p.inv_tau = single->temperature > 0.0f ? 1.0f / single->temperature : 1.0f;
            p.draws = reinterpret_cast<float2 *>(x);
            p.candidate = single->candidate;
            p.k0 = (uint32_t)single->seed;
            p.k1 = (uint32_t)(single->seed >> 32);
            p.o0 = (uint32_t)single->offset;
            p.o1 = (uint32_t)(single->offset >> 32);
        }
        overlap_previous = false;  // nothing before it to wait for
    }
    // clusters: (column pair, 256-row block, split)
    const int64_t units = (int64_t)(plan.m_tiles / 2) * (n_tiles / 2) * p.splits;
    const int cluster = kQuadCtas;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cluster * units), 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = e4 ? smem_bytes<kE4m3>() : smem_bytes<kBf16>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = overlap_previous ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const int phase = single ? single->phase : 0;
    cudaError_t e = cudaSuccess;
    if (phase != 2) {  // the second call of a shard reduces what the first one left
        e = e4 ? cudaLaunchKernelEx(&cfg, soft_embed_kernel<kE4m3>, tm_l, tm_w, tm_w4, p)
               : cudaLaunchKernelEx(&cfg, soft_embed_kernel<kBf16>, tm_l, tm_w, tm_w4, p);
        if (e != cudaSuccess) {
            *msg = "soft-embed kernel launch failed";
            return e;
        }
    }
    // the single pass's small kernels each start while the one before finishes (programmatic
    // dependent launch); each waits for its predecessor before it reads what that one wrote
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    auto small_cfg = [&](unsigned grid) {
        cudaLaunchConfig_t c = {};
        c.gridDim = dim3(grid, 1, 1);
        c.blockDim = dim3(256, 1, 1);
        c.stream = stream;
        c.attrs = pdl;
        c.numAttrs = 1;
        return c;
    };
    if (phase == 1) {
        cudaLaunchConfig_t c1 = small_cfg((unsigned)((R * 32 + 255) / 256));
        e = cudaLaunchKernelEx(&c1, shard_summary_kernel, p, reinterpret_cast<float4 *>(single->shard_state),
                               single->vocab_offset);
        if (e != cudaSuccess) *msg = "shard: row summary launch failed";
        return e;
    }
    if (phase == 2) {
        cudaLaunchConfig_t c1 = small_cfg((unsigned)(((int64_t)p.splits * R + 255) / 256));
        c1.numAttrs = 0;  // the first call's kernels (and the exchange between) come before it
        e = cudaLaunchKernelEx(&c1, shard_scale_kernel, p, (const float *)single->lse);
        if (e != cudaSuccess) {
            *msg = "shard: scale launch failed";
            return e;
        }
    } else if (single) {
        cudaLaunchConfig_t c1 = small_cfg((unsigned)((R * 32 + 255) / 256));
        e = cudaLaunchKernelEx(&c1, single_pass_stats_kernel, p, single->m, single->lse, single->H, single->kappa,
                               single->argmax);
        if (e != cudaSuccess) {
            *msg = "single pass: statistics launch failed";
            return e;
        }
    }
    // two passes: the acceptance (between) overlaps the product, then the reduce; single pass:
    // the reduce kernel also runs the acceptance, in its first CTAs, on the statistics
    if (between && !single) {
        e = between(ctx, stream);
        if (e != cudaSuccess) {
            *msg = "launch between the product and the reduce failed";
            return e;
        }
    }
    const AcceptSpec no_accept{nullptr, nullptr, nullptr, 0, 1, 0, nullptr, nullptr, nullptr, nullptr};
    const AcceptSpec &acc = (single && single->accept) ? *single->accept : no_accept;
    const int n_acc = (single && single->accept) ? acc.n_req : 0;
    const int threads = n_acc > 0 ? (accept_threads(acc.L_c) > 256 ? accept_threads(acc.L_c) : 256) : 256;
    const int vec_out = (ldo % 4 == 0) && (((uintptr_t)out & 15) == 0);
    const int64_t total = R * ((d + 3) / 4);
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 8 * 256 / threads;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t c3 = small_cfg((unsigned)(blocks + n_acc));
    c3.blockDim = dim3((unsigned)threads, 1, 1);
    c3.dynamicSmemBytes = n_acc > 0 ? threads * sizeof(unsigned long long) : 0;
    c3.numAttrs = single ? 1 : 0;  // the plain reduce follows the product without overlap
    const float4 *ws4 = static_cast<const float4 *>(workspace);
    const float *scale = single ? (const float *)p.ref : nullptr;
    const float *lse_s = single ? (const float *)single->lse : nullptr;
    const LoopSpec no_loop{};
    const LoopSpec &lp = (n_acc > 0 && single->loop) ? *single->loop : no_loop;
    e = e4 ? cudaLaunchKernelEx(&c3, splitk_reduce_kernel<kE4m3>, ws4, p, (int)d, gamma, out, ldo, vec_out, scale,
                                tab.W, ldw, lse_s, acc, n_acc, lp)
           : cudaLaunchKernelEx(&c3, splitk_reduce_kernel<kBf16>, ws4, p, (int)d, gamma, out, ldo, vec_out, scale,
                                tab.W, ldw, lse_s, acc, n_acc, lp);
    if (e != cudaSuccess) {
        *msg = "split-K reduce launch failed";
        return e;
    }
    if (between && single && !single->accept) {
        e = between(ctx, stream);
        if (e != cudaSuccess) *msg = "launch after the reduce failed";
    }
    return e;
}

}  // namespace dg
