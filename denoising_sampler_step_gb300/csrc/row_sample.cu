// Stochastic candidate per canvas position: a categorical draw from softmax(l / tau)
// taken as the Gumbel-max, argmax_v (l_v / tau - ln(-ln u_v)), with its tempered
// log-probability; optionally fused with the row statistics (one read of the logits
// for both).
//
// What it computes: agentlenshq.com, "サンプリングループとエントロピー境界デノイジング"
// (candidate tokens are sampled at every position).  The uniforms are Philox4x32-10
// (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
// entry v of row i uses word v % 4 of the block with counter (v / 4, i, offset low,
// offset high) and key (seed low, seed high); u = ((x >> 9) + 1/2) 2^-23.
//
// Design (HBM-bound like the row statistics: one cluster of CTAs per row, 128-bit loads,
// fixed-order warp / CTA / cluster merges).  The draw is kept as an exponential race,
// the same argmax written without the outer logarithm: with E_v = -ln u_v and
// e_v = exp(z_v - m) (z = l / tau, m the running max), the winner minimises E_v / e_v,
// and e_v is the term the tempered log-sum-exp adds anyway.  So each entry costs one
// exp, one logarithm and a multiply-compare; a division only when a thread's best
// changes.  Each thread keeps
//   m, s   : running max of z and sum of exp(z - m)  (for lse_tau);
//   R      : its best ratio E / e, relative to its m (R scales by exp(m' - m) when m grows);
//   idx, l : the best entry's index (lowest on ties) and its logit.
// Threads merge in the log domain, score = m - ln R = z + g of the best entry.
// Since u <= 1 - 2^-24, g <= -ln(2^-24) < 16.7: a group of four entries whose z all lie
// more than that below a score the warp already holds cannot win, and its Philox block
// and logarithms are skipped (the warp shares its best score after every batch of loads).
// Near-uniform rows, where every entry can still win, pay for every draw.
#include <cooperative_groups.h>
#include <float.h>

#include "dg_common.cuh"
#include "dg_internal.h"
#include "row_state.cuh"

namespace cg = cooperative_groups;

namespace dg {

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;              // float4 loads per thread per batch
constexpr float kGumbelMax = 16.7f;  // above every g the 23-bit uniforms can give
constexpr float kLn2 = 0.69314718055994531f;

struct Philox {
    uint32_t x0, x1, x2, x3;
};

__device__ __forceinline__ Philox philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c0 = n0;
        c1 = (uint32_t)p1;
        c2 = n2;
        c3 = (uint32_t)p0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return {c0, c1, c2, c3};
}

// E = -ln u for u = ((x >> 9) + 1/2) 2^-23, built without an integer conversion:
// f = 1 + (x >> 9) 2^-23 is the float with those mantissa bits, and f - (1 - 2^-24) = u
// exactly (both operands and the result are fp32 numbers within a factor of two).
// Near u = 1 (t = 1 - u < 1/64, exact) the series t (1 + t/2 + t^2/3) of -ln(1 - t)
// (relative error below t^3 / 4); elsewhere the fast logarithm, whose absolute error is
// then small against |ln u| >= 1/64.
__device__ __forceinline__ float neg_log_uniform(uint32_t x) {
    const float f = __uint_as_float(0x3F800000u | (x >> 9));
    const float u = f - 0.99999994039535522f;  // 1 - 2^-24
    const float t = 1.0f - u;
    return t < 0.015625f ? t * fmaf(t, fmaf(t, 0.333333343f, 0.5f), 1.0f) : -kLn2 * __log2f(u);
}

struct SampleState {
    float m, s;  // max of z and sum of exp(z - m)
    float R;     // best E / exp(z - m) (+inf: none yet)
    int idx;     // its index
    float l;     // its logit
};

__device__ __forceinline__ SampleState empty_state() { return {-INFINITY, 0.0f, INFINITY, 0x7fffffff, 0.0f}; }

// the best entry's perturbed score z + g, -inf if none
__device__ __forceinline__ float score(const SampleState &a) {
    return a.R == INFINITY ? -INFINITY : a.m - kLn2 * __log2f(a.R);
}

// A := A merged with B: the larger max carries the rescaled sums; the better score wins,
// equal scores keep the lower index; the winner's ratio is restated against the new max.
__device__ __forceinline__ void merge(SampleState &A, const SampleState &B) {
    const float sa = score(A), sb = score(B);
    const bool b_best = sb > sa || (sb == sa && B.idx < A.idx);
    float m = A.m, s = A.s;
    if (B.m > A.m) {
        s = (A.m == -INFINITY ? 0.0f : A.s * ex2_approx((A.m - B.m) * kLog2e)) + B.s;
        m = B.m;
    } else if (B.m != -INFINITY) {
        s += B.s * ex2_approx((B.m - A.m) * kLog2e);
    }
    const float wR = b_best ? B.R : A.R, wm = b_best ? B.m : A.m;
    A.R = wR == INFINITY ? INFINITY : wR * ex2_approx((m - wm) * kLog2e);
    A.idx = b_best ? B.idx : A.idx;
    A.l = b_best ? B.l : A.l;
    A.m = m;
    A.s = s;
}

__device__ __forceinline__ SampleState shfl_down(const SampleState &a, int off) {
    SampleState o;
    o.m = __shfl_down_sync(0xffffffffu, a.m, off);
    o.s = __shfl_down_sync(0xffffffffu, a.s, off);
    o.R = __shfl_down_sync(0xffffffffu, a.R, off);
    o.idx = __shfl_down_sync(0xffffffffu, a.idx, off);
    o.l = __shfl_down_sync(0xffffffffu, a.l, off);
    return o;
}

struct SampleArgs {
    float inv_tau;
    uint32_t k0, k1, o0, o1;  // key and the counter's offset words
};

// Folds the four entries 4q .. 4q+3 of row `row` (values v, -inf past V) into st.
// `bound`: a score some thread of the warp already holds.
__device__ __forceinline__ void absorb4(SampleState &st, const float4 v, int64_t q, uint32_t row, const SampleArgs &a,
                                        float bound) {
    const float l[4] = {v.x, v.y, v.z, v.w};
    float z[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) z[j] = l[j] * a.inv_tau;
    const float bm = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    if (bm == -INFINITY) return;  // four masked entries: nothing to add, nothing to draw
    if (bm > st.m) {
        if (st.m == -INFINITY) {
            st.s = 0.0f;
        } else {
            const float c = ex2_approx((st.m - bm) * kLog2e);
            st.s *= c;
            st.R = st.R == INFINITY ? INFINITY : __fdividef(st.R, c);  // c == 0: the old best cannot win
        }
        st.m = bm;
    }
    float e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        e[j] = ex2_approx((z[j] - st.m) * kLog2e);  // st.m is finite here; -inf entries give 0
        st.s += e[j];
    }
    // no entry here can beat `bound`
    if (bm + kGumbelMax < bound) return;
    const Philox w = philox4x32_10((uint32_t)q, row, a.o0, a.o1, a.k0, a.k1);
    const uint32_t words[4] = {w.x0, w.x1, w.x2, w.x3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float E = neg_log_uniform(words[j]);
        // E / e < R, written without the division (e == 0 gives NaN or 0: never a win;
        // R == inf: any e > 0 wins)
        if (E < st.R * e[j]) {
            st.R = __fdividef(E, e[j]);
            st.idx = (int)(4 * q + j);
            st.l = l[j];
        }
    }
}

// Per-row outputs of the fused kernel (statistics at temperature 1 and the draw).
struct FusedOut {
    float *m, *lse, *H, *kappa;
    int32_t *argmax;
};

// One pass over a row: the draw, and when STATS the row statistics too.
template <int CLUSTER, bool STATS>
__global__ void __launch_bounds__(kThreads, 3)
    row_sample_kernel(const float *__restrict__ logits, int64_t V, int64_t ldl, SampleArgs a,
                      int32_t *__restrict__ candidate, float *__restrict__ log_p, FusedOut fo) {
    using rowstate::RowState;
    __shared__ SampleState warp_state[kThreads / 32];
    __shared__ SampleState cta_state[CLUSTER];
    __shared__ RowState warp_stats[STATS ? kThreads / 32 : 1];
    __shared__ RowState cta_stats[STATS ? CLUSTER : 1];

    // the kernel queued next (the soft-embed product of a step) may start its CTAs now: it
    // waits for this grid to complete before it reads anything this grid writes
    if constexpr (STATS) grid_launch_dependents();
    const int rank = (int)(blockIdx.x % CLUSTER);
    const int64_t row = blockIdx.x / CLUSTER;
    const float *rowp = logits + row * ldl;
    const float4 *rowv = reinterpret_cast<const float4 *>(rowp);
    const int64_t nv = V >> 2;
    const int64_t per = (nv + CLUSTER - 1) / CLUSTER;
    const int64_t v_begin = min(nv, (int64_t)rank * per);
    const int64_t v_end = min(nv, v_begin + per);

    if constexpr (CLUSTER > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    SampleState st = empty_state();
    RowState rs = rowstate::empty_row_state();
    constexpr int64_t kStep = (int64_t)kThreads * kVec;
    float4 cur[kVec], nxt[kVec];
    auto load_batch = [&](int64_t b, float4(&v)[kVec]) {
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const int64_t vi = b + (int64_t)k * kThreads;
            v[k] = (vi < v_end) ? rowstate::ld_stream_v4(rowv + vi)
                                : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
    };
    int64_t b = v_begin + threadIdx.x;
    if (b < v_end) load_batch(b, cur);
    float bound = -INFINITY;  // the best score in the warp after the previous batch
    // every lane of a warp runs the same number of batches (the bounds are warp-uniform
    // up to the last batch, where lanes past v_end only skip their entries)
    for (int64_t b0 = v_begin; b0 < v_end; b0 += kStep, b += kStep) {
        const bool more = b + kStep < v_end;
        if (more) load_batch(b + kStep, nxt);
        if constexpr (STATS) {
            // the statistics kernel's fold, on the same batches (lanes past v_end hold -inf)
            float x[4 * kVec];
            int base[kVec];
#pragma unroll
            for (int k = 0; k < kVec; ++k) {
                base[k] = (int)(b + (int64_t)k * kThreads);
                x[4 * k + 0] = cur[k].x;
                x[4 * k + 1] = cur[k].y;
                x[4 * k + 2] = cur[k].z;
                x[4 * k + 3] = cur[k].w;
            }
            if (b < v_end) rowstate::absorb<4 * kVec>(rs, x, base);
        }
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const int64_t vi = b + (int64_t)k * kThreads;
            if (vi < v_end) absorb4(st, cur[k], vi, (uint32_t)row, a, bound);
        }
        float wb = score(st);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wb = fmaxf(wb, __shfl_xor_sync(0xffffffffu, wb, off));
        bound = wb;
        if (more) {
#pragma unroll
            for (int k = 0; k < kVec; ++k) cur[k] = nxt[k];
        }
    }
    // ragged tail (V % 4 entries), taken by the last piece's first thread
    if (rank == CLUSTER - 1 && threadIdx.x == 0 && (V & 3)) {
        float t[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) t[c] = (4 * nv + c < V) ? rowp[4 * nv + c] : -INFINITY;
        absorb4(st, make_float4(t[0], t[1], t[2], t[3]), nv, (uint32_t)row, a, -INFINITY);
        if constexpr (STATS) {
            int base[1] = {(int)nv};
            rowstate::absorb<4>(rs, t, base);
        }
    }

    // warp, then CTA, then cluster, in a fixed order
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        merge(st, shfl_down(st, off));
        if constexpr (STATS) rowstate::merge(rs, rowstate::shfl_down(rs, off));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        warp_state[warp] = st;
        if constexpr (STATS) warp_stats[warp] = rs;
    }
    __syncthreads();
    if (warp == 0) {
        st = (lane < kThreads / 32) ? warp_state[lane] : empty_state();
        if constexpr (STATS) rs = (lane < kThreads / 32) ? warp_stats[lane] : rowstate::empty_row_state();
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            merge(st, shfl_down(st, off));
            if constexpr (STATS) rowstate::merge(rs, rowstate::shfl_down(rs, off));
        }
    }
    if constexpr (CLUSTER > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        if (threadIdx.x == 0) {
            cluster.map_shared_rank(cta_state, 0)[rank] = st;
            if constexpr (STATS) cluster.map_shared_rank(cta_stats, 0)[rank] = rs;
        }
        cluster.sync();
        if (rank != 0) return;
        if (threadIdx.x == 0) {
            st = cta_state[0];
#pragma unroll
            for (int r = 1; r < CLUSTER; ++r) merge(st, cta_state[r]);
            if constexpr (STATS) {
                rs = cta_stats[0];
#pragma unroll
                for (int r = 1; r < CLUSTER; ++r) rowstate::merge(rs, cta_stats[r]);
            }
        }
    }
    if (threadIdx.x == 0) {
        const float qnan = __int_as_float(0x7fc00000);
        const bool none = st.m == -INFINITY || st.R == INFINITY;
        candidate[row] = none ? 0 : st.idx;
        if (log_p) log_p[row] = none ? qnan : st.l * a.inv_tau - (st.m + logf(st.s));
        if constexpr (STATS) {
            // statistics at temperature 1, and kappa = -ln p(candidate): ln Z for the
            // argmax itself, (m - l_c) + ln Z otherwise
            float lse = qnan, H = qnan, kappa = qnan;
            int am = 0;
            if (rs.m != -INFINITY) {
                const float lnZ = log1pf(rs.rest);
                lse = rs.m + lnZ;
                H = lnZ - rs.t / (1.0f + rs.rest);
                am = rs.a;
                kappa = none ? qnan : (st.idx == rs.a ? lnZ : (rs.m - st.l) + lnZ);
            }
            if (fo.m) fo.m[row] = rs.m;
            if (fo.lse) fo.lse[row] = lse;
            if (fo.H) fo.H[row] = H;
            if (fo.kappa) fo.kappa[row] = kappa;
            if (fo.argmax) fo.argmax[row] = am;
        }
    }
}

template <int CLUSTER, bool STATS>
cudaError_t launch(const float *logits, int64_t R, int64_t V, int64_t ldl, SampleArgs a, int32_t *cand, float *lp,
                   FusedOut fo, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * CLUSTER), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, row_sample_kernel<CLUSTER, STATS>, logits, V, ldl, a, cand, lp, fo);
}

template <bool STATS>
cudaError_t launch_any(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature, uint64_t seed,
                       uint64_t offset, int32_t *candidate, float *log_p, FusedOut fo, cudaStream_t stream) {
    SampleArgs a;
    a.inv_tau = (float)(1.0 / (double)temperature);
    a.k0 = (uint32_t)seed;
    a.k1 = (uint32_t)(seed >> 32);
    a.o0 = (uint32_t)offset;
    a.o1 = (uint32_t)(offset >> 32);
    switch (stats_cluster_size(R, V)) {
        case 1: return launch<1, STATS>(logits, R, V, ldl, a, candidate, log_p, fo, stream);
        case 2: return launch<2, STATS>(logits, R, V, ldl, a, candidate, log_p, fo, stream);
        case 4: return launch<4, STATS>(logits, R, V, ldl, a, candidate, log_p, fo, stream);
        default: return launch<8, STATS>(logits, R, V, ldl, a, candidate, log_p, fo, stream);
    }
}

}  // namespace

cudaError_t launch_row_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature, uint64_t seed,
                              uint64_t offset, int32_t *candidate, float *log_p, cudaStream_t stream) {
    return launch_any<false>(logits, R, V, ldl, temperature, seed, offset, candidate, log_p, FusedOut{}, stream);
}

cudaError_t launch_row_stats_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature,
                                    uint64_t seed, uint64_t offset, float *m, float *lse, float *H, float *kappa,
                                    int32_t *argmax, int32_t *candidate, float *log_p, cudaStream_t stream) {
    return launch_any<true>(logits, R, V, ldl, temperature, seed, offset, candidate, log_p,
                            FusedOut{m, lse, H, kappa, argmax}, stream);
}

}  // namespace dg
