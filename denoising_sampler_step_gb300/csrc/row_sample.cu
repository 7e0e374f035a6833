// Stochastic candidate per canvas position: a categorical draw from softmax(l / tau) with
// its tempered log-probability; optionally fused with the row statistics (one read of
// the logits for both).
//
// What it computes: agentlenshq.com, "サンプリングループとエントロピー境界デノイジング"
// (candidate tokens are sampled at every position).  The draw is a two-level Gumbel-max,
// an exact categorical sampler: the vocabulary is cut into groups of 16 consecutive
// entries; the group g* = argmax_g (L_g + G_g), L_g the group's log-mass logsumexp(l/tau)
// and G_g = -ln(-ln u_g); then the candidate = argmax over g*'s entries of l/tau + G_v.
// The uniforms are Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers:
// as easy as 1, 2, 3", SC 2011) with key (seed low, seed high): entry v uses word v % 4 of
// the block with counter (v / 4, row, offset low, offset high), group g word g % 4 of the
// block with counter (2^31 + g / 4, row, offset low, offset high); u = ((x >> 9) + 1/2) 2^-23.
//
// Design (HBM-bound like the row statistics: one cluster of CTAs per row, fixed-order warp /
// CTA / cluster merges).  A thread takes one group (four contiguous float4) per batch and
// keeps
//   m, s       : running max of z = l / tau and sum of exp(z - m)  (for lse_tau);
//   best, grp  : the best group score m + ln(sum of the group's exp(z - m)) + G_g and its
//                group (lowest on ties);
// so a group costs its 16 exponentials (which the tempered sum needs anyway), one Philox
// block and two logarithms.  (Skipping groups that cannot win, as G < 16.7, measured slower:
// the warp-wide bound costs more than the rare skips save.)  After the merges, 16 lanes of
// the first CTA draw inside the chosen group (four Philox blocks) and the lowest-index best
// entry is the candidate.
#include <cooperative_groups.h>
#include <float.h>

#include "dg_common.cuh"
#include "dg_internal.h"
#include "philox.cuh"
#include "row_state.cuh"

namespace cg = cooperative_groups;

namespace dg {

namespace {

constexpr int kThreads = 256;
constexpr int kGroup = 16;           // vocabulary entries per group (four float4)

using namespace philox;

struct SampleState {
    float m, s;  // max of z and sum of exp(z - m)
    float best;  // best group score (-inf: none yet)
    int grp;     // its group (INT_MAX: none)
};

__device__ __forceinline__ SampleState empty_state() { return {-INFINITY, 0.0f, -INFINITY, 0x7fffffff}; }

// A := A merged with B: the larger max carries the rescaled sums; the better group score
// wins, equal scores keep the lower group.
__device__ __forceinline__ void merge(SampleState &A, const SampleState &B) {
    if (B.m > A.m) {
        A.s = (A.m == -INFINITY ? 0.0f : A.s * ex2_approx((A.m - B.m) * kLog2e)) + B.s;
        A.m = B.m;
    } else if (B.m != -INFINITY) {
        A.s += B.s * ex2_approx((B.m - A.m) * kLog2e);
    }
    if (B.best > A.best || (B.best == A.best && B.grp < A.grp)) {
        A.best = B.best;
        A.grp = B.grp;
    }
}

__device__ __forceinline__ SampleState shfl_down(const SampleState &a, int off) {
    SampleState o;
    o.m = __shfl_down_sync(0xffffffffu, a.m, off);
    o.s = __shfl_down_sync(0xffffffffu, a.s, off);
    o.best = __shfl_down_sync(0xffffffffu, a.best, off);
    o.grp = __shfl_down_sync(0xffffffffu, a.grp, off);
    return o;
}

struct SampleArgs {
    float inv_tau;
    uint32_t k0, k1, o0, o1;  // key and the counter's offset words
};

// Folds group g of row `row` (entries 16g .. 16g + 15: z, -inf past V) into st.
__device__ __forceinline__ void absorb_group(SampleState &st, const float (&z)[kGroup], int g, uint32_t row,
                                             const SampleArgs &a) {
    float gm = z[0];
#pragma unroll
    for (int j = 1; j < kGroup; ++j) gm = fmaxf(gm, z[j]);
    if (gm == -INFINITY) return;  // a masked group: no mass, never drawn
    if (gm > st.m) {
        st.s = st.m == -INFINITY ? 0.0f : st.s * ex2_approx((st.m - gm) * kLog2e);
        st.m = gm;
    }
    const float nm = -st.m * kLog2e;
    float gs = 0.0f;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) gs += ex2_approx(fmaf(z[j], kLog2e, nm));  // -inf entries: 0
    st.s += gs;
    const Philox w = philox4x32_10(kGroupCounter + (uint32_t)(g >> 2), row, a.o0, a.o1, a.k0, a.k1);
    // score = ln(sum of exp(z)) + G = m + ln(gs) - ln(-ln u)
    const float sc = st.m + kLn2 * __log2f(gs) - kLn2 * __log2f(neg_log_uniform(philox_word(w, g & 3)));
    if (sc > st.best) {  // groups arrive in increasing order: ties keep the lower
        st.best = sc;
        st.grp = g;
    }
}

__device__ __forceinline__ float4 ld_stream(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
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
    __shared__ float draw_lse;
    __shared__ int draw_grp;

    // the kernel queued next (the soft-embed product of a step) may start its CTAs now: it
    // waits for this grid to complete before it reads anything this grid writes
    if constexpr (STATS) grid_launch_dependents();
    const int rank = (int)(blockIdx.x % CLUSTER);
    const int64_t row = blockIdx.x / CLUSTER;
    const float *rowp = logits + row * ldl;
    const float4 *rowv = reinterpret_cast<const float4 *>(rowp);
    // float4s holding the row (the last one partial when V % 4 != 0: ldl % 4 == 0 keeps it
    // inside the row), groups, and this CTA's contiguous share of the groups
    const int64_t nv = (V + 3) >> 2;
    const int64_t G = (V + kGroup - 1) / kGroup;
    const int64_t per = (G + CLUSTER - 1) / CLUSTER;
    const int64_t g_begin = min(G, (int64_t)rank * per);
    const int64_t g_end = min(G, g_begin + per);

    if constexpr (CLUSTER > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    SampleState st = empty_state();
    RowState rs = rowstate::empty_row_state();
    float4 cur[4], nxt[4];
    auto load_group = [&](int64_t g, float4(&v)[4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t q = 4 * g + k;
            v[k] = (g < g_end && q < nv) ? ld_stream(rowv + q)
                                         : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
    };
    int64_t g = g_begin + threadIdx.x;
    load_group(g, cur);
    // every lane of a warp runs the same number of batches (lanes past g_end skip their group)
    for (int64_t g0 = g_begin; g0 < g_end; g0 += kThreads, g += kThreads) {
        const bool more = g0 + kThreads < g_end;
        if (more) load_group(g + kThreads, nxt);
        if (g < g_end) {
            float x[kGroup];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[4 * k + 0] = cur[k].x;
                x[4 * k + 1] = cur[k].y;
                x[4 * k + 2] = cur[k].z;
                x[4 * k + 3] = cur[k].w;
            }
            if (kGroup * (g + 1) > V) {  // the row's last group: entries past V are not part of it
#pragma unroll
                for (int j = 0; j < kGroup; ++j)
                    if (kGroup * g + j >= V) x[j] = -INFINITY;
            }
            if constexpr (STATS) {
                float xs[kGroup];
                int bs[4];
#pragma unroll
                for (int j = 0; j < kGroup; ++j) xs[j] = x[j];
#pragma unroll
                for (int k = 0; k < 4; ++k) bs[k] = (int)(4 * g + k);
                rowstate::absorb<kGroup>(rs, xs, bs);
            }
            float z[kGroup];
#pragma unroll
            for (int j = 0; j < kGroup; ++j) z[j] = x[j] * a.inv_tau;
            absorb_group(st, z, (int)g, (uint32_t)row, a);
        }
        if (more) {
#pragma unroll
            for (int k = 0; k < 4; ++k) cur[k] = nxt[k];
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
    if (warp != 0) return;
    // the second level: lanes 0-15 draw inside the chosen group
    const bool none = st.m == -INFINITY || st.grp == 0x7fffffff;
    if (lane == 0) {
        draw_lse = none ? __int_as_float(0x7fc00000) : st.m + kLn2 * __log2f(st.s);
        draw_grp = none ? -1 : st.grp;
    }
    __syncwarp();
    const int gs = draw_grp;
    const int64_t v = (int64_t)kGroup * gs + lane;
    const bool valid = gs >= 0 && lane < kGroup && v < V;
    const float l = valid ? rowp[v] : -INFINITY;
    float sc = -INFINITY;
    if (valid && l != -INFINITY) {
        const Philox w = philox4x32_10((uint32_t)(v >> 2), (uint32_t)row, a.o0, a.o1, a.k0, a.k1);
        sc = l * a.inv_tau - kLn2 * __log2f(neg_log_uniform(philox_word(w, (int)(v & 3))));
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
        const float qnan = __int_as_float(0x7fc00000);
        const bool drawn = !none && sc > -INFINITY;
        candidate[row] = drawn ? bi : 0;
        if (log_p) log_p[row] = drawn ? bl * a.inv_tau - draw_lse : qnan;
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
                kappa = !drawn ? qnan : (bi == rs.a ? lnZ : (rs.m - bl) + lnZ);
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
