// Stochastic candidate per canvas position: a categorical draw from softmax(l / tau)
// taken as the Gumbel-max, argmax_v (l_v / tau - ln(-ln u_v)), with its tempered
// log-probability.  One pass over the logits.
//
// What it computes: agentlenshq.com, "サンプリングループとエントロピー境界デノイジング"
// (candidate tokens are sampled at every position).  The uniforms are Philox4x32-10
// (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
// entry v of row i uses word v % 4 of the block with counter (v / 4, i, offset low,
// offset high) and key (seed low, seed high); u = ((x >> 9) + 1/2) 2^-23.
//
// Design (HBM-bound like the row statistics: one cluster of CTAs per row, 128-bit loads,
// fixed-order warp / CTA / cluster merges).  Each thread keeps
//   m, s  : running max of z = l / tau and sum of exp(z - m)  (for lse_tau);
//   best  : the best perturbed score z + g, its index (lowest on ties) and its z.
// Since u <= 1 - 2^-24, g <= -ln(2^-24) < 16.7: a group of four entries whose z all lie
// more than that below a score the warp already holds cannot win, and its Philox block
// and logarithms are skipped (the warp shares its best score after every batch of loads).
// Near-uniform rows, where every entry can still win, pay for every draw.
#include <cooperative_groups.h>
#include <float.h>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace cg = cooperative_groups;

namespace dg {

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;            // float4 loads per thread per batch
constexpr float kGumbelMax = 16.7f;  // above every g the 23-bit uniforms can give

struct Philox {
    uint32_t x0, x1, x2, x3;
};

__device__ __forceinline__ Philox philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return {c0, c1, c2, c3};
}

// g = -ln(-ln u).  -ln u: near u = 1 (t = 1 - u < 1/64, exact in fp32) the series
// t (1 + t/2 + t^2/3) of -ln(1 - t) (relative error below t^3 / 4); elsewhere the fast
// logarithm, whose absolute error is then small against |ln u| >= 1/64.
__device__ __forceinline__ float gumbel(uint32_t x) {
    const float u = ((float)(x >> 9) + 0.5f) * 1.1920928955078125e-7f;  // 2^-23
    const float t = 1.0f - u;
    const float w = t < 0.015625f ? t * fmaf(t, fmaf(t, 0.333333343f, 0.5f), 1.0f) : -__logf(u);
    return -__logf(w);
}

struct SampleState {
    float m, s;       // max of z and sum of exp(z - m)
    float best;       // best perturbed score
    int idx;          // its index (INT_MAX: none yet)
    float zbest;      // its z
};

__device__ __forceinline__ SampleState empty_state() { return {-INFINITY, 0.0f, -INFINITY, 0x7fffffff, 0.0f}; }

// A := A merged with B: the larger max carries the rescaled sums; the better score wins,
// equal scores keep the lower index.
__device__ __forceinline__ void merge(SampleState &A, const SampleState &B) {
    if (B.m > A.m) {
        A.s = (A.m == -INFINITY ? 0.0f : A.s * ex2_approx((A.m - B.m) * kLog2e)) + B.s;
        A.m = B.m;
    } else if (B.m != -INFINITY) {
        A.s += B.s * ex2_approx((B.m - A.m) * kLog2e);
    }
    if (B.best > A.best || (B.best == A.best && B.idx < A.idx)) {
        A.best = B.best;
        A.idx = B.idx;
        A.zbest = B.zbest;
    }
}

__device__ __forceinline__ SampleState shfl_down(const SampleState &a, int off) {
    SampleState o;
    o.m = __shfl_down_sync(0xffffffffu, a.m, off);
    o.s = __shfl_down_sync(0xffffffffu, a.s, off);
    o.best = __shfl_down_sync(0xffffffffu, a.best, off);
    o.idx = __shfl_down_sync(0xffffffffu, a.idx, off);
    o.zbest = __shfl_down_sync(0xffffffffu, a.zbest, off);
    return o;
}

struct SampleArgs {
    float inv_tau;
    uint32_t k0, k1, o0, o1;  // key and the counter's offset words
};

// Folds the four entries 4q .. 4q+3 of row `row` (values x, -inf past V) into st.
__device__ __forceinline__ void absorb4(SampleState &st, const float4 v, int64_t q, uint32_t row, const SampleArgs &a,
                                        float bound) {
    const float z[4] = {v.x * a.inv_tau, v.y * a.inv_tau, v.z * a.inv_tau, v.w * a.inv_tau};
    const float bm = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    if (bm > st.m) {
        st.s = st.m == -INFINITY ? 0.0f : st.s * ex2_approx((st.m - bm) * kLog2e);
        st.m = bm;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (z[j] != -INFINITY) st.s += ex2_approx((z[j] - st.m) * kLog2e);
    // no entry here can beat `bound` (a score some thread of the warp already holds)
    if (bm + kGumbelMax < fmaxf(bound, st.best) || bm == -INFINITY) return;
    const Philox w = philox4x32_10((uint32_t)q, row, a.o0, a.o1, a.k0, a.k1);
    const uint32_t words[4] = {w.x0, w.x1, w.x2, w.x3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (z[j] == -INFINITY) continue;
        const float sc = z[j] + gumbel(words[j]);
        const int idx = (int)(4 * q + j);
        if (sc > st.best || (sc == st.best && idx < st.idx)) {
            st.best = sc;
            st.idx = idx;
            st.zbest = z[j];
        }
    }
}

__device__ __forceinline__ float4 ld_stream(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

template <int CLUSTER>
__global__ void __launch_bounds__(kThreads, 3)
    row_sample_kernel(const float *__restrict__ logits, int64_t V, int64_t ldl, SampleArgs a,
                      int32_t *__restrict__ candidate, float *__restrict__ log_p) {
    __shared__ SampleState warp_state[kThreads / 32];
    __shared__ SampleState cta_state[CLUSTER];

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
    constexpr int64_t kStep = (int64_t)kThreads * kVec;
    float4 cur[kVec], nxt[kVec];
    auto load_batch = [&](int64_t b, float4(&v)[kVec]) {
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const int64_t vi = b + (int64_t)k * kThreads;
            v[k] = (vi < v_end) ? ld_stream(rowv + vi) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
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
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            const int64_t vi = b + (int64_t)k * kThreads;
            if (vi < v_end) absorb4(st, cur[k], vi, (uint32_t)row, a, bound);
        }
        float wb = st.best;
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
    }

#pragma unroll
    for (int off = 16; off > 0; off >>= 1) merge(st, shfl_down(st, off));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_state[warp] = st;
    __syncthreads();
    if (warp == 0) {
        st = (lane < kThreads / 32) ? warp_state[lane] : empty_state();
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) merge(st, shfl_down(st, off));
    }
    if constexpr (CLUSTER > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        if (threadIdx.x == 0) {
            SampleState *dst = cluster.map_shared_rank(cta_state, 0);
            dst[rank] = st;
        }
        cluster.sync();
        if (rank != 0) return;
        if (threadIdx.x == 0) {
            st = cta_state[0];
#pragma unroll
            for (int r = 1; r < CLUSTER; ++r) merge(st, cta_state[r]);
        }
    }
    if (threadIdx.x == 0) {
        if (st.m == -INFINITY || st.idx == 0x7fffffff) {
            candidate[row] = 0;
            log_p[row] = __int_as_float(0x7fc00000);
        } else {
            candidate[row] = st.idx;
            log_p[row] = st.zbest - (st.m + logf(st.s));
        }
    }
}

template <int CLUSTER>
cudaError_t launch(const float *logits, int64_t R, int64_t V, int64_t ldl, SampleArgs a, int32_t *cand, float *lp,
                   cudaStream_t stream) {
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
    return cudaLaunchKernelEx(&cfg, row_sample_kernel<CLUSTER>, logits, V, ldl, a, cand, lp);
}

}  // namespace

cudaError_t launch_row_sample(const float *logits, int64_t R, int64_t V, int64_t ldl, float temperature, uint64_t seed,
                              uint64_t offset, int32_t *candidate, float *log_p, cudaStream_t stream) {
    SampleArgs a;
    a.inv_tau = (float)(1.0 / (double)temperature);
    a.k0 = (uint32_t)seed;
    a.k1 = (uint32_t)(seed >> 32);
    a.o0 = (uint32_t)offset;
    a.o1 = (uint32_t)(offset >> 32);
    switch (stats_cluster_size(R, V)) {
        case 1: return launch<1>(logits, R, V, ldl, a, candidate, log_p, stream);
        case 2: return launch<2>(logits, R, V, ldl, a, candidate, log_p, stream);
        case 4: return launch<4>(logits, R, V, ldl, a, candidate, log_p, stream);
        default: return launch<8>(logits, R, V, ldl, a, candidate, log_p, stream);
    }
}

}  // namespace dg
