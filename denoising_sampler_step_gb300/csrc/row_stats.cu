// Row statistics of the sampler step: max, argmax, log-sum-exp, entropy and
// -ln(confidence) of the softmax over the full vocabulary, one pass over the logits.
//
// What it computes: calvarado04.com, eq. e^sc (p_i is a softmax over all V tokens);
// agentlenshq.com, "サンプリングループとエントロピー境界デノイジング" (a candidate and an
// entropy at every canvas position).
//
// Design (HBM-bound: every logit is read once, 4 bytes per vocabulary entry):
//   - one thread-block cluster per row; the row is cut into CLUSTER contiguous
//     pieces, one per CTA;
//   - 128-bit read-only loads, coalesced; each thread keeps two batches of four in
//     flight (the next batch loads while the current one is folded in);
//   - each thread keeps an online state (m, a, rest, t) over the entries it saw:
//       m    = running max, a = index of its first occurrence,
//       rest = sum over the entries other than a of exp(l - m),
//       t    = sum over all entries of exp(l - m) * (l - m)   (<= 0);
//     keeping the argmax's own 1 out of `rest` preserves kappa = log1p(rest) for
//     rows that are nearly one-hot;
//   - warp-shuffle, then CTA, then cluster (distributed shared memory) merges, in a
//     fixed order so the result is bitwise reproducible.
//   Final: lnZ = log1p(rest), lse = m + lnZ, H = lnZ - t / (1 + rest), kappa = lnZ.
#include <cooperative_groups.h>
#include <float.h>
#include <stdlib.h>

#include "dg_common.cuh"
#include "dg_internal.h"
#include "row_state.cuh"

namespace cg = cooperative_groups;

namespace dg {

namespace {

constexpr int kStatsThreads = 256;
constexpr int kStatsVec = 4;  // float4 loads per thread per batch

using namespace rowstate;

__device__ __forceinline__ float4 ld_stream(const float4 *p) { return ld_stream_v4(p); }

template <int CLUSTER>
__global__ void __launch_bounds__(kStatsThreads, 4)
    row_stats_kernel(const float *__restrict__ logits, int64_t V, int64_t ldl, float *__restrict__ out_m,
                     float *__restrict__ out_lse, float *__restrict__ out_H,
                     float *__restrict__ out_kappa, int32_t *__restrict__ out_argmax,
                     float4 *__restrict__ out_state, int64_t vocab_offset) {
    __shared__ RowState warp_state[kStatsThreads / 32];
    __shared__ RowState cta_state[CLUSTER];

    // the kernel queued next (the soft-embed product of a step) may start its CTAs now: it
    // waits for this grid to complete before it reads anything this grid writes
    grid_launch_dependents();
    const int rank = (int)(blockIdx.x % CLUSTER);
    const int64_t row = blockIdx.x / CLUSTER;
    const float *rowp = logits + row * ldl;
    const float4 *rowv = reinterpret_cast<const float4 *>(rowp);
    const int64_t nv = V >> 2;  // whole float4s in the row
    const int64_t per = (nv + CLUSTER - 1) / CLUSTER;
    const int64_t v_begin = min(nv, (int64_t)rank * per);
    const int64_t v_end = min(nv, v_begin + per);

    if constexpr (CLUSTER > 1) {
        // every CTA of the cluster must be running before the distributed-shared-memory stores below
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    }

    RowState st{-INFINITY, 0x7fffffff, 0.0f, 0.0f};
    // software pipeline: the next batch's loads are in flight while this batch is folded in
    constexpr int64_t kStep = (int64_t)kStatsThreads * kStatsVec;
    float4 cur[kStatsVec], nxt[kStatsVec];
    auto load_batch = [&](int64_t b, float4 (&v)[kStatsVec]) {
#pragma unroll
        for (int k = 0; k < kStatsVec; ++k) {
            const int64_t vi = b + (int64_t)k * kStatsThreads;
            v[k] = (vi < v_end) ? ld_stream(rowv + vi) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
    };
    int64_t b = v_begin + threadIdx.x;
    if (b < v_end) load_batch(b, cur);
    for (; b < v_end; b += kStep) {
        const bool more = b + kStep < v_end;
        if (more) load_batch(b + kStep, nxt);
        float x[4 * kStatsVec];
        int base[kStatsVec];
#pragma unroll
        for (int k = 0; k < kStatsVec; ++k) {
            base[k] = (int)(b + (int64_t)k * kStatsThreads);
            x[4 * k + 0] = cur[k].x;
            x[4 * k + 1] = cur[k].y;
            x[4 * k + 2] = cur[k].z;
            x[4 * k + 3] = cur[k].w;
        }
        absorb<4 * kStatsVec>(st, x, base);
        if (more) {
#pragma unroll
            for (int k = 0; k < kStatsVec; ++k) cur[k] = nxt[k];
        }
    }
    // ragged tail (V % 4 entries), taken by the last piece's first thread
    if (rank == CLUSTER - 1 && threadIdx.x == 0 && (V & 3)) {
        float x[4];
        int base[1] = {(int)nv};
#pragma unroll
        for (int c = 0; c < 4; ++c) x[c] = (4 * nv + c < V) ? rowp[4 * nv + c] : -INFINITY;
        absorb<4>(st, x, base);
    }

    // warp, then CTA
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        RowState o = shfl_down(st, off);
        merge(st, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_state[warp] = st;
    __syncthreads();
    if (warp == 0) {
        st = (lane < kStatsThreads / 32) ? warp_state[lane]
                                         : RowState{-INFINITY, 0x7fffffff, 0.0f, 0.0f};
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            RowState o = shfl_down(st, off);
            merge(st, o);
        }
    }

    // cluster: every CTA posts its state into the leader's shared memory
    if constexpr (CLUSTER > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        if (threadIdx.x == 0) {
            RowState *dst = cluster.map_shared_rank(cta_state, 0);
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

    if (threadIdx.x == 0 && out_state) {
        // a shard's summary: (m, global argmax as int32 bits, rest, t)
        const int a = st.m == -INFINITY ? 0x7fffffff : (int)(st.a + vocab_offset);
        out_state[row] = make_float4(st.m, __int_as_float(a), st.rest, st.t);
        return;
    }
    if (threadIdx.x == 0) {
        float lse, H, kappa;
        int a = st.a;
        if (st.m == -INFINITY) {
            lse = H = kappa = __int_as_float(0x7fc00000);
            a = 0;
        } else {
            const float lnZ = log1pf(st.rest);
            lse = st.m + lnZ;
            H = lnZ - st.t / (1.0f + st.rest);
            kappa = lnZ;
        }
        if (out_m) out_m[row] = st.m;
        if (out_lse) out_lse[row] = lse;
        if (out_H) out_H[row] = H;
        if (out_kappa) out_kappa[row] = kappa;
        if (out_argmax) out_argmax[row] = a;
    }
}

// Full-row statistics from per-shard summaries [T][R] (float4: m, argmax bits, rest, t),
// merged in shard order with the statistics kernel's own merge.
__global__ void __launch_bounds__(256)
    stats_combine_kernel(const float4 *__restrict__ states, int T, int64_t R, float *__restrict__ out_m,
                         float *__restrict__ out_lse, float *__restrict__ out_H, float *__restrict__ out_kappa,
                         int32_t *__restrict__ out_argmax) {
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= R) return;
    RowState st = empty_row_state();
    for (int r = 0; r < T; ++r) {
        const float4 v = states[(int64_t)r * R + row];
        merge(st, RowState{v.x, __float_as_int(v.y), v.z, v.w});
    }
    float lse, H, kappa;
    int a = st.a;
    if (st.m == -INFINITY) {
        lse = H = kappa = __int_as_float(0x7fc00000);
        a = 0;
    } else {
        const float lnZ = log1pf(st.rest);
        lse = st.m + lnZ;
        H = lnZ - st.t / (1.0f + st.rest);
        kappa = lnZ;
    }
    if (out_m) out_m[row] = st.m;
    if (out_lse) out_lse[row] = lse;
    if (out_H) out_H[row] = H;
    if (out_kappa) out_kappa[row] = kappa;
    if (out_argmax) out_argmax[row] = a;
}

template <int CLUSTER>
cudaError_t launch_stats(const float *logits, int64_t R, int64_t V, int64_t ldl, float *m, float *lse,
                         float *H, float *kappa, int32_t *argmax, cudaStream_t stream, float4 *state = nullptr,
                         int64_t vocab_offset = 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * CLUSTER), 1, 1);
    cfg.blockDim = dim3(kStatsThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, row_stats_kernel<CLUSTER>, logits, V, ldl, m, lse, H, kappa, argmax, state,
                              vocab_offset);
}

}  // namespace

int stats_cluster_size(int64_t R, int64_t V) {
    // at least 16K entries (64 KiB) per CTA, at most 8 CTAs (the portable cluster limit),
    // and no more than about 1024 CTAs in all: few rows split finer, many rows not at all
    int c = 1;
    while (c < 8 && V / (c * 2) >= 16384 && R * c * 2 <= 1024) c *= 2;
    return c;
}

cudaError_t launch_row_stats(const float *logits, int64_t R, int64_t V, int64_t ldl, float *m, float *lse,
                             float *H, float *kappa, int32_t *argmax, cudaStream_t stream) {
    switch (stats_cluster_size(R, V)) {
        case 1: return launch_stats<1>(logits, R, V, ldl, m, lse, H, kappa, argmax, stream);
        case 2: return launch_stats<2>(logits, R, V, ldl, m, lse, H, kappa, argmax, stream);
        case 4: return launch_stats<4>(logits, R, V, ldl, m, lse, H, kappa, argmax, stream);
        default: return launch_stats<8>(logits, R, V, ldl, m, lse, H, kappa, argmax, stream);
    }
}

}  // namespace dg

namespace dg {

cudaError_t launch_row_stats_partial(const float *logits, int64_t R, int64_t V, int64_t ldl, int64_t vocab_offset,
                                     float *state, cudaStream_t stream) {
    float4 *st = reinterpret_cast<float4 *>(state);
    switch (stats_cluster_size(R, V)) {
        case 1: return launch_stats<1>(logits, R, V, ldl, nullptr, nullptr, nullptr, nullptr, nullptr, stream, st,
                                       vocab_offset);
        case 2: return launch_stats<2>(logits, R, V, ldl, nullptr, nullptr, nullptr, nullptr, nullptr, stream, st,
                                       vocab_offset);
        case 4: return launch_stats<4>(logits, R, V, ldl, nullptr, nullptr, nullptr, nullptr, nullptr, stream, st,
                                       vocab_offset);
        default: return launch_stats<8>(logits, R, V, ldl, nullptr, nullptr, nullptr, nullptr, nullptr, stream, st,
                                        vocab_offset);
    }
}

cudaError_t launch_row_stats_combine(const float *states, int32_t T, int64_t R, float *m, float *lse, float *H,
                                     float *kappa, int32_t *argmax, cudaStream_t stream) {
    const unsigned blocks = (unsigned)((R + 255) / 256);
    stats_combine_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4 *>(states), (int)T, R, m, lse, H,
                                                     kappa, argmax);
    return cudaGetLastError();
}

}  // namespace dg
