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
//   - a loader thread streams the CTA's piece into a ring of four 16 KiB shared-memory
//     stages with bulk copies (cp.async.bulk, completing on an mbarrier per stage), so
//     that the bytes in flight do not cost registers; each of the 256 folding threads
//     takes four float4 of a stage (float4 t, t + 256, t + 512, t + 768: conflict-free
//     shared-memory reads), hands the stage back, then folds its 16 values;
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

#include <atomic>

#include "dg_common.cuh"
#include "dg_internal.h"
#include "row_state.cuh"

namespace cg = cooperative_groups;

namespace dg {

namespace {

constexpr int kStatsThreads = 256;                    // folding threads
constexpr int kStatsCtaThreads = kStatsThreads + 32;  // and the loader's warp
constexpr int kStatsVec = 4;                          // float4 per folding thread per stage
constexpr int kStatsChunk = kStatsThreads * kStatsVec;  // float4 per stage (16 KiB)
constexpr int kStatsStages = 4;
constexpr int kStatsSmem = kStatsStages * kStatsChunk * 16;

using namespace rowstate;

// Global -> shared bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned),
// completing on the barrier; the lines it reads are marked first to evict.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

template <int CLUSTER>
__global__ void __launch_bounds__(kStatsCtaThreads, 3)
    row_stats_kernel(const float *__restrict__ logits, int64_t V, int64_t ldl, float *__restrict__ out_m,
                     float *__restrict__ out_lse, float *__restrict__ out_H,
                     float *__restrict__ out_kappa, int32_t *__restrict__ out_argmax,
                     float4 *__restrict__ out_state, int64_t vocab_offset) {
    extern __shared__ __align__(128) float4 ring[];
    __shared__ __align__(8) uint64_t full[kStatsStages], empty[kStatsStages];
    __shared__ int abort_flag;
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

    const int64_t len = v_end - v_begin;  // float4 of this CTA's piece
    const int nchunks = (int)((len + kStatsChunk - 1) / kStatsChunk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kStatsStages; ++st) {
            mbar_init(smem_u32(&full[st]), 1);
            mbar_init(smem_u32(&empty[st]), kStatsThreads / 32);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if constexpr (CLUSTER > 1) {
        // every CTA of the cluster must be running before the distributed-shared-memory stores below
        asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    }

    RowState st{-INFINITY, 0x7fffffff, 0.0f, 0.0f};
    if (warp == kStatsThreads / 32) {
        // ------------------------------------------------ loader: stage c % kStatsStages
        // takes chunk c once the folding warps handed back chunk c - kStatsStages
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            int issued[kStatsStages];
            for (int q = 0; q < kStatsStages; ++q) issued[q] = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int q = c % kStatsStages;
                const uint32_t u = (uint32_t)(c / kStatsStages);
                if (u > 0 && !mbar_wait(smem_u32(&empty[q]), (u - 1) & 1, &abort_flag)) break;
                const int64_t c0 = (int64_t)c * kStatsChunk;
                const int64_t n4 = min((int64_t)kStatsChunk, len - c0);
                const uint32_t bar = smem_u32(&full[q]);
                mbar_arrive_expect_tx(bar, (uint32_t)(n4 * 16));
                bulk_load(smem_u32(ring + q * kStatsChunk), rowv + v_begin + c0, (uint32_t)(n4 * 16), bar, policy);
                issued[q] = (int)u + 1;
            }
            // a CTA that gave up leaves only after its copies in flight have landed
            if (abort_flag)
                for (int q = 0; q < kStatsStages; ++q)
                    if (issued[q] > 0) drain_wait(smem_u32(&full[q]), (uint32_t)(issued[q] - 1) & 1);
        }
    } else {
        // ------------------------------------------------ folding threads
        for (int c = 0; c < nchunks; ++c) {
            const int q = c % kStatsStages;
            if (!mbar_wait(smem_u32(&full[q]), (uint32_t)(c / kStatsStages) & 1, &abort_flag)) break;
            const int64_t c0 = (int64_t)c * kStatsChunk;
            const float4 *buf = ring + q * kStatsChunk;
            float x[4 * kStatsVec];
            int base[kStatsVec];
#pragma unroll
            for (int k = 0; k < kStatsVec; ++k) {
                const int i = (int)threadIdx.x + k * kStatsThreads;
                const float4 v =
                    (c0 + i < len) ? buf[i] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                base[k] = (int)(v_begin + c0 + i);
                x[4 * k + 0] = v.x;
                x[4 * k + 1] = v.y;
                x[4 * k + 2] = v.z;
                x[4 * k + 3] = v.w;
            }
            __syncwarp();  // every lane's reads of the stage before the warp hands it back
            if (lane == 0) mbar_arrive(smem_u32(&empty[q]));
            absorb<4 * kStatsVec>(st, x, base);
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
    if (lane == 0 && warp < kStatsThreads / 32) warp_state[warp] = st;
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

// The statistics kernels' shared-memory limit, raised once per device (a function attribute
// belongs to the device's context).
constexpr int kMaxStatsDevices = 64;
cudaError_t ensure_stats_attributes() {
    static std::atomic<int> attr_set[kMaxStatsDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < kMaxStatsDevices && attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const void *fns[4] = {(const void *)row_stats_kernel<1>, (const void *)row_stats_kernel<2>,
                          (const void *)row_stats_kernel<4>, (const void *)row_stats_kernel<8>};
    for (int i = 0; i < 4 && e == cudaSuccess; ++i)
        e = cudaFuncSetAttribute(fns[i], cudaFuncAttributeMaxDynamicSharedMemorySize, kStatsSmem);
    if (e == cudaSuccess && dev < kMaxStatsDevices) attr_set[dev].store(1, std::memory_order_release);
    return e;
}

template <int CLUSTER>
cudaError_t launch_stats(const float *logits, int64_t R, int64_t V, int64_t ldl, float *m, float *lse,
                         float *H, float *kappa, int32_t *argmax, cudaStream_t stream, float4 *state = nullptr,
                         int64_t vocab_offset = 0) {
    const cudaError_t ae = ensure_stats_attributes();
    if (ae != cudaSuccess) return ae;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * CLUSTER), 1, 1);
    cfg.blockDim = dim3(kStatsCtaThreads, 1, 1);
    cfg.dynamicSmemBytes = kStatsSmem;
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
    // (the fused statistics + draw kernel, whose loads keep their bytes in registers) at
    // least 16K entries (64 KiB) per CTA, at most 8 CTAs (the portable cluster limit), and
    // no more than about 1024 CTAs in all: few rows split finer, many rows not at all
    int c = 1;
    while (c < 8 && V / (c * 2) >= 16384 && R * c * 2 <= 1024) c *= 2;
    return c;
}

// CTAs per row of the statistics kernel: at least 16K entries each, at most 8 (the portable
// cluster limit), and rows x CTAs within the CTAs the device holds at once (three per SM):
// one wave, or, when the rows alone fill it, one CTA per row.  Each CTA keeps its bytes in
// flight in shared memory, so a few large CTAs per SM stream as fast as many small ones,
// and a second, partial wave would leave SMs idle at the end.
int bulk_stats_cluster_size(int64_t R, int64_t V) {
    const int64_t slots = (int64_t)device_sm_count() * 3;
    int c = 1;
    while (c < 8 && V / (c * 2) >= 16384 && R * c * 2 <= slots) c *= 2;
    return c;
}

cudaError_t launch_row_stats(const float *logits, int64_t R, int64_t V, int64_t ldl, float *m, float *lse,
                             float *H, float *kappa, int32_t *argmax, cudaStream_t stream) {
    switch (bulk_stats_cluster_size(R, V)) {
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
    switch (bulk_stats_cluster_size(R, V)) {
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
