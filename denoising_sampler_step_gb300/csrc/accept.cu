// Entropy-bound acceptance: per request, order the canvas positions from most to
// least confident and accept them until the running entropy would pass the budget
// (agentlenshq.com, "サンプリングループとエントロピー境界デノイジング").
//
// One CTA per request, one thread per (padded) position:
//   1. key = (order-preserving bits of kappa) << 32 | position, so that a single
//      64-bit ascending sort gives confidence descending with ties broken by the
//      lower position; NaN kappa (no distribution) maps above every number;
//   2. bitonic sort of the keys: warp shuffles for partners within a warp, shared memory
//      for the others;
//   3. inclusive prefix sum of H in sorted order, in fp64 (warp shuffles, then the
//      per-warp totals);
//   4. n = the first k whose running sum is not <= B (NaN counts as passing it),
//      raised to min(min_accept, L_c); mask[order_j] = j < n.
// With an eligibility mask (a denoising loop: kept positions are not offered again) the
// ineligible positions sort after every eligible one, in position order, carry no
// entropy into the sum, are never kept, and the counts above use the eligible ones.
#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

// Monotone map from float to uint32: a < b  <=>  key(a) < key(b) for numbers
// (-0 and +0 equal); any NaN maps to the largest key.
__device__ __forceinline__ uint32_t order_bits(float x) {
    if (x != x) return 0xffffffffu;
    const uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(1024)
    accept_kernel(const float *__restrict__ H, const float *__restrict__ kappa, const uint8_t *__restrict__ eligible,
                  int L_c, const float *__restrict__ budgets, int min_accept, int32_t *__restrict__ order,
                  uint8_t *__restrict__ mask, int32_t *__restrict__ n_accepted) {
    extern __shared__ unsigned long long keys[];  // blockDim.x entries
    __shared__ float H_s[1024];
    __shared__ double warp_tot[32];
    __shared__ int first_fail;

    const int q = blockIdx.x;
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const int64_t base = (int64_t)q * L_c;

    const bool el = tid < L_c && (!eligible || eligible[base + tid]);
    // ineligible: above every eligible key (NaN included), in position order
    unsigned long long key = (tid >= L_c) ? ~0ull
                             : el ? (((unsigned long long)order_bits(kappa[base + tid]) << 32) | (unsigned)tid)
                                  : ((0xffffffffull << 32) | 0x80000000u | (unsigned)tid);
    if (tid < L_c) H_s[tid] = H[base + tid];  // gathered in sorted order below
    const int n_el = __syncthreads_count(el);
    if (tid == 0) first_fail = n_el;

    // bitonic sort: partners within a warp exchange by shuffle, farther ones through shared memory
    for (int k = 2; k <= NT; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            unsigned long long other;
            if (j >= 32) {
                keys[tid] = key;
                __syncthreads();
                other = keys[tid ^ j];
                __syncthreads();
            } else {
                other = __shfl_xor_sync(0xffffffffu, key, j);
            }
            const bool ascending = (tid & k) == 0;
            const bool lower = (tid & j) == 0;
            const unsigned long long lo = key < other ? key : other;
            const unsigned long long hi = key < other ? other : key;
            key = (lower == ascending) ? lo : hi;
        }
    }
    __syncthreads();  // H_s and first_fail visible

    const int pos = (int)(key & 0x7fffffffu);
    double h = (tid < n_el) ? (double)H_s[pos] : 0.0;
    // inclusive scan in fp64
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_up_sync(0xffffffffu, h, off);
        if (lane >= off) h += o;
    }
    if (lane == 31) warp_tot[warp] = h;
    __syncthreads();
    if (warp == 0) {
        double w = (lane < NT / 32) ? warp_tot[lane] : 0.0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double o = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += o;
        }
        if (lane < NT / 32) warp_tot[lane] = w;
    }
    __syncthreads();
    if (warp > 0) h += warp_tot[warp - 1];

    const double B = (double)budgets[q];
    if (tid < n_el && !(h <= B)) atomicMin(&first_fail, tid);
    __syncthreads();
    int n = first_fail;
    const int floor_n = min(min_accept, n_el);
    if (n < floor_n) n = floor_n;
    if (tid < L_c) {
        order[base + tid] = pos;
        mask[base + pos] = (uint8_t)(tid < n ? 1 : 0);
    }
    if (tid == 0) n_accepted[q] = n;
}

}  // namespace

cudaError_t launch_entropy_accept(const float *H, const float *kappa, int32_t n_req, int32_t L_c,
                                  const float *budgets, int32_t min_accept, int32_t *order,
                                  uint8_t *mask, int32_t *n_accepted, cudaStream_t stream, bool overlap_previous,
                                  const uint8_t *eligible) {
    int nt = 32;
    while (nt < L_c) nt <<= 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_req, 1, 1);
    cfg.blockDim = dim3((unsigned)nt, 1, 1);
    cfg.dynamicSmemBytes = nt * sizeof(unsigned long long);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    // the previous kernel on the stream signals early that this one may start (it reads
    // only data that kernels before it wrote)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = overlap_previous ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_kernel, H, kappa, eligible, (int)L_c, budgets, (int)min_accept, order,
                              mask, n_accepted);
}

}  // namespace dg
