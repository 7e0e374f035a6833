// Entropy-bound acceptance of one request, as a device function run by one CTA (the
// acceptance kernel, and the single pass's reduce kernel, which runs it in extra CTAs):
// agentlenshq.com, "サンプリングループとエントロピー境界デノイジング".
//
// One thread per (padded) position:
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
#pragma once

#include "dg_common.cuh"

namespace dg {

// The arguments of one acceptance launch (n_req requests of L_c positions).
struct AcceptSpec {
    const float *H, *kappa, *budgets;
    int32_t n_req, L_c, min_accept;
    int32_t *order;
    uint8_t *mask;
    int32_t *n_accepted;
    const uint8_t *eligible;  // NULL: every position
};

// Monotone map from float to uint32: a < b  <=>  key(a) < key(b) for numbers
// (-0 and +0 equal); any NaN maps to the largest key.
__device__ __forceinline__ uint32_t order_bits(float x) {
    if (x != x) return 0xffffffffu;
    const uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Shared memory of one acceptance: NT sort keys, L_c entropies, 32 warp totals, a count.
struct AcceptSmem {
    unsigned long long *keys;
    float *H;
    double *warp_tot;
    int *first_fail;
};

// Request q by the whole CTA.  NT is a power of two >= L_c (at most 1024) and at most
// blockDim.x; threads from NT on hold padding keys and only keep the CTA's barriers.
__device__ __forceinline__ void accept_request(const AcceptSpec &a, int q, int NT, const AcceptSmem &sm) {
    unsigned long long *keys = sm.keys;
    float *H_s = sm.H;
    double *warp_tot = sm.warp_tot;
    int &first_fail = *sm.first_fail;
    const int tid = threadIdx.x;
    const int64_t base = (int64_t)q * a.L_c;

    const bool el = tid < a.L_c && (!a.eligible || a.eligible[base + tid]);
    // ineligible: above every eligible key (NaN included), in position order
    unsigned long long key = (tid >= a.L_c) ? ~0ull
                             : el ? (((unsigned long long)order_bits(a.kappa[base + tid]) << 32) | (unsigned)tid)
                                  : ((0xffffffffull << 32) | 0x80000000u | (unsigned)tid);
    if (tid < a.L_c) H_s[tid] = a.H[base + tid];  // gathered in sorted order below
    const int n_el = __syncthreads_count(el);
    if (tid == 0) first_fail = n_el;

    // bitonic sort: partners within a warp exchange by shuffle, farther ones through shared memory
    for (int k = 2; k <= NT; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            unsigned long long other;
            if (j >= 32) {
                if (tid < NT) keys[tid] = key;
                __syncthreads();
                other = tid < NT ? keys[tid ^ j] : key;
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

    const double B = (double)a.budgets[q];
    if (tid < n_el && !(h <= B)) atomicMin(&first_fail, tid);
    __syncthreads();
    int n = first_fail;
    const int floor_n = min(a.min_accept, n_el);
    if (n < floor_n) n = floor_n;
    if (tid < a.L_c) {
        a.order[base + tid] = pos;
        a.mask[base + pos] = (uint8_t)(tid < n ? 1 : 0);
    }
    if (tid == 0) a.n_accepted[q] = n;
}

}  // namespace dg
