// Online softmax statistics of one row (shared by the statistics kernel, the fused
// statistics + sampling kernel and the product's fallback fold: the same arithmetic, so
// their maxima and argmax agree exactly and their sums up to the order in which each
// kernel visits the entries).
//
// Each thread keeps an online state (m, a, rest, t) over the entries it saw:
//   m    = running max, a = index of its first occurrence,
//   rest = sum over the entries other than a of exp(l - m),
//   t    = sum over all entries of exp(l - m) * (l - m)   (<= 0);
// keeping the argmax's own 1 out of `rest` preserves kappa = log1p(rest) for rows that
// are nearly one-hot.  Final: lnZ = log1p(rest), lse = m + lnZ,
// H = lnZ - t / (1 + rest), kappa = lnZ.
#pragma once

#include <float.h>

#include "dg_common.cuh"

namespace dg {
namespace rowstate {

struct RowState {
    float m;
    int a;
    float rest;
    float t;
};

__device__ __forceinline__ float4 ld_stream_v4(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// A := A merged with B.  The larger max wins; equal maxima keep the lower index.
__device__ __forceinline__ void merge(RowState &A, const RowState &B) {
    const bool b_wins = (B.m > A.m) || (B.m == A.m && B.a < A.a);
    RowState hi = b_wins ? B : A;
    const RowState lo = b_wins ? A : B;
    if (lo.m != -INFINITY) {
        const float dm = lo.m - hi.m;              // <= 0
        const float s = ex2_approx(dm * kLog2e);   // rescale lo to hi's max
        const float S_lo = lo.rest + 1.0f;         // lo's full sum, its argmax included
        hi.rest = fmaf(s, S_lo, hi.rest);
        hi.t = fmaf(s, fmaf(dm, S_lo, lo.t), hi.t);
    }
    A = hi;
}

__device__ __forceinline__ RowState shfl_down(const RowState &s, int off) {
    RowState o;
    o.m = __shfl_down_sync(0xffffffffu, s.m, off);
    o.a = __shfl_down_sync(0xffffffffu, s.a, off);
    o.rest = __shfl_down_sync(0xffffffffu, s.rest, off);
    o.t = __shfl_down_sync(0xffffffffu, s.t, off);
    return o;
}

// Folds N values x[j] (vocabulary index 4*base[j/4] + j%4, increasing in j) into st.
template <int N>
__device__ __forceinline__ void absorb(RowState &st, float (&x)[N], const int (&base)[N / 4]) {
    float bm = x[0];
#pragma unroll
    for (int j = 1; j < N; ++j) bm = fmaxf(bm, x[j]);
    if (bm > st.m) {
        // a new maximum: rebase the state, then take its first occurrence out of the sums
        if (st.m == -INFINITY) {
            st.rest = 0.0f;
            st.t = 0.0f;
        } else {
            const float dm = st.m - bm;
            const float s = ex2_approx(dm * kLog2e);
            const float S = st.rest + 1.0f;
            st.t = s * fmaf(dm, S, st.t);
            st.rest = s * S;
        }
        st.m = bm;
        int ja = N;
#pragma unroll
        for (int j = N - 1; j >= 0; --j)
            if (x[j] == bm) ja = j;
#pragma unroll
        for (int j = 0; j < N; ++j)
            if (j == ja) {
                st.a = 4 * base[j / 4] + (j % 4);
                x[j] = -INFINITY;
            }
    }
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const float d = fmaxf(x[j] - st.m, -FLT_MAX);  // -inf entries: exp gives 0 and 0*d = 0
        const float e = ex2_approx(d * kLog2e);
        st.rest += e;
        st.t = fmaf(e, d, st.t);
    }
}

__device__ __forceinline__ RowState empty_row_state() { return RowState{-INFINITY, 0x7fffffff, 0.0f, 0.0f}; }

}  // namespace rowstate
}  // namespace dg
