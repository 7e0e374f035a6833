// Per-row E4M3 quantisation of a bf16 embedding table, the input format of the 8-bit
// soft-embedding product: scale_v = amax_v / 448 (fp32, correctly rounded), Q[v, j] = the
// E4M3 code nearest to W[v, j] / scale_v (correctly rounded fp32 quotient; ties to even,
// magnitudes past 448 saturate); a zero row gets scale 0 and codes 0.  E4M3 is the OCP 8-bit
// format (bias 7, subnormals, no infinity, 448 the largest finite value).  The pages name FP8
// checkpoints (agentlenshq.com, "量子化チェックポイント") without a layout for the table;
// this per-row layout is the reading the product takes.
// Rows of whole 16-byte groups take a warp each (below); others one CTA per row (grid-stride):
// a max-reduction over the row, then the codes, two per thread step.  HBM-bound and run once
// per table.
#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ float bf16_value(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__global__ void __launch_bounds__(kQuantThreads)
    quantize_e4m3_kernel(const uint16_t *__restrict__ W, int64_t V, int64_t d, int64_t ldw, uint8_t *__restrict__ Q,
                         int64_t ldq, float *__restrict__ scale) {
    __shared__ float warp_max[kQuantThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t v = blockIdx.x; v < V; v += gridDim.x) {
        const uint16_t *w = W + v * ldw;
        float amax = 0.0f;
        for (int64_t j = threadIdx.x; j < d; j += kQuantThreads) amax = fmaxf(amax, fabsf(bf16_value(w[j])));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) warp_max[warp] = amax;
        __syncthreads();
        amax = warp_max[0];
#pragma unroll
        for (int i = 1; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, warp_max[i]);
        __syncthreads();  // warp_max is rewritten by the next row
        const float s = __fdiv_rn(amax, 448.0f);
        if (threadIdx.x == 0) scale[v] = s;
        uint8_t *q = Q + v * ldq;
        for (int64_t j = 2 * (int64_t)threadIdx.x; j < d; j += 2 * kQuantThreads) {
            const bool two = j + 1 < d;
            float x0 = 0.0f, x1 = 0.0f;
            if (s > 0.0f) {
                x0 = __fdiv_rn(bf16_value(w[j]), s);
                if (two) x1 = __fdiv_rn(bf16_value(w[j + 1]), s);
            }
            const uint32_t c = pack_e4m3x2(x0, x1);
            if (two)
                *reinterpret_cast<uint16_t *>(q + j) = (uint16_t)c;  // j is even and ldq is even
            else
                q[j] = (uint8_t)c;
        }
    }
}

// The same with a warp per row and 16-byte accesses (8 entries per lane and step), for rows
// whose bases and lengths are multiples of 8 entries: the maximum over the row, then the
// codes from a second read of the row (it is in L1 by then).
__global__ void __launch_bounds__(kQuantThreads)
    quantize_e4m3_vec_kernel(const uint16_t *__restrict__ W, int64_t V, int64_t d, int64_t ldw,
                             uint8_t *__restrict__ Q, int64_t ldq, float *__restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kQuantThreads / 32);
    for (int64_t v = (int64_t)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5); v < V; v += warps) {
        const uint4 *w = reinterpret_cast<const uint4 *>(W + v * ldw);
        const int64_t n8 = d / 8;
        float amax = 0.0f;
        for (int64_t c = lane; c < n8; c += 32) {
            const uint4 u = __ldg(w + c);
            const uint32_t h[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int t = 0; t < 4; ++t)
                amax = fmaxf(amax, fmaxf(fabsf(bf16_value((uint16_t)(h[t] & 0xFFFFu))), fabsf(bf16_value((uint16_t)(h[t] >> 16)))));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float s = __fdiv_rn(amax, 448.0f);
        if (lane == 0) scale[v] = s;
        uint2 *q = reinterpret_cast<uint2 *>(Q + v * ldq);
        for (int64_t c = lane; c < n8; c += 32) {
            const uint4 u = __ldg(w + c);
            const uint32_t h[4] = {u.x, u.y, u.z, u.w};
            uint32_t codes[2] = {0u, 0u};
            if (s > 0.0f) {
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float x0 = __fdiv_rn(bf16_value((uint16_t)(h[t] & 0xFFFFu)), s);
                    const float x1 = __fdiv_rn(bf16_value((uint16_t)(h[t] >> 16)), s);
                    codes[t >> 1] |= pack_e4m3x2(x0, x1) << (16 * (t & 1));
                }
            }
            q[c] = make_uint2(codes[0], codes[1]);
        }
    }
}

}  // namespace

cudaError_t launch_quantize_e4m3(const uint16_t *W, int64_t V, int64_t d, int64_t ldw, uint8_t *Q, int64_t ldq,
                                 float *scale, cudaStream_t stream) {
    const int64_t cap = (int64_t)device_sm_count() * 16;
    const bool vec = (reinterpret_cast<uintptr_t>(W) & 15) == 0 && (ldw & 7) == 0 && (d & 7) == 0 &&
                     (reinterpret_cast<uintptr_t>(Q) & 7) == 0 && (ldq & 7) == 0;
    if (vec) {
        int64_t blocks = (V + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
        if (cap > 0 && blocks > cap) blocks = cap;
        quantize_e4m3_vec_kernel<<<(unsigned)blocks, kQuantThreads, 0, stream>>>(W, V, d, ldw, Q, ldq, scale);
    } else {
        int64_t blocks = V;
        if (cap > 0 && blocks > cap) blocks = cap;
        quantize_e4m3_kernel<<<(unsigned)blocks, kQuantThreads, 0, stream>>>(W, V, d, ldw, Q, ldq, scale);
    }
    return cudaGetLastError();
}

}  // namespace dg
