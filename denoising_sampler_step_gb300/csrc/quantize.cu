// Per-row E4M3 quantisation of a bf16 embedding table, the input format of the 8-bit
// soft-embedding product: scale_v = amax_v / 448 (fp32, correctly rounded), Q[v, j] = the
// E4M3 code nearest to W[v, j] / scale_v (correctly rounded fp32 quotient; ties to even,
// magnitudes past 448 saturate); a zero row gets scale 0 and codes 0.  E4M3 is the OCP 8-bit
// format (bias 7, subnormals, no infinity, 448 the largest finite value).  The pages name FP8
// checkpoints (agentlenshq.com, "量子化チェックポイント") without a layout for the table;
// this per-row layout is the reading the product takes.
// One CTA per row (grid-stride): a max-reduction over the row, then the codes, two per thread
// step.  HBM-bound and run once per table.
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

}  // namespace

cudaError_t launch_quantize_e4m3(const uint16_t *W, int64_t V, int64_t d, int64_t ldw, uint8_t *Q, int64_t ldq,
                                 float *scale, cudaStream_t stream) {
    int64_t blocks = V;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (cap > 0 && blocks > cap) blocks = cap;
    quantize_e4m3_kernel<<<(unsigned)blocks, kQuantThreads, 0, stream>>>(W, V, d, ldw, Q, ldq, scale);
    return cudaGetLastError();
}

}  // namespace dg
