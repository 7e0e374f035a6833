// Denoising-loop state after a step (agentlenshq.com, "サンプリングループとエントロピー境界
// デノイジング": kept tokens; a canvas has converged when the argmax predictions have been
// stable for several steps and the mean entropy per token is below a threshold, or when
// the step limit is reached).
//
// One CTA per request, one thread per position:
//   canvas[p] = candidate[p] and eligible[p] = 0 where the step kept p (mask[p]);
//   stable    = stable + 1 if every argmax equals the previous step's, else 0;
//   prev[p]   = argmax[p];  steps += 1;
//   converged = (stable >= stable_steps && mean H < threshold) || steps >= step_limit,
//   mean H summed in fp64 in a fixed order (warp shuffles, then the warp totals in order).
#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

__global__ void __launch_bounds__(1024)
    loop_update_kernel(const int32_t *__restrict__ candidate, const int32_t *__restrict__ argmax,
                       const float *__restrict__ H,
                       const uint8_t *__restrict__ mask, int L_c, int stable_steps, float threshold, int step_limit,
                       int32_t *__restrict__ canvas, uint8_t *__restrict__ eligible, int32_t *__restrict__ prev,
                       int32_t *__restrict__ stable, int32_t *__restrict__ steps, uint8_t *__restrict__ converged) {
    __shared__ double warp_sum[32];
    const int q = blockIdx.x, tid = threadIdx.x;
    const int64_t base = (int64_t)q * L_c;
    const bool in = tid < L_c;
    int32_t am = 0;
    double h = 0.0;
    bool same = true;
    if (in) {
        am = argmax[base + tid];
        h = (double)H[base + tid];
        same = am == prev[base + tid];
    }
    const bool all_same = __syncthreads_and(same);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) h += __shfl_down_sync(0xffffffffu, h, off);
    if ((tid & 31) == 0) warp_sum[tid >> 5] = h;
    __syncthreads();
    if (in) {
        if (mask[base + tid]) {
            canvas[base + tid] = candidate[base + tid];
            eligible[base + tid] = 0;
        }
        prev[base + tid] = am;
    }
    if (tid == 0) {
        double total = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += warp_sum[w];
        const double mean_H = total / (double)L_c;
        const int32_t s = all_same ? stable[q] + 1 : 0;
        const int32_t n = steps[q] + 1;
        stable[q] = s;
        steps[q] = n;
        converged[q] = ((s >= stable_steps && mean_H < (double)threshold) || n >= step_limit) ? 1 : 0;
    }
}

}  // namespace

cudaError_t launch_loop_update(const int32_t *candidate, const int32_t *argmax, const float *H, const uint8_t *mask,
                               int32_t n_req, int32_t L_c, int32_t stable_steps, float entropy_threshold,
                               int32_t step_limit, int32_t *canvas, uint8_t *eligible, int32_t *prev_argmax,
                               int32_t *stable, int32_t *steps, uint8_t *converged, cudaStream_t stream) {
    int nt = 32;
    while (nt < L_c) nt <<= 1;
    loop_update_kernel<<<(unsigned)n_req, (unsigned)nt, 0, stream>>>(
        candidate, argmax, H, mask, (int)L_c, (int)stable_steps, entropy_threshold, (int)step_limit, canvas, eligible,
        prev_argmax, stable, steps, converged);
    return cudaGetLastError();
}

}  // namespace dg
