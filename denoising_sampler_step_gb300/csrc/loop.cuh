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
// Used by the loop-update kernel and, in a single-pass step, by the CTAs of the reduce
// kernel that run a request's acceptance (right after it, on the mask they wrote).
#pragma once

#include <cstdint>

namespace dg {

struct LoopSpec {
    const int32_t *candidate, *argmax;
    const float *H;
    const uint8_t *mask;
    int32_t L_c, stable_steps, step_limit;
    float threshold;
    int32_t *canvas;  // NULL: no loop state to update
    uint8_t *eligible;
    int32_t *prev, *stable, *steps;
    uint8_t *converged;
};

// Request q's update by the whole CTA (blockDim.x >= L_c, at most 1024 threads); warp_sum:
// 32 doubles of shared memory.  Every thread of the CTA must call it.
__device__ __forceinline__ void loop_update_request(const LoopSpec &l, int q, double *warp_sum) {
    const int tid = (int)threadIdx.x;
    const int64_t base = (int64_t)q * l.L_c;
    const bool in = tid < l.L_c;
    int32_t am = 0;
    double h = 0.0;
    bool same = true;
    if (in) {
        am = l.argmax[base + tid];
        h = (double)l.H[base + tid];
        same = am == l.prev[base + tid];
    }
    const bool all_same = __syncthreads_and(same);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) h += __shfl_down_sync(0xffffffffu, h, off);
    if ((tid & 31) == 0) warp_sum[tid >> 5] = h;
    __syncthreads();
    if (in) {
        if (l.mask[base + tid]) {
            l.canvas[base + tid] = l.candidate[base + tid];
            l.eligible[base + tid] = 0;
        }
        l.prev[base + tid] = am;
    }
    if (tid == 0) {
        double total = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += warp_sum[w];
        const double mean_H = total / (double)l.L_c;
        const int32_t s = all_same ? l.stable[q] + 1 : 0;
        const int32_t n = l.steps[q] + 1;
        l.stable[q] = s;
        l.steps[q] = n;
        l.converged[q] = ((s >= l.stable_steps && mean_H < (double)l.threshold) || n >= l.step_limit) ? 1 : 0;
    }
}

}  // namespace dg
