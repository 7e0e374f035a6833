// The denoising-loop update as its own kernel (the steps that do not run it inside the
// reduce kernel): one CTA per request, as loop_update_request describes.
#include "dg_common.cuh"
#include "dg_internal.h"
#include "loop.cuh"

namespace dg {

namespace {

__global__ void __launch_bounds__(1024)
    loop_update_kernel(const int32_t *__restrict__ candidate, const int32_t *__restrict__ argmax,
                       const float *__restrict__ H,
                       const uint8_t *__restrict__ mask, int L_c, int stable_steps, float threshold, int step_limit,
                       int32_t *__restrict__ canvas, uint8_t *__restrict__ eligible, int32_t *__restrict__ prev,
                       int32_t *__restrict__ stable, int32_t *__restrict__ steps, uint8_t *__restrict__ converged) {
    __shared__ double warp_sum[32];
    const LoopSpec l{candidate, argmax, H, mask, L_c, stable_steps, step_limit, threshold,
                     canvas, eligible, prev, stable, steps, converged};
    loop_update_request(l, (int)blockIdx.x, warp_sum);
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
