// The acceptance kernel: one CTA per request (the body in accept.cuh).
#include "accept.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

__global__ void __launch_bounds__(1024) accept_kernel(const AcceptSpec a) {
    extern __shared__ unsigned long long keys[];  // blockDim.x entries
    __shared__ float H_s[1024];
    __shared__ double warp_tot[32];
    __shared__ int first_fail;
    accept_request(a, blockIdx.x, blockDim.x, AcceptSmem{keys, H_s, warp_tot, &first_fail});
}

}  // namespace

int accept_threads(int32_t L_c) {
    int nt = 32;
    while (nt < L_c) nt <<= 1;
    return nt;
}

cudaError_t launch_entropy_accept(const float *H, const float *kappa, int32_t n_req, int32_t L_c,
                                  const float *budgets, int32_t min_accept, int32_t *order,
                                  uint8_t *mask, int32_t *n_accepted, cudaStream_t stream, bool overlap_previous,
                                  const uint8_t *eligible) {
    const int nt = accept_threads(L_c);
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
    const AcceptSpec a{H, kappa, budgets, n_req, L_c, min_accept, order, mask, n_accepted, eligible};
    return cudaLaunchKernelEx(&cfg, accept_kernel, a);
}

}  // namespace dg
