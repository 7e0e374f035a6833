// Sum of per-slice partial products on one device, then the normaliser:
// E = gamma * (S_0 + ... + S_{T-1}), added in index order (calvarado04.com,
// "The fix": each rank's partial over its vocabulary slice, one sum, gamma after it).
// A memory-bound elementwise kernel: T reads and one write per element.
#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

struct PartialPtrs {
    const float *p[kMaxPartials];
};

__global__ void sum_partials_kernel(const __grid_constant__ PartialPtrs P, int T, int64_t R, int64_t d,
                                    int64_t ldp, float gamma, float *__restrict__ out, int64_t ldo, int vec4) {
    const int64_t cols = vec4 ? d / 4 : d;
    const int64_t total = R * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        if (vec4) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int t = 0; t < T; ++t) {
                const float4 v = *reinterpret_cast<const float4 *>(P.p[t] + r * ldp + 4 * c);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            *reinterpret_cast<float4 *>(out + r * ldo + 4 * c) =
                make_float4(gamma * acc.x, gamma * acc.y, gamma * acc.z, gamma * acc.w);
        } else {
            float acc = 0.f;
            for (int t = 0; t < T; ++t) acc += P.p[t][r * ldp + c];
            out[r * ldo + c] = gamma * acc;
        }
    }
}

__global__ void fill_zero_kernel(float *__restrict__ out, int64_t R, int64_t d, int64_t ldo) {
    const int64_t total = R * d;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x)
        out[(i / d) * ldo + (i % d)] = 0.0f;
}

unsigned grid_for(int64_t work, int threads) {
    const int64_t cap = (int64_t)(device_sm_count() > 0 ? device_sm_count() : 1) * 8;
    int64_t g = (work + threads - 1) / threads;
    if (g > cap) g = cap;
    return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_sum_partials(const float *const *partials, int32_t T, int64_t R, int64_t d, int64_t ldp,
                                float gamma, float *out, int64_t ldo, cudaStream_t stream) {
    PartialPtrs P = {};
    int vec4 = (d % 4 == 0 && ldp % 4 == 0 && ldo % 4 == 0 && ((uintptr_t)out & 15) == 0);
    for (int t = 0; t < T; ++t) {
        P.p[t] = partials[t];
        if ((uintptr_t)partials[t] & 15) vec4 = 0;
    }
    const int64_t work = R * (vec4 ? d / 4 : d);
    sum_partials_kernel<<<grid_for(work, 256), 256, 0, stream>>>(P, T, R, d, ldp, gamma, out, ldo, vec4);
    return cudaGetLastError();
}

namespace {

// The timeout path of the bounded barrier waits, on a barrier whose phase never completes
// (count 2, one arrival): the wait gives up after limit_ns and records the timeout.
__global__ void wait_timeout_check_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 2);
    fence_mbar_init();
    mbar_arrive(b);
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(b, 0)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            record_timeout();
            return;
        }
    }
}

}  // namespace

cudaError_t launch_wait_timeout_check(uint32_t limit_us, cudaStream_t stream) {
    wait_timeout_check_kernel<<<1, 1, 0, stream>>>(1000ull * limit_us);
    return cudaGetLastError();
}

cudaError_t launch_fill_zero(float *out, int64_t R, int64_t d, int64_t ldo, cudaStream_t stream) {
    fill_zero_kernel<<<grid_for(R * d, 256), 256, 0, stream>>>(out, R, d, ldo);
    return cudaGetLastError();
}

}  // namespace dg
