// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2,
// 3", SC 2011) and the uniforms the samplers take from it: u = ((x >> 9) + 1/2) 2^-23 and
// E = -ln u.  Shared by the stand-alone draw and the single-pass product's folded draw.
#pragma once

#include <stdint.h>

#include "dg_common.cuh"

namespace dg {
namespace philox {

constexpr float kLn2 = 0.69314718055994531f;
constexpr uint32_t kGroupCounter = 0x80000000u;  // counter word 0 of the group uniforms

struct Philox {
    uint32_t x0, x1, x2, x3;
};

__device__ __forceinline__ Philox philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c0 = n0;
        c1 = (uint32_t)p1;
        c2 = n2;
        c3 = (uint32_t)p0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return {c0, c1, c2, c3};
}

// E = -ln u for u = ((x >> 9) + 1/2) 2^-23, built without an integer conversion:
// f = 1 + (x >> 9) 2^-23 is the float with those mantissa bits, and f - (1 - 2^-24) = u
// exactly (both operands and the result are fp32 numbers within a factor of two).
// Near u = 1 (t = 1 - u < 1/64, exact) the series t (1 + t/2 + t^2/3) of -ln(1 - t)
// (relative error below t^3 / 4); elsewhere the fast logarithm, whose absolute error is
// then small against |ln u| >= 1/64.
__device__ __forceinline__ float neg_log_uniform(uint32_t x) {
    const float f = __uint_as_float(0x3F800000u | (x >> 9));
    const float u = f - 0.99999994039535522f;  // 1 - 2^-24
    const float t = 1.0f - u;
    return t < 0.015625f ? t * fmaf(t, fmaf(t, 0.333333343f, 0.5f), 1.0f) : -kLn2 * __log2f(u);
}

__device__ __forceinline__ uint32_t philox_word(const Philox &w, int j) {
    return j == 0 ? w.x0 : j == 1 ? w.x1 : j == 2 ? w.x2 : w.x3;
}

}  // namespace philox
}  // namespace dg
