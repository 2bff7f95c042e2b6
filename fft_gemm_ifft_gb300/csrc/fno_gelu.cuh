// fno_gelu.cuh -- the GELU of the FNO stack, GELU(v) = v/2 (1 + erf(v / sqrt 2)),
// with erf evaluated by the rational approximation 7.1.26 of Abramowitz and
// Stegun's Handbook of Mathematical Functions:
//   erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) e^{-x^2},
//   t = 1 / (1 + p x),  x >= 0,  |error| <= 1.5e-7,
// and erf(-x) = -erf(x).  With r = 1 - erf(|v| / sqrt 2) = poly(t) e^{-v^2/2},
// GELU(v) = v (1 - r/2) for v >= 0 and v r / 2 for v < 0, i.e. max(v, 0) -
// |v| r / 2 (one fused multiply-add, no branch), so the small values on the
// negative side keep their relative precision.  __host__ __device__ so
// that the host check in tests/host can compare it with a double-precision
// erf; on the device the exponential and the reciprocal are the fast
// hardware approximations (a few ulp, far below the formula's own error).
#pragma once

#include <cmath>

namespace fno {

__host__ __device__ __forceinline__ float gelu_erf(float v) {
    constexpr float p = 0.3275911f;
    constexpr float a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f,
                    a4 = -1.453152027f, a5 = 1.061405429f;
    const float x = fabsf(v) * 0.70710678118654752f;
#ifdef __CUDA_ARCH__
    const float t = __fdividef(1.0f, fmaf(p, x, 1.0f));
    const float e = __expf(-x * x);
#else
    const float t = 1.0f / fmaf(p, x, 1.0f);
    const float e = expf(-x * x);
#endif
    const float q = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, a5, a4), a3), a2), a1);
    const float r = q * e;
    return fmaf(-0.5f * fabsf(v), r, fmaxf(v, 0.0f));
}

// Two GELUs at once: the same operations in the same order as gelu_erf, the
// multiplies and fused multiply-adds as packed f32x2 instructions (each lane
// rounded to nearest like its scalar form), the reciprocal and exponential per
// lane, so that each result equals gelu_erf of its input.
namespace gelu2_detail {
__device__ __forceinline__ unsigned long long pk(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk(unsigned long long r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long splat(float a) { return pk(a, a); }
}  // namespace gelu2_detail

__device__ __forceinline__ void gelu_erf2(float &v0, float &v1) {
    using namespace gelu2_detail;
    constexpr float p = 0.3275911f;
    constexpr float a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f,
                    a4 = -1.453152027f, a5 = 1.061405429f;
    const float m0 = fabsf(v0), m1 = fabsf(v1);
    const unsigned long long m = pk(m0, m1);
    const unsigned long long x = mul2(m, splat(0.70710678118654752f));
    float y0, y1, x0, x1;
    upk(fma2(splat(p), x, splat(1.0f)), y0, y1);
    upk(x, x0, x1);
    const unsigned long long t = pk(__fdividef(1.0f, y0), __fdividef(1.0f, y1));
    const unsigned long long e = pk(__expf(-x0 * x0), __expf(-x1 * x1));
    unsigned long long h = fma2(t, splat(a5), splat(a4));
    h = fma2(t, h, splat(a3));
    h = fma2(t, h, splat(a2));
    h = fma2(t, h, splat(a1));
    const unsigned long long r = mul2(mul2(t, h), e);
    const unsigned long long hm = mul2(splat(-0.5f), m);
    upk(fma2(hm, r, pk(fmaxf(v0, 0.0f), fmaxf(v1, 0.0f))), v0, v1);
}

}  // namespace fno
