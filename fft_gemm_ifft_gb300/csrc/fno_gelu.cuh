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

}  // namespace fno
