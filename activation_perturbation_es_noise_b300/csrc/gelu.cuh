// gelu.cuh -- the GELU of the interior layer's fixed downstream (exact-erf
// form, GELU(u) = u Phi(u)), on a one-form erf approximation.
#pragma once

#include "noise.cuh"

namespace dust {

__device__ __forceinline__ float ex2a(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// erf by the rational-exponential approximation of Abramowitz & Stegun,
// Handbook of Mathematical Functions, 7.1.26 (after Hastings):
// erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-x^2),
// t = 1 / (1 + p x) for x >= 0, odd extension; |error| < 1.5e-7.  One form on
// the whole line, so lanes do not diverge.  The clean GELU(y1) is computed
// with the same function, so its smooth error largely cancels in the
// difference GELU(y1 + sigma a) - GELU(y1) (about 4e-7 relative, float64 model).
__device__ __forceinline__ float erf_as(float x) {
    const float ax = fabsf(x);
    const float t = rcp_approx(fmaf(0.3275911f, ax, 1.0f));
    float q = fmaf(t, 1.061405429f, -1.453152027f);
    q = fmaf(t, q, 1.421413741f);
    q = fmaf(t, q, -0.284496736f);
    q = fmaf(t, q, 0.254829592f);
    const float e = ex2a(ax * (ax * -1.4426950408889634f));
    return copysignf(fmaf(-q * t, e, 1.0f), x);
}

// GELU(u) = u Phi(u) = u (1 + erf(u / sqrt 2)) / 2.
__device__ __forceinline__ float gelu_as(float u) {
    return u * fmaf(0.5f, erf_as(u * 0.70710678118654752f), 0.5f);
}

}  // namespace dust
