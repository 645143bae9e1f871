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

// gelu_as on a packed pair, the same operations in the same order (so the
// same bits as two gelu_as calls).  Two rewrites keep it free of sign
// operations: x (x c) equals |x| (|x| c) exactly, and 1 - q t e is formed
// as q t e - 1, whose magnitude copysign takes.
__device__ __forceinline__ float2 gelu_as2(float2 u) {
    const float2 x = mul2(u, make_float2(0.70710678118654752f, 0.70710678118654752f));
    const float2 den = fma2(make_float2(0.3275911f, 0.3275911f),
                            make_float2(fabsf(x.x), fabsf(x.y)), make_float2(1.0f, 1.0f));
    const float2 t = make_float2(rcp_approx(den.x), rcp_approx(den.y));
    float2 q = fma2(t, make_float2(1.061405429f, 1.061405429f),
                    make_float2(-1.453152027f, -1.453152027f));
    q = fma2(t, q, make_float2(1.421413741f, 1.421413741f));
    q = fma2(t, q, make_float2(-0.284496736f, -0.284496736f));
    q = fma2(t, q, make_float2(0.254829592f, 0.254829592f));
    const float2 m = mul2(x, mul2(x, make_float2(-1.4426950408889634f, -1.4426950408889634f)));
    const float2 e = make_float2(ex2a(m.x), ex2a(m.y));
    const float2 r = fma2(mul2(q, t), e, make_float2(-1.0f, -1.0f));
    const float2 erf = make_float2(copysignf(r.x, x.x), copysignf(r.y, x.y));
    return mul2(u, fma2(make_float2(0.5f, 0.5f), erf, make_float2(0.5f, 0.5f)));
}

// Taylor coefficients of d -> GELU(y + d) - GELU(y) about d = 0 for small
// perturbations (the coefficient kernel in reforward.cu states them), for
// blocks of four channels, in two arrays of nblk entries laid out one after
// the other: c1 (float4) and c2, c3 as fp16 pairs (c2.x c2.y | c2.z c2.w |
// c3.x c3.y | c3.z c3.w, first lane in the low half); 8 bytes per channel,
// read once per draw by the on-chip producers.  With |d| <= 5.77 sigma <=
// 0.15 the cubic drops d^4 G(y)/24 (|G|/24 < 0.07: under 1e-8 at a
// typical draw, |d| = sigma = 0.02, and 3.4e-5 at the largest), and the fp16
// rounding of c2 and c3 (|c2| <= 0.4, |c3| <= 0.13, both in fp16's normal
// range but for values whose terms are negligible) moves the difference by
// under 2^-11 of its d^2 and d^3 terms.  The first error is even in d, so it
// does not bias the estimate, which weights each draw by its own a; the
// estimator's parity tests bound what is left.  (bf16, with 2^-9, measured
// five times the ĝ error of fp32 coefficients; fp16 is below their noise.)
struct GeluCoefs {
    const float4* c1;
    const uint4* c23;
};

__host__ __device__ inline GeluCoefs gelu_coefs(const void* base, int64_t nblk) {
    const float4* f = static_cast<const float4*>(base);
    return GeluCoefs{f, reinterpret_cast<const uint4*>(f + nblk)};
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t u) {
    return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// GELU(y + d) - GELU(y) = d (c1 + d (c2 + d c3)) for channel pairs (0, 1)
// and (2, 3) of one block, d = e per channel.
__device__ __forceinline__ void gelu_taylor_pairs(float4 c1, uint4 c23, float4 e, float2& d01,
                                                  float2& d23) {
    const float2 e01 = make_float2(e.x, e.y), e23 = make_float2(e.z, e.w);
    float2 q01 = fma2(e01, f16x2_to_float2(c23.z), f16x2_to_float2(c23.x));
    float2 q23 = fma2(e23, f16x2_to_float2(c23.w), f16x2_to_float2(c23.y));
    q01 = fma2(e01, q01, make_float2(c1.x, c1.y));
    q23 = fma2(e23, q23, make_float2(c1.z, c1.w));
    d01 = mul2(e01, q01);
    d23 = mul2(e23, q23);
}

}  // namespace dust
