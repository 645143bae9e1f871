// noise.cuh -- counter-based Gaussian noise for the activation perturbation
// y_t + sigma a_t (laoyaoba.com article, section 机制拆解; Dust translation,
// hn.213312.xyz, §2.2 信用分配).  The pages only say the noise is Gaussian and
// independent per token and per linear layer; it is regenerated from a
// counter here so that it is never stored.
//
// Generator: Philox4x32-10 as defined by Salmon, Moraes, Dror and Shaw,
// "Parallel random numbers: as easy as 1, 2, 3" (SC'11).  A round multiplies
// counter words 0 and 2 by two fixed odd constants into 64-bit products; the
// next state is (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1,
// lo(M0 x0)); the key is bumped by the Weyl constants (golden ratio and
// sqrt(3) - 1 in 32-bit fixed point) after every round.
//
// Counter of channel block j (channels 4j .. 4j+3) of token t, draw i, layer
// L: (j, t, i, L); key (seed low word, seed high word).  Uniform of a word w:
// ((w >> 9) + 0.5) 2^-23, in [2^-24, 1 - 2^-24].  Box-Muller (Box & Muller,
// 1958) turns words (0, 1) into channels 4j, 4j+1 and words (2, 3) into
// 4j+2, 4j+3: rho = sqrt(-2 ln u_even), theta = 2 pi u_odd, (rho cos theta,
// rho sin theta).
#pragma once

#include <stdint.h>

#include "pairs.cuh"

namespace dust {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// Round keys of all ten rounds, computed once on the host and passed as a
// kernel parameter so that the xors read them from the constant bank.
struct PhiloxKeys {
    uint32_t k0[10];
    uint32_t k1[10];
};

inline PhiloxKeys philox_round_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t a = static_cast<uint32_t>(seed & 0xFFFFFFFFu);
    uint32_t b = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        k.k0[r] = a;
        k.k1[r] = b;
        a += kPhiloxW0;
        b += kPhiloxW1;
    }
    return k;
}

__device__ __forceinline__ void philox_round(uint32_t& x0, uint32_t& x1, uint32_t& x2,
                                             uint32_t& x3, uint32_t k0, uint32_t k1) {
    const uint64_t p0 = static_cast<uint64_t>(x0) * kPhiloxM0;
    const uint64_t p1 = static_cast<uint64_t>(x2) * kPhiloxM1;
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ x1 ^ k0;
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ x3 ^ k1;
    x0 = n0;
    x1 = static_cast<uint32_t>(p1);
    x2 = n2;
    x3 = static_cast<uint32_t>(p0);
}

// The first round split into its two independent halves.  With the counter
// (j, t, i, L), the half that multiplies word 0 depends only on the channel
// block j and the layer, the other only on the draw i and the token t, so
// kernels compute each half once and reuse it across the other loop.
struct BlockHalf {  // words 2, 3 after round 1
    uint32_t x2, x3;
};
struct DrawHalf {  // words 0, 1 after round 1
    uint32_t x0, x1;
};

__device__ __forceinline__ BlockHalf philox_block_half(uint32_t j, uint32_t layer,
                                                       const PhiloxKeys& k) {
    const uint64_t p0 = static_cast<uint64_t>(j) * kPhiloxM0;
    return {static_cast<uint32_t>(p0 >> 32) ^ layer ^ k.k1[0], static_cast<uint32_t>(p0)};
}

__device__ __forceinline__ DrawHalf philox_draw_half(uint32_t draw, uint32_t token,
                                                     const PhiloxKeys& k) {
    const uint64_t p1 = static_cast<uint64_t>(draw) * kPhiloxM1;
    return {static_cast<uint32_t>(p1 >> 32) ^ token ^ k.k0[0], static_cast<uint32_t>(p1)};
}

// Rounds 2..10 from the state after round 1.
__device__ __forceinline__ uint4 philox_rest(DrawHalf d, BlockHalf b, const PhiloxKeys& k) {
    uint32_t x0 = d.x0, x1 = d.x1, x2 = b.x2, x3 = b.x3;
#pragma unroll
    for (int r = 1; r < 10; ++r) philox_round(x0, x1, x2, x3, k.k0[r], k.k1[r]);
    return make_uint4(x0, x1, x2, x3);
}

// The second round splits too: from the state after round 1, its product of
// word 2 depends only on the block half and its product of word 0 only on
// the draw half.  Kernels that pair every block with several draws (and
// every draw with several blocks) compute each side once.
struct BlockHalf2 {  // hi(M1 x2) ^ k0[1], lo(M1 x2), x3 ^ k1[1] after round 1
    uint32_t bh, bl, b3;
};
struct DrawHalf2 {  // hi(M0 x0), lo(M0 x0), x1 after round 1
    uint32_t dh, dl, d1;
};

__device__ __forceinline__ BlockHalf2 philox_block_half2(BlockHalf b, const PhiloxKeys& k) {
    const uint64_t p1 = static_cast<uint64_t>(b.x2) * kPhiloxM1;
    return {static_cast<uint32_t>(p1 >> 32) ^ k.k0[1], static_cast<uint32_t>(p1), b.x3 ^ k.k1[1]};
}

__device__ __forceinline__ DrawHalf2 philox_draw_half2(DrawHalf d) {
    const uint64_t p0 = static_cast<uint64_t>(d.x0) * kPhiloxM0;
    return {static_cast<uint32_t>(p0 >> 32), static_cast<uint32_t>(p0), d.x1};
}

// Rounds 3..10 from the two halves of round 2 (the same words as philox_rest).
__device__ __forceinline__ uint4 philox_rest2(DrawHalf2 d, BlockHalf2 b, const PhiloxKeys& k) {
    uint32_t x0 = b.bh ^ d.d1, x1 = b.bl, x2 = d.dh ^ b.b3, x3 = d.dl;
#pragma unroll
    for (int r = 2; r < 10; ++r) philox_round(x0, x1, x2, x3, k.k0[r], k.k1[r]);
    return make_uint4(x0, x1, x2, x3);
}

__device__ __forceinline__ uint4 philox4x32_10(uint32_t j, uint32_t token, uint32_t draw,
                                               uint32_t layer, const PhiloxKeys& k) {
    return philox_rest(philox_draw_half(draw, token, k), philox_block_half(j, layer, k), k);
}

// ((w >> 9) + 0.5) 2^-23, exactly: the 23 high bits of w as the mantissa of
// a float in [1, 2), minus (1 - 2^-24).  The difference (2m + 1) 2^-24 has at
// most 24 significant bits, so the subtraction is exact.  (Shift and or run on
// the integer ALU, leaving the multiply pipe to Philox.)
__device__ __forceinline__ float word_to_uniform(uint32_t w) {
    const float f = __uint_as_float((w >> 9) | 0x3F800000u);
    return __fadd_rn(f, -0x1.fffffep-1f);
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rsqrt_approx(float x) {
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// -2 ln u for a positive normal float u (the noise uses u in [2^-24, 1)).
// u = 2^k f with f in [sqrt(1/2),
// sqrt(2)) (k from the exponent field, f by moving the exponent), and
// ln f = 2 atanh(s), s = (f - 1) / (f + 1), |s| <= 3 - 2 sqrt(2).  atanh(s)/s
// is the series 1 + s^2/3 + s^4/5 + ... ; its first four terms, refitted for
// the interval by least squares on Chebyshev nodes, stay within 1e-9
// relative.  f - 1 is exact (Sterbenz), so u close to 1 keeps full relative
// accuracy.  k is turned into a float by adding it to the bits of 1.5 * 2^23.
__device__ __forceinline__ float neg2_log_unit(float u) {
    const int32_t bits = __float_as_int(u);
    const int32_t k = (bits - 0x3F3504F3) >> 23;
    const float f = __int_as_float(bits - (k << 23));
    const float kf = __int_as_float(0x4B400000 + k) - 12582912.0f;
    const float s = (f - 1.0f) * rcp_approx(f + 1.0f);
    const float z = s * s;
    float p = fmaf(z, 0.14935468f, 0.19988787f);
    p = fmaf(z, p, 0.33333388f);
    p = fmaf(z, p, 1.0f);
    return fmaf(s * p, -4.0f, kf * -1.3862943611198906f);  // -2 k ln 2 - 4 s p
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// -2 ln u for the uniforms of the noise, u in [2^-24, 1 - 2^-24].  Near 1
// (v = 1 - u < 1/50, exact since u > 1/2) the series -ln(1 - v) = v + v^2/2
// + v^3/3 (the dropped terms are below 2.1e-6 of the sum); elsewhere the
// hardware log2, whose absolute error (about 3e-7 in -2 ln u) moves the radius
// by at most 1e-6 because the radius is at least 0.2 there.  Both are
// computed and one is selected, so lanes do not diverge.
__device__ __forceinline__ float neg2_log_uniform(float u) {
    const float v = 1.0f - u;
    const float near1 = v * fmaf(v, fmaf(v, 2.0f / 3.0f, 1.0f), 2.0f);
    const float far = lg2_approx(u) * -1.3862943611198906f;  // -2 ln 2 log2 u
    return v < 0.02f ? near1 : far;
}

// Box-Muller pair from two words: rho = sqrt(-2 ln u_even), theta =
// 2 pi u_odd; a_cos = rho cos theta, a_sin = rho sin theta, both multiplied by
// `scale` (a kernel that only ever uses s a folds s into the radius).  With
// theta' = 2 pi u_odd - pi in (-pi, pi), cos theta = -cos theta' and
// sin theta = -sin theta'; sin and cos of theta' come from the hardware
// approximations (absolute error about 4e-7 on that interval), so the normals
// are within about 3e-6 of the exact ones at the largest radius (5.77).
__device__ __forceinline__ void box_muller(uint32_t w_even, uint32_t w_odd, float& a_cos,
                                           float& a_sin, float scale = 1.0f) {
    const float x = neg2_log_uniform(word_to_uniform(w_even));
    const float neg_rho = (x * rsqrt_approx(x)) * -scale;
    const float th = fmaf(word_to_uniform(w_odd), 6.2831853071795865f, -3.1415926535897932f);
    float s, c;
    __sincosf(th, &s, &c);
    a_cos = neg_rho * c;
    a_sin = neg_rho * s;
}

__device__ __forceinline__ float4 words_to_normals(uint4 w, float scale = 1.0f) {
    float4 a;
    box_muller(w.x, w.y, a.x, a.y, scale);
    box_muller(w.z, w.w, a.z, a.w, scale);
    return a;
}

// The same Box-Muller pair in fewer operations, for kernels whose outputs are
// held only to the estimate's tolerance (their own parity tests against the
// oracle bound the effect):
//  - the float 1 + (w >> 9) 2^-23 of a word is one funnel shift (the word's
//    23 high bits under the exponent bits of 1.0);
//  - x = scale^2 (-2 ln u) is the hardware log2 times one constant,
//    clog = -2 ln(2) scale^2, with no series near u = 1, and the radius is the
//    hardware square root of x.  Run on every one of the 2^23 values the
//    uniform map can produce, the log2 is negative for all of them (so x > 0
//    and no clamp is needed) and within 7.6e-8 of log2 u wherever u > 0.98
//    (2e-6 overall, where |log2 u| is up to 24);
//  - theta' = 2 pi u_odd - pi = 2 pi f_odd - 3 pi + 2 pi 2^-24 is one fma on
//    the float f_odd; its two rounded constants leave under 9e-7 in theta',
//    5e-6 on the largest normal.
__device__ __forceinline__ float unit_float(uint32_t w) {
    return __uint_as_float(__funnelshift_r(w, 0x7Fu, 9));
}

__device__ __forceinline__ float sqrt_approx(float x) {
    float y;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void box_muller_fast(uint32_t w_even, uint32_t w_odd, float& a_cos,
                                                float& a_sin, float clog) {
    const float u = unit_float(w_even) - 0x1.fffffep-1f;
    const float rho = sqrt_approx(lg2_approx(u) * clog);
    const float th = fmaf(unit_float(w_odd), 6.2831853071795865f, -9.4247779f);
    float s, c;
    __sincosf(th, &s, &c);
    a_cos = -rho * c;
    a_sin = -rho * s;
}

// clog = -2 ln(2) scale^2: the normals come out multiplied by scale (the
// default, kClogUnit, gives standard normals).  Every estimator kernel draws
// its noise through this form, so the perturbation of a draw and the noise
// its error estimate is weighted by are the same numbers.
constexpr float kClogUnit = -1.3862943611198906f;

// The four normals of a word quadruple by box_muller_fast, its two pairs side
// by side on packed fp32 pairs: the same operations in the same order as two
// box_muller_fast calls, so the same bits, in fewer instructions.
__device__ __forceinline__ float4 words_to_normals_fast(uint4 w, float clog = kClogUnit) {
    const float2 u = add2(make_float2(unit_float(w.x), unit_float(w.z)),
                          make_float2(-0x1.fffffep-1f, -0x1.fffffep-1f));
    const float2 x = mul2(make_float2(lg2_approx(u.x), lg2_approx(u.y)), make_float2(clog, clog));
    const float r0 = sqrt_approx(x.x), r1 = sqrt_approx(x.y);
    const float2 th = fma2(make_float2(unit_float(w.y), unit_float(w.w)),
                           make_float2(6.2831853071795865f, 6.2831853071795865f),
                           make_float2(-9.4247779f, -9.4247779f));
    float s0, c0, s1, c1;
    __sincosf(th.x, &s0, &c0);
    __sincosf(th.y, &s1, &c1);
    const float2 a01 = mul2(make_float2(-r0, -r0), make_float2(c0, s0));
    const float2 a23 = mul2(make_float2(-r1, -r1), make_float2(c1, s1));
    return make_float4(a01.x, a01.y, a23.x, a23.y);
}

}  // namespace dust
