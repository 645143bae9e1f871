// pairs.cuh -- arithmetic on packed fp32 pairs.  Blackwell issues add, sub,
// mul and fma on two fp32 lanes as one instruction (the f32x2 forms, sm_100
// and later); each lane is rounded exactly as the scalar operation (round to
// nearest even, no flush to zero), so a computation moved onto pairs gives
// the same bits as its scalar form with half the instructions.  The operands
// are float2 values; the asm packs them into 64-bit registers, which costs
// nothing when the two floats already sit in an aligned register pair.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dust {

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 pa, pb, pc, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
        " mov.b64 pc, {%6, %7};\n fma.rn.f32x2 pd, pa, pb, pc;\n mov.b64 {%0, %1}, pd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
        " mul.rn.f32x2 pd, pa, pb;\n mov.b64 {%0, %1}, pd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
        " add.rn.f32x2 pd, pa, pb;\n mov.b64 {%0, %1}, pd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 pa, pb, pd;\n mov.b64 pa, {%2, %3};\n mov.b64 pb, {%4, %5};\n"
        " sub.rn.f32x2 pd, pa, pb;\n mov.b64 {%0, %1}, pd;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// bf16 hi and lo parts of a pair: hi = bf16(v), lo = bf16(v - hi) per lane
// (v = hi + lo to about 2^-16 relative), each as a packed bf16x2 word (the
// first lane in the low half); the difference is one packed subtraction.
__device__ __forceinline__ void split_pair2(float2 v, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v.x, v.y);
    hi = *reinterpret_cast<uint32_t*>(&h2);
    const float2 h = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
    const float2 d = sub2(v, h);
    __nv_bfloat162 l2 = __floats2bfloat162_rn(d.x, d.y);
    lo = *reinterpret_cast<uint32_t*>(&l2);
}

}  // namespace dust
