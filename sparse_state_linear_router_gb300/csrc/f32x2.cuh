// f32x2.cuh -- Blackwell's packed float32 pair arithmetic (add / mul /
// fma.rn.f32x2): two float32 lanes in one 64-bit register, each lane the
// scalar IEEE operation rounded to nearest, so a result equals two scalar
// instructions' results, issued as one.
#pragma once

#include <stdint.h>

namespace sse {

#ifndef SSE_F32X2
#define SSE_F32X2 1
#endif
struct F2 { uint64_t v; };
__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ F2 f2_bits(uint32_t lo, uint32_t hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_get(F2 x) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x.v));
    return r;
}
__device__ __forceinline__ F2 add2(F2 a, F2 b) {
#if SSE_F32X2
    F2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
#else
    const float2 x = f2_get(a), y = f2_get(b);
    return f2(x.x + y.x, x.y + y.y);
#endif
}
__device__ __forceinline__ F2 mul2(F2 a, F2 b) {
#if SSE_F32X2
    F2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
    return r;
#else
    const float2 x = f2_get(a), y = f2_get(b);
    return f2(x.x * y.x, x.y * y.y);
#endif
}
__device__ __forceinline__ F2 fma2(F2 a, F2 b, F2 c) {
#if SSE_F32X2
    F2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
    return r;
#else
    const float2 x = f2_get(a), y = f2_get(b), z = f2_get(c);
    return f2(fmaf(x.x, y.x, z.x), fmaf(x.y, y.y, z.y));
#endif
}

}  // namespace sse
