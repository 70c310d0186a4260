// Packed pairs of floats for the f32x2 arithmetic of sm_100 and later: one
// instruction computes two results, each rounded exactly as the scalar
// operation would round it.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdpa {

// Two floats in one 64-bit register for the f32x2 arithmetic of sm_100 and
// later (two results per instruction).
__device__ __forceinline__ uint64_t f2_make(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_split(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// the two bf16 values of a packed word (low half first) as a float pair
__device__ __forceinline__ uint64_t f2_bf16x2(uint32_t w) {
    return f2_make(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

}  // namespace gdpa
