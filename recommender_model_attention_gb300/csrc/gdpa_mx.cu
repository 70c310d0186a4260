// MXFP8 (OCP Microscaling, E4M3 elements with one E8M0 power-of-two scale
// per 32 consecutive values) encoding of Q and K for GDPA.
//
// The GEM page ("GEM 트레이닝: Meta가 LLM 규모의 광고 파운데이션 모델 효율성을
// 두 배로 높인 방법", techlist.io, section "GPU 연산 효율을 높인 맞춤형 커널과
// 정밀도") trains attention in mixed precision that includes MXFP8.  Blocks
// run along the head dimension d (the contraction of S = Q K^T).  For a block
// with largest magnitude a > 0 the scale exponent is E = floor(log2 a) - 8 (8
// being the exponent of E4M3's largest normal), clamped to [-127, 127]; an
// all-zero block takes E = -127.  Elements are x / 2^E rounded to the nearest
// E4M3 value (ties to the even mantissa) and saturated at +-448.  Stored:
// element codes as bytes, scales as E + 127 (the E8M0 byte).
//
// Each dequantised value m 2^(e + E) has at most four significant bits, so
// it is a bf16 number whenever its exponent is in bf16's range: expanding a
// tile to bf16 and running the bf16 kernels computes GDPA of exactly the
// values the MXFP8 tensor stands for.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gdpa_internal.h"

namespace gdpa {
namespace {

constexpr int kBlock = 32;

// 2^e as a float for e in [-127, 127] (2^-127 is a subnormal), exactly
__device__ __forceinline__ float exp2i(int e) {
    return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(0x00400000);
}

// two floats -> two E4M3 codes (round to nearest even, saturate at 448)
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// two E4M3 codes -> two floats (exact: every E4M3 value is an f16 value)
__device__ __forceinline__ float2 from_e4m3x2(uint16_t v) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
    __half2 p;
    *reinterpret_cast<uint32_t*>(&p) = h;
    return __half22float2(p);
}

// one thread per block of 32 values: 64 bytes in, 32 element bytes and one
// scale byte out
__global__ void __launch_bounds__(256)
mx_quantise_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ el,
                   uint8_t* __restrict__ sc, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (b >= nblocks) return;
    const uint4* src = reinterpret_cast<const uint4*>(x + b * kBlock);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(src + i);
        w[4 * i] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    float f[kBlock];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
    }
    int e = -127;
    if (amax > 0.0f) {
        int fe;
        frexpf(amax, &fe);           // amax = m 2^fe, m in [0.5, 1): floor(log2) = fe - 1
        e = fe - 1 - 8;
        e = e < -127 ? -127 : (e > 127 ? 127 : e);
    }
    const float inv = exp2i(-e);     // x / 2^E, exact (or below E4M3's range)
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint16_t a = to_e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv);
        const uint16_t c = to_e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv);
        out[i] = (uint32_t)a | ((uint32_t)c << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(el + b * kBlock);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    sc[b] = (uint8_t)(e + 127);
}

// one thread per block: 32 element bytes and the scale in, 64 bytes of bf16 out
__global__ void __launch_bounds__(256)
mx_dequantise_kernel(const uint8_t* __restrict__ el, const uint8_t* __restrict__ sc,
                     __nv_bfloat16* __restrict__ x, int64_t nblocks) {
    const int64_t b = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (b >= nblocks) return;
    const float s = exp2i((int)__ldg(sc + b) - 127);
    const uint4* src = reinterpret_cast<const uint4*>(el + b * kBlock);
    uint32_t out[16];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint4 v = __ldg(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 a = from_e4m3x2((uint16_t)(w[j] & 0xffffu));
            const float2 c = from_e4m3x2((uint16_t)(w[j] >> 16));
            const __nv_bfloat162 pa = __floats2bfloat162_rn(a.x * s, a.y * s);
            const __nv_bfloat162 pc = __floats2bfloat162_rn(c.x * s, c.y * s);
            out[8 * i + 2 * j] = *reinterpret_cast<const uint32_t*>(&pa);
            out[8 * i + 2 * j + 1] = *reinterpret_cast<const uint32_t*>(&pc);
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(x + b * kBlock);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
}

unsigned grid_for(int64_t n) { return (unsigned)((n + 255) / 256); }

}  // namespace

gdpa_status launch_mx_quantise(const void* x, int64_t n_values, uint8_t* el, uint8_t* sc,
                               cudaStream_t st) {
    const int64_t nb = n_values / kBlock;
    if (nb == 0) return GDPA_OK;
    mx_quantise_kernel<<<grid_for(nb), 256, 0, st>>>((const __nv_bfloat16*)x, el, sc, nb);
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

gdpa_status launch_mx_dequantise(const uint8_t* el, const uint8_t* sc, int64_t n_values, void* x,
                                 cudaStream_t st) {
    const int64_t nb = n_values / kBlock;
    if (nb == 0) return GDPA_OK;
    mx_dequantise_kernel<<<grid_for(nb), 256, 0, st>>>(el, sc, (__nv_bfloat16*)x, nb);
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

}  // namespace gdpa
