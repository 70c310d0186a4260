// Element-wise GDPA activations and their derivatives, as device functions.
//
// The GDPA page (aitrends.kr, "범용 내적 어텐션(GDPA) ...") replaces the
// softmax by GELU, SiLU and similar functions, and replaces the tanh-based
// GELU by an ALU-only 6th-order Taylor polynomial to avoid the SFU (the SFU
// paragraph and its code figure):  x/2 + c2 x^2 + c4 x^4 + c6 x^6 with
// c2 = 1/sqrt(2 pi), c4 = -c2/6, c6 = c2/40.
//
// Two flavours:
//  * Precise (CUDA-core float32 path): CUDA's erff / tanhf / expf.
//  * Fast (bf16 tensor-core path, whose P is rounded to bf16 anyway), all
//    branch-free with at most one or two special-function ops per element:
//    GELU-tanh through the tanh.approx.f32 instruction; SiLU as
//    x/2 (1 + tanh(x/2)); GELU-erf with Phi from the rational approximation
//    of Abramowitz & Stegun, Handbook of Mathematical Functions, eq. 7.1.28
//    (erf z = 1 - (1 + a1 z + ... + a6 z^6)^-16, |error| <= 3e-7), one
//    reciprocal per element.  act and act' together (backward) use A&S eq.
//    7.1.26 instead (erfc z = t (a1 + ... + a5 t^4) exp(-z^2), t = 1/(1 + p z),
//    |error| <= 1.5e-7), whose exp(-z^2) = exp(-x^2/2) is also the normal
//    density's, so one reciprocal and one ex2 serve both.
//    The Taylor polynomial is the same FMA chain in both flavours.
#pragma once

#include <cuda_runtime.h>

namespace gdpa {

enum : int { kGeluErf = 0, kGeluTanh = 1, kSilu = 2, kTaylor6 = 3, kIdentity = 4 };

constexpr float kRsqrt2 = 0.70710678118654752440f;     // 1/sqrt(2)
constexpr float kRsqrt2Pi = 0.39894228040143267794f;   // 1/sqrt(2 pi)
constexpr float kSqrt2OverPi = 0.79788456080286535588f;
constexpr float kTanhCubic = 0.044715f;
constexpr float kT6c2 = kRsqrt2Pi;
constexpr float kT6c4 = -kRsqrt2Pi / 6.0f;
constexpr float kT6c6 = kRsqrt2Pi / 40.0f;

// Abramowitz & Stegun 7.1.28 coefficients
constexpr float kAS1 = 0.0705230784f;
constexpr float kAS2 = 0.0422820123f;
constexpr float kAS3 = 0.0092705272f;
constexpr float kAS4 = 0.0001520143f;
constexpr float kAS5 = 0.0002765672f;
constexpr float kAS6 = 0.0000430638f;
constexpr float kLog2e = 1.44269504088896340736f;

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Phi(x) = (1 + erf(x / sqrt 2)) / 2 with erf from A&S 7.1.28 (z >= 0; the
// polynomial's 16th power overflows to +inf for large z, giving erf = 1).
__device__ __forceinline__ float normal_cdf_fast(float x) {
    const float z = fabsf(x) * kRsqrt2;
    float p = fmaf(kAS6, z, kAS5);
    p = fmaf(p, z, kAS4);
    p = fmaf(p, z, kAS3);
    p = fmaf(p, z, kAS2);
    p = fmaf(p, z, kAS1);
    p = fmaf(p, z, 1.0f);
    p = p * p;
    p = p * p;
    p = p * p;
    p = p * p;                          // (1 + ...)^16
    const float half_tail = 0.5f * rcp_approx(p);   // (1 - erf z) / 2
    return x >= 0.0f ? 1.0f - half_tail : half_tail;
}

// A&S 7.1.26 coefficients
constexpr float kASp = 0.3275911f;
constexpr float kASb1 = 0.254829592f;
constexpr float kASb2 = -0.284496736f;
constexpr float kASb3 = 1.421413741f;
constexpr float kASb4 = -1.453152027f;
constexpr float kASb5 = 1.061405429f;

// x Phi(x) and Phi(x) + x phi(x) with one reciprocal and one ex2
__device__ __forceinline__ void gelu_erf_and_grad_fast(float x, float& a, float& da) {
    const float z = fabsf(x) * kRsqrt2;
    const float t = rcp_approx(fmaf(kASp, z, 1.0f));
    float q = fmaf(kASb5, t, kASb4);
    q = fmaf(q, t, kASb3);
    q = fmaf(q, t, kASb2);
    q = fmaf(q, t, kASb1);
    const float e = ex2_approx(-0.5f * kLog2e * x * x);   // exp(-x^2 / 2)
    const float half_tail = 0.5f * q * t * e;             // erfc(z) / 2
    const float cdf = x >= 0.0f ? 1.0f - half_tail : half_tail;
    a = x * cdf;
    da = fmaf(x * kRsqrt2Pi, e, cdf);
}

__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x * (1/2 + x (c2 + x^2 (c4 + c6 x^2)))  ==  x/2 + c2 x^2 + c4 x^4 + c6 x^6
__device__ __forceinline__ float taylor6(float x) {
    const float x2 = x * x;
    float t = fmaf(kT6c6, x2, kT6c4);
    t = fmaf(t, x2, kT6c2);
    t = fmaf(t, x, 0.5f);
    return t * x;
}

// 1/2 + 2 c2 x + 4 c4 x^3 + 6 c6 x^5
__device__ __forceinline__ float dtaylor6(float x) {
    const float x2 = x * x;
    float t = fmaf(6.0f * kT6c6, x2, 4.0f * kT6c4);
    t = fmaf(t, x2, 2.0f * kT6c2);
    return fmaf(t, x, 0.5f);
}

template <int ACT, bool FAST>
__device__ __forceinline__ float act_f(float x) {
    if constexpr (ACT == kGeluErf) {
        if constexpr (FAST) {
            return x * normal_cdf_fast(x);
        } else {
            return 0.5f * x * (1.0f + erff(x * kRsqrt2));
        }
    } else if constexpr (ACT == kGeluTanh) {
        const float u = kSqrt2OverPi * fmaf(kTanhCubic * x, x * x, x);
        const float t = FAST ? tanh_approx(u) : tanhf(u);
        return 0.5f * x * (1.0f + t);
    } else if constexpr (ACT == kSilu) {
        if constexpr (FAST) {
            const float hx = 0.5f * x;
            return fmaf(hx, tanh_approx(hx), hx);
        } else {
            return x / (1.0f + expf(-x));
        }
    } else if constexpr (ACT == kTaylor6) {
        return taylor6(x);
    } else {
        return x;
    }
}

template <int ACT, bool FAST>
__device__ __forceinline__ float dact_f(float x) {
    if constexpr (ACT == kGeluErf) {
        const float cdf = FAST ? normal_cdf_fast(x) : 0.5f * (1.0f + erff(x * kRsqrt2));
        const float pdf = kRsqrt2Pi * (FAST ? ex2_approx(-0.5f * kLog2e * x * x)
                                           : expf(-0.5f * x * x));
        return fmaf(x, pdf, cdf);
    } else if constexpr (ACT == kGeluTanh) {
        const float u = kSqrt2OverPi * fmaf(kTanhCubic * x, x * x, x);
        const float t = FAST ? tanh_approx(u) : tanhf(u);
        const float du = kSqrt2OverPi * fmaf(3.0f * kTanhCubic, x * x, 1.0f);
        return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * du;
    } else if constexpr (ACT == kSilu) {
        const float s = FAST ? fmaf(0.5f, tanh_approx(0.5f * x), 0.5f) : 1.0f / (1.0f + expf(-x));
        return s * fmaf(x, 1.0f - s, 1.0f);
    } else if constexpr (ACT == kTaylor6) {
        return dtaylor6(x);
    } else {
        return 1.0f;
    }
}

// act and act' together (backward recompute).
template <int ACT, bool FAST>
__device__ __forceinline__ void act_dact_f(float x, float& a, float& da) {
    if constexpr (ACT == kGeluErf) {
        if constexpr (FAST) {
            gelu_erf_and_grad_fast(x, a, da);
        } else {
            const float cdf = 0.5f * (1.0f + erff(x * kRsqrt2));
            a = x * cdf;
            da = fmaf(x, kRsqrt2Pi * expf(-0.5f * x * x), cdf);
        }
    } else if constexpr (ACT == kGeluTanh) {
        const float u = kSqrt2OverPi * fmaf(kTanhCubic * x, x * x, x);
        const float t = FAST ? tanh_approx(u) : tanhf(u);
        const float du = kSqrt2OverPi * fmaf(3.0f * kTanhCubic, x * x, 1.0f);
        a = 0.5f * x * (1.0f + t);
        da = 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * du;
    } else if constexpr (ACT == kSilu) {
        const float s = FAST ? fmaf(0.5f, tanh_approx(0.5f * x), 0.5f) : 1.0f / (1.0f + expf(-x));
        a = x * s;
        da = s * fmaf(x, 1.0f - s, 1.0f);
    } else if constexpr (ACT == kTaylor6) {
        a = taylor6(x);
        da = dtaylor6(x);
    } else {
        a = x;
        da = 1.0f;
    }
}

// Runtime activation id -> template instantiation.
#define GDPA_DISPATCH_ACT(act, ACTC, ...)                      \
    switch (act) {                                             \
    case kGeluErf: { constexpr int ACTC = kGeluErf; __VA_ARGS__; } break;   \
    case kGeluTanh: { constexpr int ACTC = kGeluTanh; __VA_ARGS__; } break; \
    case kSilu: { constexpr int ACTC = kSilu; __VA_ARGS__; } break;         \
    case kTaylor6: { constexpr int ACTC = kTaylor6; __VA_ARGS__; } break;   \
    default: { constexpr int ACTC = kIdentity; __VA_ARGS__; } break;        \
    }

}  // namespace gdpa
