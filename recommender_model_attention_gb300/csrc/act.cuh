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
//  * Fast (bf16 tensor-core path, whose P and dS are rounded to bf16, 2^-9
//    relative, anyway): one tanh.approx.f32 per element and a few FMAs.
//    GELU-tanh is its own definition; SiLU is x/2 (1 + tanh(x/2)); GELU-erf
//    takes the tanh form of the Gaussian CDF used by Hendrycks & Gimpel
//    ("Gaussian Error Linear Units", 2016), Phi(x) ~ (1 + tanh(x (g0 +
//    g1 x^2))) / 2, with g0, g1 refitted here to x Phi(x) itself: a minimax
//    fit on [-10, 10] of the value and, at half weight, its derivative gives
//    max |error| 3.4e-4 (value) and 6.7e-4 (derivative) in exact arithmetic;
//    the backward uses the exact derivative of this same approximation.
//    The Taylor polynomial is the same FMA chain in both flavours.
#pragma once

#include <cuda_runtime.h>

#include "f2.cuh"

namespace gdpa {

// kSoftmax is not element-wise: it selects the softmax variant (Jagged Flash
// Attention) of the forward kernels, whose rows are normalised.
enum : int { kGeluErf = 0, kGeluTanh = 1, kSilu = 2, kTaylor6 = 3, kIdentity = 4, kSoftmax = 5 };

constexpr float kRsqrt2 = 0.70710678118654752440f;     // 1/sqrt(2)
constexpr float kRsqrt2Pi = 0.39894228040143267794f;   // 1/sqrt(2 pi)
constexpr float kSqrt2OverPi = 0.79788456080286535588f;
constexpr float kTanhCubic = 0.044715f;
constexpr float kT6c2 = kRsqrt2Pi;
constexpr float kT6c4 = -kRsqrt2Pi / 6.0f;
constexpr float kT6c6 = kRsqrt2Pi / 40.0f;

// tanh-form Gaussian CDF for GELU-erf (see the header)
constexpr float kG0 = 0.7999136459f;
constexpr float kG1 = 0.0349731511f;
constexpr float kLog2e = 1.44269504088896340736f;

// 2^x (the softmax variant's weights)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
__device__ __forceinline__ void act_dact_f(float x, float& a, float& da);

template <int ACT, bool FAST>
__device__ __forceinline__ float act_f(float x) {
    if constexpr (ACT == kGeluErf) {
        if constexpr (FAST) {
            const float hx = 0.5f * x;
            return fmaf(hx, tanh_approx(x * fmaf(kG1, x * x, kG0)), hx);
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
        if constexpr (FAST) {
            float a, da;
            act_dact_f<ACT, true>(x, a, da);
            return da;
        } else {
            const float cdf = 0.5f * (1.0f + erff(x * kRsqrt2));
            return fmaf(x, kRsqrt2Pi * expf(-0.5f * x * x), cdf);
        }
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
            // d/dx [x/2 (1 + tanh(u))] = (1 + t)/2 + x/2 (1 - t^2) u',
            // u = x (g0 + g1 x^2), u' = g0 + 3 g1 x^2
            const float x2 = x * x;
            const float t = tanh_approx(x * fmaf(kG1, x2, kG0));
            const float hx = 0.5f * x;
            a = fmaf(hx, t, hx);
            da = fmaf(hx * fmaf(-t, t, 1.0f), fmaf(3.0f * kG1, x2, kG0), fmaf(0.5f, t, 0.5f));
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

// The tensor-core kernels' form: the scale folded into the constants.
// GELU-erf, GELU-tanh and SiLU are all x/2 (1 + tanh(u)) with u = x (g0 +
// g1 x^2) (SiLU: g0 = 1/2, g1 = 0); with x = alpha s the kernels evaluate
// them from the raw score s: x/2 = h s, u = s (c0 + c1 s^2), and
// u'(x) = d0 + d1 s^2, so the scaling costs nothing per element.
struct ActScale {
    float alpha, h, c0, c1, d0, d1;
};

template <int ACT>
__host__ __device__ constexpr bool tanh_form() {
    return ACT == kGeluErf || ACT == kGeluTanh || ACT == kSilu;
}

template <int ACT>
__device__ __forceinline__ ActScale act_scale(float alpha) {
    float g0 = 0.0f, g1 = 0.0f;
    if constexpr (ACT == kGeluErf) {
        g0 = kG0;
        g1 = kG1;
    } else if constexpr (ACT == kGeluTanh) {
        g0 = kSqrt2OverPi;
        g1 = kSqrt2OverPi * kTanhCubic;
    } else if constexpr (ACT == kSilu) {
        g0 = 0.5f;
    } else if constexpr (ACT == kSoftmax) {
        g0 = kLog2e;   // c0 = alpha log2(e): exponents in base 2
    }
    const float a2 = alpha * alpha;
    return ActScale{alpha, 0.5f * alpha, g0 * alpha, g1 * a2 * alpha, g0, 3.0f * g1 * a2};
}

// act(alpha s), fast flavour
template <int ACT>
__device__ __forceinline__ float act_s(float s, const ActScale& k) {
    if constexpr (ACT == kSilu) {   // g1 = 0
        const float hx = k.h * s;
        return fmaf(hx, tanh_approx(hx), hx);
    } else if constexpr (tanh_form<ACT>()) {
        const float t = tanh_approx(s * fmaf(k.c1, s * s, k.c0));
        const float hx = k.h * s;
        return fmaf(hx, t, hx);
    } else {
        return act_f<ACT, true>(k.alpha * s);
    }
}

// act(alpha s) and act'(alpha s), fast flavour
template <int ACT>
__device__ __forceinline__ void act_dact_s(float s, const ActScale& k, float& a, float& da) {
    if constexpr (ACT == kSilu) {   // u = x/2, u' = 1/2
        const float hx = k.h * s;
        const float t = tanh_approx(hx);
        a = fmaf(hx, t, hx);
        da = fmaf(hx * fmaf(-t, t, 1.0f), 0.5f, fmaf(0.5f, t, 0.5f));
    } else if constexpr (tanh_form<ACT>()) {
        // d/dx [x/2 (1 + tanh(u))] = (1 + t)/2 + x/2 (1 - t^2) u'
        const float s2 = s * s;
        const float t = tanh_approx(s * fmaf(k.c1, s2, k.c0));
        const float hx = k.h * s;
        a = fmaf(hx, t, hx);
        da = fmaf(hx * fmaf(-t, t, 1.0f), fmaf(k.d1, s2, k.d0), fmaf(0.5f, t, 0.5f));
    } else {
        act_dact_f<ACT, true>(k.alpha * s, a, da);
    }
}

// act_s of two scores at once: the same operations lane by lane in f32x2
// form (half the instructions; the same results, bit for bit).  The
// derivative's 1 - t^2 is formed as t^2 - 1 and the sign carried by -u'
// (both exact negations under round-to-nearest).
template <int ACT>
__device__ __forceinline__ void act_s2(float s0, float s1, const ActScale& k, float& a0, float& a1) {
    if constexpr (tanh_form<ACT>()) {
        const uint64_t s = f2_make(s0, s1);
        const uint64_t hx = f2_mul(f2_make(k.h, k.h), s);
        float2 u;
        if constexpr (ACT == kSilu) {
            u = f2_split(hx);
        } else {
            u = f2_split(f2_mul(s, f2_fma(f2_make(k.c1, k.c1), f2_mul(s, s), f2_make(k.c0, k.c0))));
        }
        const float2 a = f2_split(f2_fma(hx, f2_make(tanh_approx(u.x), tanh_approx(u.y)), hx));
        a0 = a.x;
        a1 = a.y;
    } else if constexpr (ACT == kTaylor6) {   // taylor6 of x = alpha s, lane by lane
        const uint64_t x = f2_mul(f2_make(k.alpha, k.alpha), f2_make(s0, s1));
        const uint64_t x2 = f2_mul(x, x);
        uint64_t t = f2_fma(f2_make(kT6c6, kT6c6), x2, f2_make(kT6c4, kT6c4));
        t = f2_fma(t, x2, f2_make(kT6c2, kT6c2));
        t = f2_fma(t, x, f2_make(0.5f, 0.5f));
        const float2 a = f2_split(f2_mul(t, x));
        a0 = a.x;
        a1 = a.y;
    } else {
        a0 = act_s<ACT>(s0, k);
        a1 = act_s<ACT>(s1, k);
    }
}

// act_dact_s of two scores at once (f32x2 form of the same operations).
template <int ACT>
__device__ __forceinline__ void act_dact_s2(float s0, float s1, const ActScale& k, float& a0,
                                            float& a1, float& da0, float& da1) {
    if constexpr (tanh_form<ACT>()) {
        const uint64_t s = f2_make(s0, s1);
        const uint64_t hx = f2_mul(f2_make(k.h, k.h), s);
        uint64_t nup;   // -u'(x)
        float2 u;
        if constexpr (ACT == kSilu) {
            u = f2_split(hx);
            nup = f2_make(-0.5f, -0.5f);
        } else {
            const uint64_t s2 = f2_mul(s, s);
            u = f2_split(f2_mul(s, f2_fma(f2_make(k.c1, k.c1), s2, f2_make(k.c0, k.c0))));
            nup = f2_fma(f2_make(-k.d1, -k.d1), s2, f2_make(-k.d0, -k.d0));
        }
        const uint64_t t = f2_make(tanh_approx(u.x), tanh_approx(u.y));
        const float2 a = f2_split(f2_fma(hx, t, hx));
        const uint64_t y = f2_mul(hx, f2_fma(t, t, f2_make(-1.0f, -1.0f)));   // -x/2 (1 - t^2)
        const uint64_t half_t = f2_fma(f2_make(0.5f, 0.5f), t, f2_make(0.5f, 0.5f));
        const float2 da = f2_split(f2_fma(y, nup, half_t));
        a0 = a.x;
        a1 = a.y;
        da0 = da.x;
        da1 = da.y;
    } else if constexpr (ACT == kTaylor6) {   // taylor6 and dtaylor6 of x = alpha s
        const uint64_t x = f2_mul(f2_make(k.alpha, k.alpha), f2_make(s0, s1));
        const uint64_t x2 = f2_mul(x, x);
        uint64_t t = f2_fma(f2_make(kT6c6, kT6c6), x2, f2_make(kT6c4, kT6c4));
        t = f2_fma(t, x2, f2_make(kT6c2, kT6c2));
        t = f2_fma(t, x, f2_make(0.5f, 0.5f));
        const float2 a = f2_split(f2_mul(t, x));
        constexpr float e6 = 6.0f * kT6c6, e4 = 4.0f * kT6c4, e2 = 2.0f * kT6c2;
        uint64_t g = f2_fma(f2_make(e6, e6), x2, f2_make(e4, e4));
        g = f2_fma(g, x2, f2_make(e2, e2));
        const float2 da = f2_split(f2_fma(g, x, f2_make(0.5f, 0.5f)));
        a0 = a.x;
        a1 = a.y;
        da0 = da.x;
        da1 = da.y;
    } else {
        act_dact_s<ACT>(s0, k, a0, da0);
        act_dact_s<ACT>(s1, k, a1, da1);
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
