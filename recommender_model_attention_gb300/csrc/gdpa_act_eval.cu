// Element-wise evaluation of the activation device functions exactly as the
// kernels apply them (fast: the tensor-core kernels' flavour; precise: the
// CUDA-core float32 path's), so that they can be checked against reference
// values directly rather than through a whole attention product.
#include "act.cuh"
#include "gdpa_internal.h"

namespace gdpa {
namespace {

// MODE 0: the float32 CUDA-core flavour; 1: the tensor-core flavour one
// element at a time; 2: the same in the f32x2 pair form (elements 2k, 2k + 1)
template <int ACT, int MODE>
__global__ void act_eval_kernel(const float* x, float* y, float* dy, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const ActScale sc = act_scale<ACT>(1.0f);   // the scale folded into the constants
    if constexpr (MODE == 2) {
        for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; 2 * k < n; k += stride) {
            const int64_t i0 = 2 * k, i1 = i0 + 1 < n ? i0 + 1 : i0;
            float a0, a1, da0, da1, b0, b1;
            act_dact_s2<ACT>(x[i0], x[i1], sc, a0, a1, da0, da1);
            act_s2<ACT>(x[i0], x[i1], sc, b0, b1);
            // the value from the value-and-derivative form (the backward's
            // P) must have the bits of the value-only form (the forward's):
            // a NaN in y flags a difference
            const bool same0 = __float_as_uint(a0) == __float_as_uint(b0);
            const bool same1 = __float_as_uint(a1) == __float_as_uint(b1);
            y[i0] = same0 ? b0 : __uint_as_float(0x7fc00000u);
            dy[i0] = da0;
            if (i1 != i0) {
                y[i1] = same1 ? b1 : __uint_as_float(0x7fc00000u);
                dy[i1] = da1;
            }
        }
    } else {
        for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n; k += stride) {
            float a, da;
            if constexpr (MODE == 1) {
                act_dact_s<ACT>(x[k], sc, a, da);
                y[k] = act_s<ACT>(x[k], sc);
            } else {
                act_dact_f<ACT, false>(x[k], a, da);
                y[k] = act_f<ACT, false>(x[k]);
            }
            dy[k] = da;
        }
    }
}

template <int MODE>
void launch_eval(int act, const float* x, float* y, float* dy, int64_t n, cudaStream_t st) {
    const int64_t blocks = (n + 255) / 256;
    const int grid = (int)(blocks < 4096 ? blocks : 4096);
    GDPA_DISPATCH_ACT(act, A, (act_eval_kernel<A, MODE><<<grid, 256, 0, st>>>(x, y, dy, n)))
}

}  // namespace
}  // namespace gdpa

extern "C" gdpa_status gdpa_act_eval(gdpa_act act, int fast, const float* x, float* y, float* dy,
                                     int64_t n, void* stream) {
    if (act < GDPA_ACT_GELU_ERF || act > GDPA_ACT_IDENTITY || n < 0 || fast < 0 || fast > 2)
        return GDPA_ERR_INVALID_ARG;
    // (the softmax variant is a row operation, not an element-wise one)
    if (n == 0) return GDPA_OK;
    if (!x || !y || !dy) return GDPA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (fast == 2)
        gdpa::launch_eval<2>((int)act, x, y, dy, n, st);
    else if (fast == 1)
        gdpa::launch_eval<1>((int)act, x, y, dy, n, st);
    else
        gdpa::launch_eval<0>((int)act, x, y, dy, n, st);
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}
