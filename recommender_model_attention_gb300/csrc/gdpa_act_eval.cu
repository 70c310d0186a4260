// Element-wise evaluation of the activation device functions exactly as the
// kernels apply them (fast: the tensor-core kernels' flavour; precise: the
// CUDA-core float32 path's), so that they can be checked against reference
// values directly rather than through a whole attention product.
#include "act.cuh"
#include "gdpa_internal.h"

namespace gdpa {
namespace {

template <int ACT, bool FAST>
__global__ void act_eval_kernel(const float* x, float* y, float* dy, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n; k += stride) {
        float a, da;
        if constexpr (FAST) {
            // the tensor-core kernels' form (scale folded into the constants)
            const ActScale sc = act_scale<ACT>(1.0f);
            act_dact_s<ACT>(x[k], sc, a, da);
            y[k] = act_s<ACT>(x[k], sc);
        } else {
            act_dact_f<ACT, false>(x[k], a, da);
            y[k] = act_f<ACT, false>(x[k]);
        }
        dy[k] = da;
    }
}

template <bool FAST>
void launch_eval(int act, const float* x, float* y, float* dy, int64_t n, cudaStream_t st) {
    const int64_t blocks = (n + 255) / 256;
    const int grid = (int)(blocks < 4096 ? blocks : 4096);
    GDPA_DISPATCH_ACT(act, A, (act_eval_kernel<A, FAST><<<grid, 256, 0, st>>>(x, y, dy, n)))
}

}  // namespace
}  // namespace gdpa

extern "C" gdpa_status gdpa_act_eval(gdpa_act act, int fast, const float* x, float* y, float* dy,
                                     int64_t n, void* stream) {
    if (act < GDPA_ACT_GELU_ERF || act > GDPA_ACT_IDENTITY || n < 0) return GDPA_ERR_INVALID_ARG;
    // (the softmax variant is a row operation, not an element-wise one)
    if (n == 0) return GDPA_OK;
    if (!x || !y || !dy) return GDPA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (fast)
        gdpa::launch_eval<true>((int)act, x, y, dy, n, st);
    else
        gdpa::launch_eval<false>((int)act, x, y, dy, n, st);
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}
