// CUDA-core (SIMT) GDPA kernels: float32 arithmetic for float32 and bf16
// inputs, walking the host plan.  They are the float32 path of the library
// (tensor-core tf32 would round the products to a 10-bit mantissa) and the
// path for head dims the tensor-core kernels do not take.
//
// One CTA of four warps per tile; one warp per row; lane c holds elements
// c, c + 32, c + 64, c + 96 of the row (d <= 128).  Scores are warp
// reductions.  The key loop of a row is limited to its valid keys, so no
// masking is needed inside it.  Key-split plans add each tile's partial O
// into a float32 workspace (rounded into O afterwards) and their dQ rows
// with atomic adds; in shared-query mode a row's Q (and dQ) is the seed at
// its position in the sample.
#include <cuda_bf16.h>

#include <algorithm>

#include "act.cuh"
#include "gdpa_internal.h"

namespace gdpa {
namespace {

constexpr int kWarps = 4;
constexpr int kPer = 4;  // elements per lane (d <= 128)

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename T>
__device__ __forceinline__ void load_row(float (&x)[kPer], const T* p, int d, int lane) {
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
        const int e = lane + 32 * c;
        x[c] = e < d ? ldf(p + e) : 0.0f;
    }
}

__device__ __forceinline__ float dot_row(const float (&a)[kPer], const float (&b)[kPer]) {
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kPer; ++c) s = fmaf(a[c], b[c], s);
    return warp_sum(s);
}

// valid keys of query position i: [lo, hi)
__device__ __forceinline__ void key_range(int i, int kb0, int kb1, int lkv, int mask, int window,
                                          int& lo, int& hi) {
    lo = kb0 * kBN;
    hi = min(kb1 * kBN, lkv);
    if (mask == GDPA_MASK_CAUSAL_WINDOW) {
        lo = max(lo, i - window + 1);
        hi = min(hi, i + 1);
    }
}

template <int ACT, typename T>
__global__ void __launch_bounds__(kWarps * 32)
simt_fwd_kernel(const FwdTile* __restrict__ tiles, const T* __restrict__ Q, const T* __restrict__ K,
                const T* __restrict__ V, T* __restrict__ O, float* __restrict__ W, int H, int d,
                float alpha, int mask, int window, int shared_q) {
    const FwdTile t = tiles[blockIdx.x];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)H * d;
    for (int r = warp; r < t.nq; r += kWarps) {
        const int64_t qrow = (int64_t)(t.qt0 + r) * row + (int64_t)t.h * d;
        const int64_t qin = (int64_t)((shared_q ? t.i0 : t.qt0) + r) * row + (int64_t)t.h * d;
        float q[kPer], o[kPer] = {0.f, 0.f, 0.f, 0.f};
        load_row(q, Q + qin, d, lane);
        int lo, hi;
        key_range(t.i0 + r, t.kb0, t.kb1, t.lkv, mask, window, lo, hi);
        for (int j = lo; j < hi; ++j) {
            const int64_t krow = (int64_t)(t.kvt0 + j) * row + (int64_t)t.h * d;
            float kx[kPer], vx[kPer];
            load_row(kx, K + krow, d, lane);
            load_row(vx, V + krow, d, lane);
            const float p = act_f<ACT, false>(alpha * dot_row(q, kx));
#pragma unroll
            for (int c = 0; c < kPer; ++c) o[c] = fmaf(p, vx[c], o[c]);
        }
#pragma unroll
        for (int c = 0; c < kPer; ++c) {
            const int e = lane + 32 * c;
            if (e < d) {
                if (W)
                    atomicAdd(W + qrow + e, o[c]);   // one key chunk of a split plan
                else
                    stf(O + qrow + e, o[c]);
            }
        }
    }
}

// Softmax variant (Jagged Flash Attention): O_i = sum_j w_j V_j over the
// valid keys of row i, w = softmax_j(alpha q_i.k_j), one pass with a running
// maximum m and sum l (O rescaled by exp(m_old - m_new) when m grows); a row
// without a valid key gets zero.
template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
simt_softmax_fwd_kernel(const FwdTile* __restrict__ tiles, const T* __restrict__ Q,
                        const T* __restrict__ K, const T* __restrict__ V, T* __restrict__ O,
                        float* __restrict__ lse, int H, int d, float alpha, int mask, int window,
                        int shared_q) {
    const FwdTile t = tiles[blockIdx.x];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)H * d;
    for (int r = warp; r < t.nq; r += kWarps) {
        const int64_t qrow = (int64_t)(t.qt0 + r) * row + (int64_t)t.h * d;
        const int64_t qin = (int64_t)((shared_q ? t.i0 : t.qt0) + r) * row + (int64_t)t.h * d;
        float q[kPer], o[kPer] = {0.f, 0.f, 0.f, 0.f};
        load_row(q, Q + qin, d, lane);
        int lo, hi;
        key_range(t.i0 + r, t.kb0, t.kb1, t.lkv, mask, window, lo, hi);
        float m = -INFINITY, l = 0.0f;
        for (int j = lo; j < hi; ++j) {
            const int64_t krow = (int64_t)(t.kvt0 + j) * row + (int64_t)t.h * d;
            float kx[kPer], vx[kPer];
            load_row(kx, K + krow, d, lane);
            load_row(vx, V + krow, d, lane);
            const float x = alpha * dot_row(q, kx);
            const float mn = fmaxf(m, x);
            const float scale = expf(m - mn);   // 0 on the first key (m = -inf)
            const float w = expf(x - mn);
            l = fmaf(l, scale, w);
#pragma unroll
            for (int c = 0; c < kPer; ++c) o[c] = fmaf(w, vx[c], o[c] * scale);
            m = mn;
        }
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
        for (int c = 0; c < kPer; ++c) {
            const int e = lane + 32 * c;
            if (e < d) stf(O + qrow + e, o[c] * inv);
        }
        if (lse && lane == 0) lse[(int64_t)(t.qt0 + r) * H + t.h] = l > 0.0f ? m + logf(l) : -INFINITY;
    }
}

// dQ_i = alpha sum_j (dO_i . V_j) act'(x_ij) K_j over the tile's rows
template <int ACT, typename T>
__global__ void __launch_bounds__(kWarps * 32)
simt_bwd_dq_kernel(const FwdTile* __restrict__ tiles, const T* __restrict__ Q,
                   const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO,
                   float* __restrict__ dQ, int H, int d, float alpha, int mask, int window,
                   const float* __restrict__ lse, const float* __restrict__ delta, int shared_q,
                   int accumulate) {
    const FwdTile t = tiles[blockIdx.x];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)H * d;
    for (int r = warp; r < t.nq; r += kWarps) {
        const int64_t qrow = (int64_t)(t.qt0 + r) * row + (int64_t)t.h * d;
        const int64_t qin = (int64_t)((shared_q ? t.i0 : t.qt0) + r) * row + (int64_t)t.h * d;
        float q[kPer], go[kPer], acc[kPer] = {0.f, 0.f, 0.f, 0.f};
        load_row(q, Q + qin, d, lane);
        load_row(go, dO + qrow, d, lane);
        int lo, hi;
        key_range(t.i0 + r, t.kb0, t.kb1, t.lkv, mask, window, lo, hi);
        float lse_i = 0.0f, d_i = 0.0f;   // softmax variant: the row's lse and dO.O
        if constexpr (ACT == kSoftmax) {
            lse_i = lse[(int64_t)(t.qt0 + r) * H + t.h];
            d_i = delta[(int64_t)(t.qt0 + r) * H + t.h];
        }
        for (int j = lo; j < hi; ++j) {
            const int64_t krow = (int64_t)(t.kvt0 + j) * row + (int64_t)t.h * d;
            float kx[kPer], vx[kPer];
            load_row(kx, K + krow, d, lane);
            load_row(vx, V + krow, d, lane);
            const float x = alpha * dot_row(q, kx);
            float g;
            if constexpr (ACT == kSoftmax)
                g = expf(x - lse_i) * (dot_row(go, vx) - d_i);
            else
                g = dot_row(go, vx) * dact_f<ACT, false>(x);
#pragma unroll
            for (int c = 0; c < kPer; ++c) acc[c] = fmaf(g, kx[c], acc[c]);
        }
#pragma unroll
        for (int c = 0; c < kPer; ++c) {
            const int e = lane + 32 * c;
            if (e < d) {
                if (accumulate)   // several key chunks or samples add into this row
                    atomicAdd(dQ + qin + e, alpha * acc[c]);
                else
                    dQ[qin + e] = alpha * acc[c];
            }
        }
    }
}

// dK_j = alpha sum_i g_ij Q_i and dV_j = sum_i act(x_ij) dO_i over the unit's keys
template <int ACT, typename T>
__global__ void __launch_bounds__(kWarps * 32)
simt_bwd_dkdv_kernel(const BwdUnit* __restrict__ units, const T* __restrict__ Q,
                     const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO,
                     float* __restrict__ dK, float* __restrict__ dV, int H, int d, float alpha,
                     int mask, int window, const float* __restrict__ lse,
                     const float* __restrict__ delta, int shared_q) {
    const BwdUnit u = units[blockIdx.x];
    const int h = u.hf & 0xffff;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)H * d;
    for (int c0 = warp; c0 < u.nkv; c0 += kWarps) {
        const int j = u.c0 + c0;
        const int64_t krow = (int64_t)(u.kvt0 + c0) * row + (int64_t)h * d;
        float kx[kPer], vx[kPer], ak[kPer] = {0.f, 0.f, 0.f, 0.f}, av[kPer] = {0.f, 0.f, 0.f, 0.f};
        load_row(kx, K + krow, d, lane);
        load_row(vx, V + krow, d, lane);
        int lo = u.m0 * kBM, hi = min(u.m1 * kBM, u.lq);
        if (mask == GDPA_MASK_CAUSAL_WINDOW) {
            lo = max(lo, j);
            hi = min(hi, j + window);
        }
        for (int i = lo; i < hi; ++i) {
            const int64_t qrow = (int64_t)(u.qt0 + i) * row + (int64_t)h * d;
            const int64_t qin = (int64_t)(shared_q ? i : u.qt0 + i) * row + (int64_t)h * d;
            float q[kPer], go[kPer];
            load_row(q, Q + qin, d, lane);
            load_row(go, dO + qrow, d, lane);
            const float x = alpha * dot_row(q, kx);
            float a, g;
            if constexpr (ACT == kSoftmax) {
                const int64_t ri = (int64_t)(u.qt0 + i) * H + h;
                a = expf(x - lse[ri]);
                g = a * (dot_row(go, vx) - delta[ri]);
            } else {
                float da;
                act_dact_f<ACT, false>(x, a, da);
                g = dot_row(go, vx) * da;
            }
#pragma unroll
            for (int c = 0; c < kPer; ++c) {
                ak[c] = fmaf(g, q[c], ak[c]);
                av[c] = fmaf(a, go[c], av[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < kPer; ++c) {
            const int e = lane + 32 * c;
            if (e < d) {
                dK[krow + e] = alpha * ak[c];
                dV[krow + e] = av[c];
            }
        }
    }
}

// key-split plans: O = W rounded to the output type
template <typename T>
__global__ void __launch_bounds__(256) split_round_kernel(const float* __restrict__ w,
                                                          T* __restrict__ o, int64_t n) {
    for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256)
        stf(o + i, w[i]);
}

template <typename T>
gdpa_status fwd_impl(Plan& p, const void* q, const void* k, const void* v, void* o, float* lse,
                     float alpha, int act, cudaStream_t st) {
    const unsigned grid = (unsigned)p.n_fwd;
    const int sq = p.shared_q > 0;
    if (act == kSoftmax) {
        if (p.fwd_split) return GDPA_ERR_UNSUPPORTED;   // chunks would need a max/sum merge
        simt_softmax_fwd_kernel<T><<<grid, kWarps * 32, 0, st>>>(
            p.d_fwd, (const T*)q, (const T*)k, (const T*)v, (T*)o, lse, p.H, p.d, alpha, p.mask,
            p.window, sq);
        p.launches += 1;
        return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
    }
    float* w = nullptr;
    const int64_t n = p.Tq * p.H * p.d;
    if (p.fwd_split) {
        const size_t bytes = (size_t)n * sizeof(float);
        if (!p.d_wsplit && cudaMallocAsync((void**)&p.d_wsplit, bytes, st) != cudaSuccess) {
            p.d_wsplit = nullptr;
            return GDPA_ERR_ALLOC;
        }
        if (cudaMemsetAsync(p.d_wsplit, 0, bytes, st) != cudaSuccess) return GDPA_ERR_CUDA;
        w = p.d_wsplit;
    }
    GDPA_DISPATCH_ACT(act, A,
        simt_fwd_kernel<A, T><<<grid, kWarps * 32, 0, st>>>(
            p.d_fwd, (const T*)q, (const T*)k, (const T*)v, (T*)o, w, p.H, p.d, alpha, p.mask,
            p.window, sq))
    p.launches += 1;
    if (w && n > 0) {
        const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 8);
        split_round_kernel<T><<<blocks, 256, 0, st>>>(w, (T*)o, n);
        p.launches += 1;
    }
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

template <typename T>
gdpa_status bwd_impl(Plan& p, const void* q, const void* k, const void* v, const void* d_o,
                     float* dq, float* dk, float* dv, float alpha, int act, const float* lse,
                     const float* delta, cudaStream_t st) {
    // dQ rows receive adds from several tiles (key-split plans) or samples
    // (shared queries): clear first
    const int sq = p.shared_q > 0;
    const int acc = sq || p.fwd_split;
    const int64_t dq_rows = sq ? p.shared_q : p.Tq;
    if (acc && dq_rows > 0 &&
        cudaMemsetAsync(dq, 0, (size_t)dq_rows * p.H * p.d * sizeof(float), st) != cudaSuccess)
        return GDPA_ERR_CUDA;
    if (act == kSoftmax) {
        if (p.n_fwd > 0) {
            simt_bwd_dq_kernel<kSoftmax, T><<<(unsigned)p.n_fwd, kWarps * 32, 0, st>>>(
                p.d_fwd, (const T*)q, (const T*)k, (const T*)v, (const T*)d_o, dq, p.H, p.d,
                alpha, p.mask, p.window, lse, delta, sq, acc);
            p.launches += 1;
        }
        if (p.n_bwd > 0) {
            simt_bwd_dkdv_kernel<kSoftmax, T><<<(unsigned)p.n_bwd, kWarps * 32, 0, st>>>(
                p.d_bwd, (const T*)q, (const T*)k, (const T*)v, (const T*)d_o, dk, dv, p.H, p.d,
                alpha, p.mask, p.window, lse, delta, sq);
            p.launches += 1;
        }
        return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
    }
    // Otherwise the forward tiles (zero tiles included) cover every query row
    // once and the backward units every key row once, so both kernels store
    // their rows directly.
    if (p.n_fwd > 0) {
        GDPA_DISPATCH_ACT(act, A,
            simt_bwd_dq_kernel<A, T><<<(unsigned)p.n_fwd, kWarps * 32, 0, st>>>(
                p.d_fwd, (const T*)q, (const T*)k, (const T*)v, (const T*)d_o, dq, p.H, p.d,
                alpha, p.mask, p.window, nullptr, nullptr, sq, acc))
        p.launches += 1;
    }
    if (p.n_bwd > 0) {
        GDPA_DISPATCH_ACT(act, A,
            simt_bwd_dkdv_kernel<A, T><<<(unsigned)p.n_bwd, kWarps * 32, 0, st>>>(
                p.d_bwd, (const T*)q, (const T*)k, (const T*)v, (const T*)d_o, dk, dv, p.H, p.d,
                alpha, p.mask, p.window, nullptr, nullptr, sq))
        p.launches += 1;
    }
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

}  // namespace

gdpa_status launch_simt_fwd(Plan& p, gdpa_dtype dt, const void* q, const void* k, const void* v,
                            void* o, float* lse, float alpha, int act, cudaStream_t st) {
    if (dt == GDPA_F32) return fwd_impl<float>(p, q, k, v, o, lse, alpha, act, st);
    return fwd_impl<__nv_bfloat16>(p, q, k, v, o, lse, alpha, act, st);
}

gdpa_status launch_simt_bwd(Plan& p, gdpa_dtype dt, const void* q, const void* k, const void* v,
                            const void* d_o, float* dq, float* dk, float* dv, float alpha, int act,
                            const float* lse, const float* delta, cudaStream_t st) {
    if (dt == GDPA_F32)
        return bwd_impl<float>(p, q, k, v, d_o, dq, dk, dv, alpha, act, lse, delta, st);
    return bwd_impl<__nv_bfloat16>(p, q, k, v, d_o, dq, dk, dv, alpha, act, lse, delta, st);
}

namespace {

// one warp per (token, head) row
template <typename T>
__global__ void __launch_bounds__(256)
row_dot_kernel(const T* __restrict__ a, const T* __restrict__ b, float* __restrict__ out,
               int64_t rows, int d) {
    const int64_t rw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (rw >= rows) return;
    float x[kPer], y[kPer];
    load_row(x, a + rw * d, d, lane);
    load_row(y, b + rw * d, d, lane);
    const float s = dot_row(x, y);
    if (lane == 0) out[rw] = s;
}

}  // namespace

gdpa_status launch_row_dot(Plan& p, gdpa_dtype dt, const void* d_o, const void* o, float* delta,
                           cudaStream_t st) {
    const int64_t rows = p.Tq * p.H;
    if (rows == 0) return GDPA_OK;
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (dt == GDPA_F32)
        row_dot_kernel<float><<<grid, 256, 0, st>>>((const float*)d_o, (const float*)o, delta, rows,
                                                    p.d);
    else
        row_dot_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            (const __nv_bfloat16*)d_o, (const __nv_bfloat16*)o, delta, rows, p.d);
    p.launches += 1;
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

namespace {

// Fused RMSNorm of the keys, one warp per (token, head) row of a bf16
// [rows][H][d] tensor: c = gain / sqrt(mean(k^2) + eps) into
// scale[h][t] (leading dimension ld) and the normalised row c k, rounded to
// bf16, into khat.  V = d / 32 values per lane (d = 64 or 128).
template <int V>
__global__ void __launch_bounds__(256)
key_norm_kernel(const __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ khat,
                float* __restrict__ scale, int64_t rows, int H, int64_t ld, float gain, float eps) {
    const int64_t rw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (rw >= rows * H) return;
    constexpr int d = 32 * V;
    const __nv_bfloat16* src = k + rw * d + lane * V;
    float x[V];
    if constexpr (V == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        x[0] = __uint_as_float(w.x << 16);
        x[1] = __uint_as_float(w.x & 0xffff0000u);
        x[2] = __uint_as_float(w.y << 16);
        x[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
        x[0] = __uint_as_float(w << 16);
        x[1] = __uint_as_float(w & 0xffff0000u);
    }
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < V; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float c = gain / sqrtf(ss / (float)d + eps);
    __nv_bfloat16* dst = khat + rw * d + lane * V;
    const __nv_bfloat162 p0 = __floats2bfloat162_rn(c * x[0], c * x[1]);
    if constexpr (V == 4) {
        const __nv_bfloat162 p1 = __floats2bfloat162_rn(c * x[2], c * x[3]);
        *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&p0),
                                                    *reinterpret_cast<const uint32_t*>(&p1));
    } else {
        *reinterpret_cast<__nv_bfloat162*>(dst) = p0;
    }
    if (lane == 0) {
        const int64_t t = rw / H, h = rw % H;
        scale[h * ld + t] = c;
    }
}

}  // namespace

const void* plan_key_norm(Plan& p, const void* k, cudaStream_t st, gdpa_status* s) {
    *s = GDPA_OK;
    if (p.d != 64 && p.d != 128) {
        *s = GDPA_ERR_UNSUPPORTED;
        return nullptr;
    }
    const int64_t ld = p.Tkv + 128;
    if (!p.d_kscale) {
        const size_t bytes = (size_t)p.H * ld * sizeof(float);
        if (cudaMallocAsync((void**)&p.d_kscale, bytes, st) != cudaSuccess) {
            p.d_kscale = nullptr;
            *s = GDPA_ERR_ALLOC;
            return nullptr;
        }
        if (cudaMemsetAsync(p.d_kscale, 0, bytes, st) != cudaSuccess) {
            *s = GDPA_ERR_CUDA;
            return nullptr;
        }
    }
    const int64_t n = p.Tkv * p.H;
    if (!p.d_khat && n > 0 &&
        cudaMallocAsync(&p.d_khat, (size_t)n * p.d * sizeof(__nv_bfloat16), st) != cudaSuccess) {
        p.d_khat = nullptr;
        *s = GDPA_ERR_ALLOC;
        return nullptr;
    }
    if (n == 0) return k;
    const unsigned grid = (unsigned)((n + 7) / 8);
    if (p.d == 128)
        key_norm_kernel<4><<<grid, 256, 0, st>>>((const __nv_bfloat16*)k, (__nv_bfloat16*)p.d_khat,
                                                 p.d_kscale, p.Tkv, p.H, ld, p.qk_gain, p.qk_eps);
    else
        key_norm_kernel<2><<<grid, 256, 0, st>>>((const __nv_bfloat16*)k, (__nv_bfloat16*)p.d_khat,
                                                 p.d_kscale, p.Tkv, p.H, ld, p.qk_gain, p.qk_eps);
    if (cudaGetLastError() != cudaSuccess) {
        *s = GDPA_ERR_CUDA;
        return nullptr;
    }
    p.launches += 1;
    return p.d_khat;
}

}  // namespace gdpa
