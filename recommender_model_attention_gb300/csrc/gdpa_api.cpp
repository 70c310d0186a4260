// C ABI of the GDPA library: argument checks, plan ownership, dispatch to
// the kernel launchers, and device error reporting.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "gdpa_internal.h"

using gdpa::Plan;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Plan buffers come from the stream-ordered allocator on the creation
// stream and go back to it on a stream that has waited for the plan's work,
// so neither creating nor destroying a plan synchronises the device.
template <typename T>
gdpa_status upload(T** dst, const void* src, size_t bytes, cudaStream_t st) {
    if (bytes == 0) return GDPA_OK;
    if (cudaMallocAsync((void**)dst, bytes, st) != cudaSuccess) {
        *dst = nullptr;
        return GDPA_ERR_ALLOC;
    }
    if (cudaMemcpyAsync(*dst, src, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return GDPA_ERR_CUDA;
    return GDPA_OK;
}

template <typename T>
gdpa_status alloc_dev(T** dst, size_t bytes, cudaStream_t st) {
    if (cudaMallocAsync((void**)dst, bytes, st) != cudaSuccess) {
        *dst = nullptr;
        return GDPA_ERR_ALLOC;
    }
    return GDPA_OK;
}

// Host wait for every launch this plan has enqueued (its own events only).
gdpa_status wait_plan_work(const Plan& p) {
    for (const gdpa::StreamEvent& w : p.work)
        if (cudaEventSynchronize(w.event) != cudaSuccess) return GDPA_ERR_CUDA;
    return GDPA_OK;
}

void free_plan(Plan* p) {
    if (!p) return;
    if (!p->host_only) {
        int cur = -1;
        if (cudaGetDevice(&cur) == cudaSuccess && cur != p->device) cudaSetDevice(p->device);
        // A private stream waits (on the device) for every stream the plan
        // has launched on and for the upload, then returns the buffers; the
        // host does not wait.  If the stream cannot be made, fall back to a
        // host wait on the plan's own events.
        cudaStream_t fs = nullptr;
        if (cudaStreamCreateWithFlags(&fs, cudaStreamNonBlocking) != cudaSuccess) {
            fs = nullptr;
            wait_plan_work(*p);
            if (p->ready) cudaEventSynchronize(p->ready);
        } else {
            if (p->ready) cudaStreamWaitEvent(fs, p->ready, 0);
            for (const gdpa::StreamEvent& w : p->work) cudaStreamWaitEvent(fs, w.event, 0);
        }
        void* bufs[] = {p->d_fwd, p->d_fwd_seg, p->d_bwd, p->d_bwd_seg, p->d_err,
                        p->d_times, p->d_smid, p->d_delta, p->d_wsplit, p->d_kscale, p->d_mxqk,
                        p->d_khat};
        for (void* b : bufs)
            if (b) cudaFreeAsync(b, fs);
        for (const gdpa::StreamEvent& w : p->work) cudaEventDestroy(w.event);
        if (p->ready) cudaEventDestroy(p->ready);
        if (fs) cudaStreamDestroy(fs);   // released once its work has run
        if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    }
    delete p;
}

// Calls that touch a plan's device buffers must run with the plan's device
// current (the buffers live there).
gdpa_status check_device(const Plan& p) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return GDPA_ERR_CUDA;
    return cur == p.device ? GDPA_OK : GDPA_ERR_INVALID_ARG;
}

// Order a launch on `st` after the plan's upload, and remember `st` so that
// the plan's destruction and timing reads wait for this work.
gdpa_status begin_work(Plan& p, cudaStream_t st) {
    if (p.ready && cudaStreamWaitEvent(st, p.ready, 0) != cudaSuccess) return GDPA_ERR_CUDA;
    return GDPA_OK;
}

void end_work(Plan& p, cudaStream_t st) {
    for (gdpa::StreamEvent& w : p.work)
        if (w.stream == st) {
            cudaEventRecord(w.event, st);
            return;
        }
    gdpa::StreamEvent w{st, nullptr};
    if (cudaEventCreateWithFlags(&w.event, cudaEventDisableTiming) != cudaSuccess) {
        // no event: fall back to waiting for this stream now
        cudaStreamSynchronize(st);
        return;
    }
    cudaEventRecord(w.event, st);
    p.work.push_back(w);
}

bool valid_act(int a) { return a >= GDPA_ACT_GELU_ERF && a <= GDPA_ACT_SOFTMAX; }

// true when this plan/dtype combination runs on the tcgen05 kernels
bool use_tc(const Plan& p, gdpa_dtype dt) {
    if (dt != GDPA_BF16) return false;
    if (p.kernel == GDPA_KERNEL_SIMT) return false;
    return p.d == 64 || p.d == 128;
}


}  // namespace

extern "C" const char* gdpa_status_str(gdpa_status s) {
    switch (s) {
    case GDPA_OK: return "ok";
    case GDPA_ERR_INVALID_ARG: return "invalid argument";
    case GDPA_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDPA_ERR_CUDA: return "CUDA error";
    case GDPA_ERR_ALLOC: return "allocation failed";
    case GDPA_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case GDPA_ERR_DEVICE: return "kernel reported an internal error";
    case GDPA_ERR_SCRATCH_LIMIT: return "batch exceeds the static scratch of gdpa_fwd_noalloc";
    }
    return "unknown status";
}

namespace {

gdpa_status create_common(const int32_t* q_off_host, const int32_t* kv_off_host, int B, int H,
                          int d, gdpa_mask mask, int window, gdpa_sched sched, int num_sms,
                          int max_kv_blocks_per_tile, bool host_only, cudaStream_t s,
                          gdpa_plan* out) {
    if (!out) return GDPA_ERR_INVALID_ARG;
    *out = nullptr;
    if (!q_off_host || !kv_off_host || B < 0 || H < 1 || d < 1) return GDPA_ERR_INVALID_ARG;
    if (mask != GDPA_MASK_NONE && mask != GDPA_MASK_CAUSAL_WINDOW) return GDPA_ERR_INVALID_ARG;
    if (mask == GDPA_MASK_CAUSAL_WINDOW && window < 1) return GDPA_ERR_INVALID_ARG;
    if (sched != GDPA_SCHED_ZIGZAG && sched != GDPA_SCHED_ROUND_ROBIN &&
        sched != GDPA_SCHED_ZIGZAG_TIMED)
        return GDPA_ERR_INVALID_ARG;
    if (num_sms < 0 || max_kv_blocks_per_tile < GDPA_KV_SPLIT_AUTO) return GDPA_ERR_INVALID_ARG;
    if (host_only && num_sms == 0) return GDPA_ERR_INVALID_ARG;
    if (d > 128 || d % 4 != 0) return GDPA_ERR_UNSUPPORTED;
    if ((int64_t)H * d > (1 << 20)) return GDPA_ERR_UNSUPPORTED;

    Plan* p = new (std::nothrow) Plan();
    if (!p) return GDPA_ERR_ALLOC;
    p->host_only = host_only;
    if (!host_only) {
        if (cudaGetDevice(&p->device) != cudaSuccess) {
            delete p;
            return GDPA_ERR_CUDA;
        }
        if (num_sms == 0 && cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount,
                                                   p->device) != cudaSuccess) {
            delete p;
            return GDPA_ERR_CUDA;
        }
    }
    p->B = B;
    p->H = H;
    p->d = d;
    p->mask = mask;
    p->window = mask == GDPA_MASK_CAUSAL_WINDOW ? window : 0;
    p->sched = sched;
    p->S = num_sms;
    p->max_kvb = max_kv_blocks_per_tile;
    gdpa_status st = gdpa::build_plan_host(*p, q_off_host, kv_off_host);
    if (st != GDPA_OK) {
        delete p;
        return st;
    }
    if (!host_only) {
        const size_t S1 = (size_t)p->S + 1;
        if ((st = upload(&p->d_fwd, p->fwd_dev_host.data(),
                         p->fwd_dev_host.size() * sizeof(gdpa::FwdTile), s)) ||
            (st = upload(&p->d_fwd_seg, p->fwd_seg.data(), S1 * sizeof(int32_t), s)) ||
            (st = upload(&p->d_bwd, p->bwd_dev_host.data(),
                         p->bwd_dev_host.size() * sizeof(gdpa::BwdUnit), s)) ||
            (st = upload(&p->d_bwd_seg, p->bwd_seg.data(), S1 * sizeof(int32_t), s)) ||
            (st = alloc_dev(&p->d_err, 4 * sizeof(int32_t), s)) ||
            (st = alloc_dev(&p->d_times, 2 * (size_t)p->S * 2 * sizeof(unsigned long long), s)) ||
            (st = alloc_dev(&p->d_smid, 2 * (size_t)p->S * sizeof(int32_t), s))) {
            cudaStreamSynchronize(s);
            free_plan(p);
            return st;
        }
        // the upload is ordered on `s`; launches on any stream wait for this
        // event instead of the host waiting here
        if (cudaMemsetAsync(p->d_err, 0, 4 * sizeof(int32_t), s) != cudaSuccess ||
            cudaEventCreateWithFlags(&p->ready, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventRecord(p->ready, s) != cudaSuccess) {
            cudaStreamSynchronize(s);
            free_plan(p);
            return GDPA_ERR_CUDA;
        }
        // the kernel-layout records stay with the plan (host memory) until it
        // is destroyed, so their copies never read freed memory
        *out = (gdpa_plan)p;
        return GDPA_OK;
    }
    std::vector<gdpa::FwdTile>().swap(p->fwd_dev_host);
    std::vector<gdpa::BwdUnit>().swap(p->bwd_dev_host);
    *out = (gdpa_plan)p;
    return GDPA_OK;
}

}  // namespace

extern "C" {

gdpa_status gdpa_plan_create(const int32_t* q_off_host, const int32_t* kv_off_host, int B, int H,
                             int d, gdpa_mask mask, int window, gdpa_sched sched, int num_sms,
                             int max_kv_blocks_per_tile, void* stream, gdpa_plan* out) {
    return create_common(q_off_host, kv_off_host, B, H, d, mask, window, sched, num_sms,
                         max_kv_blocks_per_tile, false, (cudaStream_t)stream, out);
}

gdpa_status gdpa_plan_create_host(const int32_t* q_off_host, const int32_t* kv_off_host, int B,
                                  int H, int d, gdpa_mask mask, int window, gdpa_sched sched,
                                  int num_sms, int max_kv_blocks_per_tile, gdpa_plan* out) {
    return create_common(q_off_host, kv_off_host, B, H, d, mask, window, sched, num_sms,
                         max_kv_blocks_per_tile, true, nullptr, out);
}

gdpa_status gdpa_plan_sizes(gdpa_plan plan, int64_t* n_fwd, int64_t* n_bwd, int* num_sms) {
    if (!plan) return GDPA_ERR_INVALID_ARG;
    Plan* p = (Plan*)plan;
    if (n_fwd) *n_fwd = p->n_fwd;
    if (n_bwd) *n_bwd = p->n_bwd;
    if (num_sms) *num_sms = p->S;
    return GDPA_OK;
}

gdpa_status gdpa_plan_export(gdpa_plan plan, int32_t* tiles_out, int64_t cap, int64_t* n_out,
                             int32_t* seg_start_out) {
    if (!plan) return GDPA_ERR_INVALID_ARG;
    Plan* p = (Plan*)plan;
    if (n_out) *n_out = p->n_fwd;
    if (seg_start_out) memcpy(seg_start_out, p->fwd_seg.data(), p->fwd_seg.size() * sizeof(int32_t));
    if (cap < p->n_fwd || (p->n_fwd > 0 && !tiles_out)) return GDPA_ERR_INVALID_ARG;
    if (p->n_fwd) memcpy(tiles_out, p->fwd_export.data(), p->fwd_export.size() * sizeof(int32_t));
    return GDPA_OK;
}

gdpa_status gdpa_plan_export_bwd(gdpa_plan plan, int32_t* units_out, int64_t cap, int64_t* n_out,
                                 int32_t* seg_start_out, int* zero_dq_out) {
    if (!plan) return GDPA_ERR_INVALID_ARG;
    Plan* p = (Plan*)plan;
    if (n_out) *n_out = p->n_bwd;
    if (zero_dq_out) *zero_dq_out = p->zero_dq;
    if (seg_start_out) memcpy(seg_start_out, p->bwd_seg.data(), p->bwd_seg.size() * sizeof(int32_t));
    if (cap < p->n_bwd || (p->n_bwd > 0 && !units_out)) return GDPA_ERR_INVALID_ARG;
    if (p->n_bwd) memcpy(units_out, p->bwd_export.data(), p->bwd_export.size() * sizeof(int32_t));
    return GDPA_OK;
}

gdpa_status gdpa_plan_set_kernel(gdpa_plan plan, gdpa_kernel kernel) {
    if (!plan || kernel < GDPA_KERNEL_AUTO || kernel > GDPA_KERNEL_SIMT) return GDPA_ERR_INVALID_ARG;
    ((Plan*)plan)->kernel = kernel;
    return GDPA_OK;
}

gdpa_status gdpa_plan_set_shared_q(gdpa_plan plan, int n_seeds) {
    if (!plan || n_seeds < 0) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (n_seeds > 0 && p.max_lq > n_seeds) return GDPA_ERR_INVALID_ARG;
    p.shared_q = n_seeds;
    return GDPA_OK;
}

gdpa_status gdpa_plan_set_qk_norm(gdpa_plan plan, float gain, float eps) {
    if (!plan || !(gain >= 0.0f) || !(eps >= 0.0f)) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (gain > 0.0f && eps == 0.0f) return GDPA_ERR_INVALID_ARG;   // rows of zeros
    p.qk_gain = gain;
    p.qk_eps = eps;
    return GDPA_OK;
}

gdpa_status gdpa_plan_set_timing(gdpa_plan plan, int enable) {
    if (!plan) return GDPA_ERR_INVALID_ARG;
    ((Plan*)plan)->timing = enable ? 1 : 0;
    return GDPA_OK;
}

int64_t gdpa_plan_launches(gdpa_plan plan) { return plan ? ((Plan*)plan)->launches : -1; }

namespace {

gdpa_status fwd_common(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                       const void* v, void* o, float* lse, float alpha, gdpa_act act,
                       void* stream) {
    if (!plan || ((Plan*)plan)->host_only) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (dtype != GDPA_BF16 && dtype != GDPA_F32) return GDPA_ERR_INVALID_ARG;
    if (!valid_act(act)) return GDPA_ERR_INVALID_ARG;
    if (p.Tq > 0 && (!q || !o)) return GDPA_ERR_INVALID_ARG;
    if (p.Tkv > 0 && (!k || !v)) return GDPA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return GDPA_ERR_INVALID_ARG;
    if (gdpa_status ds = check_device(p)) return ds;
    if (p.n_fwd == 0) return GDPA_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (p.kernel == GDPA_KERNEL_TCGEN05 && !use_tc(p, dtype)) return GDPA_ERR_UNSUPPORTED;
    // key-split tiles: the softmax variant's chunks would need a max/sum
    // merge; the tensor-core forward splits only d = 128 (AUTO runs other
    // head dims' split plans on the CUDA-core kernels)
    if (p.fwd_split && act == GDPA_ACT_SOFTMAX) return GDPA_ERR_UNSUPPORTED;
    const bool tc =
        use_tc(p, dtype) && !(p.fwd_split && p.d != 128 && p.kernel == GDPA_KERNEL_AUTO);
    // the fused RMSNorm runs in the tensor-core kernels only
    if (p.qk_gain > 0.0f && !tc) return GDPA_ERR_UNSUPPORTED;
    if (gdpa_status bs = begin_work(p, st)) return bs;
    const gdpa_status s = tc ? gdpa::launch_tc_fwd(p, q, k, v, o, lse, alpha, act, st)
                             : gdpa::launch_simt_fwd(p, dtype, q, k, v, o, lse, alpha, act, st);
    if (tc && p.timing) p.timed_stream[0] = st;
    end_work(p, st);
    return s;
}

gdpa_status bwd_common(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                       const void* v, const void* o, const void* d_o, const float* lse, float* dq,
                       float* dk, float* dv, float alpha, gdpa_act act, void* stream) {
    if (!plan || ((Plan*)plan)->host_only) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (dtype != GDPA_BF16 && dtype != GDPA_F32) return GDPA_ERR_INVALID_ARG;
    if (!valid_act(act)) return GDPA_ERR_INVALID_ARG;
    const bool sm = act == GDPA_ACT_SOFTMAX;
    if (sm && p.Tq > 0 && (!o || !lse)) return GDPA_ERR_INVALID_ARG;
    if (sm && !aligned16(o)) return GDPA_ERR_INVALID_ARG;
    if (p.Tq > 0 && (!q || !d_o || !dq)) return GDPA_ERR_INVALID_ARG;
    if (p.Tkv > 0 && (!k || !v || !dk || !dv)) return GDPA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(d_o) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv))
        return GDPA_ERR_INVALID_ARG;
    if (gdpa_status ds = check_device(p)) return ds;
    cudaStream_t st = (cudaStream_t)stream;
    if (p.kernel == GDPA_KERNEL_TCGEN05 && !use_tc(p, dtype)) return GDPA_ERR_UNSUPPORTED;
    if (p.qk_gain > 0.0f && !use_tc(p, dtype)) return GDPA_ERR_UNSUPPORTED;
    if (gdpa_status bs = begin_work(p, st)) return bs;
    const float* delta = nullptr;
    gdpa_status s = GDPA_OK;
    if (sm && p.Tq > 0) {
        // D = dO . O per row, in the plan's workspace (allocated once, stream
        // ordered on this call's stream)
        if (!p.d_delta &&
            cudaMallocAsync((void**)&p.d_delta, (size_t)p.Tq * p.H * sizeof(float), st) !=
                cudaSuccess) {
            p.d_delta = nullptr;
            s = GDPA_ERR_ALLOC;
        }
        if (s == GDPA_OK) s = gdpa::launch_row_dot(p, dtype, d_o, o, p.d_delta, st);
        delta = p.d_delta;
    }
    if (s == GDPA_OK) {
        if (use_tc(p, dtype)) {
            s = gdpa::launch_tc_bwd(p, q, k, v, d_o, dq, dk, dv, alpha, act, lse, delta, st);
            if (p.timing) p.timed_stream[1] = st;
        } else {
            s = gdpa::launch_simt_bwd(p, dtype, q, k, v, d_o, dq, dk, dv, alpha, act, lse, delta,
                                      st);
        }
    }
    end_work(p, st);
    return s;
}

}  // namespace

gdpa_status gdpa_fwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k, const void* v,
                     void* o, float alpha, gdpa_act act, void* stream) {
    return fwd_common(plan, dtype, q, k, v, o, nullptr, alpha, act, stream);
}

gdpa_status gdpa_bwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k, const void* v,
                     const void* d_o, float* dq, float* dk, float* dv, float alpha, gdpa_act act,
                     void* stream) {
    // the softmax variant's gradients need O and the row statistics
    if (act == GDPA_ACT_SOFTMAX) return GDPA_ERR_UNSUPPORTED;
    return bwd_common(plan, dtype, q, k, v, nullptr, d_o, nullptr, dq, dk, dv, alpha, act, stream);
}

gdpa_status gdpa_softmax_fwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                             const void* v, void* o, float* lse, float alpha, void* stream) {
    if (plan && ((Plan*)plan)->Tq > 0 && !lse) return GDPA_ERR_INVALID_ARG;
    return fwd_common(plan, dtype, q, k, v, o, lse, alpha, GDPA_ACT_SOFTMAX, stream);
}

gdpa_status gdpa_softmax_bwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                             const void* v, const void* o, const void* d_o, const float* lse,
                             float* dq, float* dk, float* dv, float alpha, void* stream) {
    return bwd_common(plan, dtype, q, k, v, o, d_o, lse, dq, dk, dv, alpha, GDPA_ACT_SOFTMAX,
                      stream);
}

gdpa_status gdpa_mx_quantise(const void* x, int64_t n, uint8_t* elements, uint8_t* scales,
                             void* stream) {
    if (n < 0 || n % 32) return GDPA_ERR_INVALID_ARG;
    if (n == 0) return GDPA_OK;
    if (!x || !elements || !scales || !aligned16(x) || !aligned16(elements))
        return GDPA_ERR_INVALID_ARG;
    return gdpa::launch_mx_quantise(x, n, elements, scales, (cudaStream_t)stream);
}

gdpa_status gdpa_mx_dequantise(const uint8_t* elements, const uint8_t* scales, int64_t n, void* x,
                               void* stream) {
    if (n < 0 || n % 32) return GDPA_ERR_INVALID_ARG;
    if (n == 0) return GDPA_OK;
    if (!x || !elements || !scales || !aligned16(x) || !aligned16(elements))
        return GDPA_ERR_INVALID_ARG;
    return gdpa::launch_mx_dequantise(elements, scales, n, x, (cudaStream_t)stream);
}

}  // extern "C"

namespace {

// Expands MXFP8 Q and K into the plan's bf16 workspace (allocated on the
// stream on first use) and returns where the expansions start.
gdpa_status mx_expand(Plan& p, const uint8_t* q_el, const uint8_t* q_sc, const uint8_t* k_el,
                      const uint8_t* k_sc, cudaStream_t st, const void** q, const void** k) {
    if (p.d % 32) return GDPA_ERR_INVALID_ARG;
    const int64_t q_rows = p.shared_q > 0 ? p.shared_q : p.Tq;
    const int64_t row = (int64_t)p.H * p.d;
    if (!q_el && !q_sc && !k_el && !k_sc && (q_rows > 0 || p.Tkv > 0)) {
        // reuse the expansion of the plan's previous MXFP8 call
        if (!p.mx_ready || (size_t)(q_rows + p.Tkv) * row * 2 > p.mxqk_bytes)
            return GDPA_ERR_INVALID_ARG;
        if (gdpa_status ds = check_device(p)) return ds;
        *q = p.d_mxqk;
        *k = (uint8_t*)p.d_mxqk + (size_t)q_rows * row * 2;
        return GDPA_OK;
    }
    if (q_rows > 0 && (!q_el || !q_sc || !aligned16(q_el))) return GDPA_ERR_INVALID_ARG;
    if (p.Tkv > 0 && (!k_el || !k_sc || !aligned16(k_el))) return GDPA_ERR_INVALID_ARG;
    if (gdpa_status ds = check_device(p)) return ds;
    const size_t bytes = (size_t)(q_rows + p.Tkv) * row * 2;
    if (p.d_mxqk && bytes > p.mxqk_bytes) {
        // the shared-query mode changed Q's row count: replace the workspace
        // once the plan's earlier work has run
        for (const gdpa::StreamEvent& w : p.work) cudaStreamWaitEvent(st, w.event, 0);
        cudaFreeAsync(p.d_mxqk, st);
        p.d_mxqk = nullptr;
        p.mx_ready = false;
    }
    if (!p.d_mxqk && bytes > 0) {
        if (cudaMallocAsync(&p.d_mxqk, bytes, st) != cudaSuccess) {
            p.d_mxqk = nullptr;
            return GDPA_ERR_ALLOC;
        }
        p.mxqk_bytes = bytes;
    }
    uint8_t* base = (uint8_t*)p.d_mxqk;
    *q = base;
    *k = base + (size_t)q_rows * row * 2;
    gdpa_status s = GDPA_OK;
    if (q_rows > 0) {
        s = gdpa::launch_mx_dequantise(q_el, q_sc, q_rows * row, (void*)*q, st);
        if (s == GDPA_OK) p.launches += 1;
    }
    if (s == GDPA_OK && p.Tkv > 0) {
        s = gdpa::launch_mx_dequantise(k_el, k_sc, p.Tkv * row, (void*)*k, st);
        if (s == GDPA_OK) p.launches += 1;
    }
    end_work(p, st);   // the workspace is in use until these have run
    p.mx_ready = s == GDPA_OK;
    return s;
}

}  // namespace

extern "C" {

gdpa_status gdpa_fwd_mx(gdpa_plan plan, const uint8_t* q_el, const uint8_t* q_sc,
                        const uint8_t* k_el, const uint8_t* k_sc, const void* v, void* o,
                        float alpha, gdpa_act act, void* stream) {
    if (!plan || ((Plan*)plan)->host_only) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (!valid_act(act)) return GDPA_ERR_INVALID_ARG;
    if (p.Tq > 0 && !o) return GDPA_ERR_INVALID_ARG;
    if (p.Tkv > 0 && !v) return GDPA_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(o)) return GDPA_ERR_INVALID_ARG;
    if (p.kernel == GDPA_KERNEL_TCGEN05 && !use_tc(p, GDPA_BF16)) return GDPA_ERR_UNSUPPORTED;
    const void *q = nullptr, *k = nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    if (gdpa_status s = mx_expand(p, q_el, q_sc, k_el, k_sc, st, &q, &k)) return s;
    return fwd_common(plan, GDPA_BF16, q, k, v, o, nullptr, alpha, act, stream);
}

gdpa_status gdpa_bwd_mx(gdpa_plan plan, const uint8_t* q_el, const uint8_t* q_sc,
                        const uint8_t* k_el, const uint8_t* k_sc, const void* v, const void* d_o,
                        float* dq, float* dk, float* dv, float alpha, gdpa_act act, void* stream) {
    if (!plan || ((Plan*)plan)->host_only) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (!valid_act(act)) return GDPA_ERR_INVALID_ARG;
    if (act == GDPA_ACT_SOFTMAX) return GDPA_ERR_UNSUPPORTED;
    if (p.Tq > 0 && (!d_o || !dq)) return GDPA_ERR_INVALID_ARG;
    if (p.Tkv > 0 && (!v || !dk || !dv)) return GDPA_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(d_o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return GDPA_ERR_INVALID_ARG;
    if (p.kernel == GDPA_KERNEL_TCGEN05 && !use_tc(p, GDPA_BF16)) return GDPA_ERR_UNSUPPORTED;
    const void *q = nullptr, *k = nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    if (gdpa_status s = mx_expand(p, q_el, q_sc, k_el, k_sc, st, &q, &k)) return s;
    return bwd_common(plan, GDPA_BF16, q, k, v, nullptr, d_o, nullptr, dq, dk, dv, alpha, act,
                      stream);
}

gdpa_status gdpa_check(gdpa_plan plan, void* stream) {
    if (!plan || ((Plan*)plan)->host_only) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (gdpa_status ds = check_device(p)) return ds;
    cudaStream_t st = (cudaStream_t)stream;
    // the plan's own launches (on whatever streams), then `stream`
    if (wait_plan_work(p) != GDPA_OK || cudaStreamSynchronize(st) != cudaSuccess)
        return GDPA_ERR_CUDA;
    int32_t err[4] = {0, 0, 0, 0};
    if (cudaMemcpyAsync(err, p.d_err, sizeof(err), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return GDPA_ERR_CUDA;
    if (err[0] == gdpa::kDevOk) return GDPA_OK;
    for (int j = 0; j < 4; ++j) p.last_err[j] = err[j];
    if (cudaMemsetAsync(p.d_err, 0, sizeof(err), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return GDPA_ERR_CUDA;
    return err[0] == gdpa::kDevTimeout ? GDPA_ERR_TIMEOUT : GDPA_ERR_DEVICE;
}

gdpa_status gdpa_error_detail(gdpa_plan plan, int32_t* detail) {
    if (!plan || !detail) return GDPA_ERR_INVALID_ARG;
    const Plan& p = *(const Plan*)plan;
    for (int j = 0; j < 4; ++j) detail[j] = p.last_err[j];
    return GDPA_OK;
}

gdpa_status gdpa_sm_times(gdpa_plan plan, int which, uint64_t* start_end, int32_t* smid) {
    if (!plan || ((Plan*)plan)->host_only || which < 0 || which > 1 || !start_end || !smid)
        return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    if (!p.timed[which]) return GDPA_ERR_INVALID_ARG;
    if (gdpa_status ds = check_device(p)) return ds;
    // waits for this plan's launches only, and reads on the stream of the
    // timed launch
    cudaStream_t st = p.timed_stream[which];
    if (wait_plan_work(p) != GDPA_OK ||
        cudaMemcpyAsync(start_end, p.d_times + (size_t)which * p.S * 2,
                        (size_t)p.S * 2 * sizeof(uint64_t), cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyAsync(smid, p.d_smid + (size_t)which * p.S, (size_t)p.S * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return GDPA_ERR_CUDA;
    return GDPA_OK;
}

gdpa_status gdpa_plan_set_wait_test(gdpa_plan plan, int limit_us, int stall) {
    if (!plan || limit_us < 0) return GDPA_ERR_INVALID_ARG;
    Plan& p = *(Plan*)plan;
    p.wait_limit_us = (uint32_t)limit_us;
    p.stall = stall ? 1 : 0;
    return GDPA_OK;
}

void gdpa_plan_destroy(gdpa_plan plan) { free_plan((Plan*)plan); }

}  // extern "C"
