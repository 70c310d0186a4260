// Internal declarations shared by the host planner, the ABI layer and the
// kernel launchers of the GDPA library.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "gdpa.h"

namespace gdpa {

constexpr int kBM = GDPA_BLOCK_M;  // query rows per tile
constexpr int kBN = GDPA_BLOCK_N;  // key rows per block

// One forward tile as the kernels read it: query rows [qt0, qt0 + nq) of a
// sample whose keys are rows [kvt0, kvt0 + lkv); key blocks [kb0, kb1) of
// kBN rows; i0 = position of the tile's first query inside its sample.
struct FwdTile {
    int32_t qt0, nq, kvt0, lkv, h, kb0, kb1, i0;
};
static_assert(sizeof(FwdTile) == 32, "FwdTile layout");

// One backward unit: key rows [kvt0, kvt0 + nkv) at position c0 inside a
// sample whose queries are rows [qt0, qt0 + lq); query tiles [m0, m1).
// hf = head | flags << 16 (flag bit 0: dQ by atomic add).
struct BwdUnit {
    int32_t kvt0, nkv, qt0, lq, hf, m0, m1, c0;
};
static_assert(sizeof(BwdUnit) == 32, "BwdUnit layout");

constexpr int kUnitAtomicDQ = 1;

// Device error word layout (int32[4]): code, where, cta, detail.
enum DevErr : int32_t { kDevOk = 0, kDevTimeout = 1, kDevBad = 2 };

// Stream-ordered bookkeeping of a plan's device work: one event per stream
// the plan has launched on, recorded after each call, so that destroying the
// plan or reading its timings waits for this plan's work only.
struct StreamEvent {
    cudaStream_t stream;
    cudaEvent_t event;
};

struct Plan {
    int device = 0;
    bool host_only = false;
    int B = 0, H = 0, d = 0, mask = 0, window = 0, sched = 0, S = 0;
    int max_kvb = 0;
    int kernel = GDPA_KERNEL_AUTO;
    int timing = 0;
    int64_t Tq = 0, Tkv = 0;
    int zero_dq = 0;
    int fwd_split = 0;
    std::vector<int32_t> fwd_export;  // [n][6] b, h, m, kb0, kb1, sm
    std::vector<int32_t> fwd_seg;     // [S + 1]
    std::vector<int32_t> bwd_export;  // [n][7] b, h, j, m0, m1, flags, sm
    std::vector<int32_t> bwd_seg;     // [S + 1]
    std::vector<FwdTile> fwd_dev_host;  // kernel records in queue order
    std::vector<BwdUnit> bwd_dev_host;
    int64_t n_fwd = 0, n_bwd = 0;
    int64_t max_fwd_kvb = 0;          // largest kb1 - kb0 over forward tiles
    // device copies (owned)
    FwdTile* d_fwd = nullptr;
    int32_t* d_fwd_seg = nullptr;
    BwdUnit* d_bwd = nullptr;
    int32_t* d_bwd_seg = nullptr;
    int32_t* d_err = nullptr;                // [4]
    int32_t last_err[4] = {0, 0, 0, 0};      // the last failure gdpa_check read
    unsigned long long* d_times = nullptr;   // [2][S][2]
    int32_t* d_smid = nullptr;               // [2][S]
    int timed[2] = {0, 0};
    cudaStream_t timed_stream[2] = {nullptr, nullptr};
    int64_t launches = 0;
    // the upload of the plan (recorded on the creation stream); every launch
    // waits for it on its own stream
    cudaEvent_t ready = nullptr;
    std::vector<StreamEvent> work;
    // failure-path test hook: bounded-wait limit in microseconds (0 = the
    // kernels' default) and whether CTA 0's loader skips its first query-tile
    // load so that a wait expires
    uint32_t wait_limit_us = 0;
    int stall = 0;
    // fused RMSNorm of Q and K rows (gain > 0 enables): the keys' g / rms in
    // a [H][Tkv + 128] float workspace and the normalised keys (bf16,
    // [Tkv][H][d]), refreshed by every launch
    float qk_gain = 0.0f, qk_eps = 0.0f;
    float* d_kscale = nullptr;
    void* d_khat = nullptr;
    // MXFP8 entry points: bf16 expansion of Q's rows then K's rows,
    // [q_rows + Tkv][H][d], allocated on first use
    void* d_mxqk = nullptr;
    size_t mxqk_bytes = 0;
    bool mx_ready = false;   // it holds the last MXFP8 call's Q and K
    // softmax-variant backward: dO_t . O_t per row and head, [Tq][H] float,
    // allocated on first use
    float* d_delta = nullptr;
    // key-split forward (d = 128): float32 partial sums of O, [Tq][H][d],
    // allocated on first use
    float* d_wsplit = nullptr;
    // shared-query mode: > 0 = number of seed rows in Q (every sample's
    // queries are seeds 0 .. Lq_b - 1); dQ is then [shared_q][H][d]
    int shared_q = 0;
    int64_t max_lq = 0;   // longest sample (query rows)
};

// Host planner (gdpa_plan.cpp): fills the host-side vectors of `p` from the
// offsets; returns GDPA_OK or INVALID_ARG.
gdpa_status build_plan_host(Plan& p, const int32_t* q_off, const int32_t* kv_off);

// Kernel launchers.  Arguments are already validated by the ABI layer.
// lse (softmax variant, may be NULL): row log-sum-exp out; lse / delta in
// the backward: that output and dO.O per row (softmax variant only).
gdpa_status launch_simt_fwd(Plan& p, gdpa_dtype dt, const void* q, const void* k, const void* v,
                            void* o, float* lse, float alpha, int act, cudaStream_t st);
gdpa_status launch_simt_bwd(Plan& p, gdpa_dtype dt, const void* q, const void* k, const void* v,
                            const void* d_o, float* dq, float* dk, float* dv, float alpha, int act,
                            const float* lse, const float* delta, cudaStream_t st);
gdpa_status launch_tc_fwd(Plan& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, float alpha, int act, cudaStream_t st);
// Forward tensor-core launch on explicit device buffers (tile queue, queue
// starts, error word; times/smid may be NULL to skip per-CTA timing).
// qk_gain > 0: fused RMSNorm, with k already normalised (plan_key_norm).
gdpa_status launch_tc_fwd_raw(const FwdTile* tiles, const int32_t* seg, int S, int32_t* err,
                              unsigned long long* times, int32_t* smid, int H, int d, int64_t Tq,
                              int64_t Tkv, int mask, int window, const void* q, int64_t q_rows,
                              int shared_q, const void* k, const void* v, void* o, float* lse,
                              float* w, float alpha, int act, cudaStream_t st,
                              uint32_t wait_limit_us = 0, int stall = 0,
                              float qk_gain = 0.0f, float qk_eps = 0.0f);
gdpa_status launch_tc_bwd(Plan& p, const void* q, const void* k, const void* v, const void* d_o,
                          float* dq, float* dk, float* dv, float alpha, int act, const float* lse,
                          const float* delta, cudaStream_t st);
// Fused RMSNorm of the keys (d = 64 or 128): c = gain / sqrt(mean(k^2) +
// eps) of every (token, head) row of `k` into the plan's d_kscale
// ([H][Tkv + 128] floats) and the normalised rows c k (bf16) into d_khat
// ([Tkv][H][d]); both allocated on first use, stream ordered.  Returns
// d_khat (k itself when Tkv = 0) or NULL (status in *s).
const void* plan_key_norm(Plan& p, const void* k, cudaStream_t st, gdpa_status* s);
// MXFP8 (32-value blocks): bf16 x[n] <-> E4M3 codes el[n] + scale bytes
// sc[n / 32]; n a multiple of 32
gdpa_status launch_mx_quantise(const void* x, int64_t n_values, uint8_t* el, uint8_t* sc,
                               cudaStream_t st);
gdpa_status launch_mx_dequantise(const uint8_t* el, const uint8_t* sc, int64_t n_values, void* x,
                                 cudaStream_t st);
// delta[t][h] = dO[t][h][:] . O[t][h][:] over rows t < Tq (softmax variant)
gdpa_status launch_row_dot(Plan& p, gdpa_dtype dt, const void* d_o, const void* o, float* delta,
                           cudaStream_t st);

}  // namespace gdpa
