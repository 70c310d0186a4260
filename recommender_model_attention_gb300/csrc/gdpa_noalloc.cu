// gdpa_fwd_noalloc: the tensor-core forward for callers that cannot allocate
// device memory.
//
// Some callers run where cudaMalloc is not available to them: code inside a
// custom allocator or a memory pool's own bookkeeping, plugins handed a fixed
// device arena, or processes whose allocations must all be reserved up front.
// They cannot create a gdpa_plan (its tile queue and error word are
// allocated on the device).  This entry point plans on the host into static host
// buffers, uploads the tile queue into a file-scope static device array, and
// launches the same forward kernel.  It calls no cudaMalloc, cudaFree or
// other allocating routine and keeps its host state in static buffers; the
// only object it creates is one CUDA event per device, at set-up.
//
// The device array is GDPA_NOALLOC_SCRATCH_BYTES (about 1 MiB); every GPU
// that loads the library keeps it until the process exits.  All calls share
// it and it keeps the last call's contents, so calls whose launches overlap
// on the GPU (for example on two streams) race on it.  The error word in it
// is cleared by each call.
#include <mutex>

#include "gdpa_internal.h"

namespace gdpa {
namespace {

constexpr int kMaxTiles = GDPA_NOALLOC_MAX_TILES;
constexpr int kMaxSms = 1024;
constexpr int kMaxDevices = 64;

// layout of the device scratch: error word, SM queue starts, tile queue
constexpr size_t kOffErr = 0;
constexpr size_t kOffSeg = 256;
constexpr size_t kOffTiles = kOffSeg + ((sizeof(int32_t) * (kMaxSms + 1) + 255) / 256) * 256;
constexpr size_t kScratchBytes = kOffTiles + sizeof(FwdTile) * (size_t)kMaxTiles;
static_assert(kScratchBytes <= GDPA_NOALLOC_SCRATCH_BYTES, "scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDPA_NOALLOC_SCRATCH_BYTES];

// per-device set-up: the scratch's device address and an event that orders
// the reuse of the static host staging buffers after the previous upload
struct DeviceSlot {
    bool ready = false;
    unsigned char* scratch = nullptr;
    cudaEvent_t uploaded = nullptr;
    bool pending = false;
};
DeviceSlot g_slots[kMaxDevices];

// static host staging (no heap)
FwdTile h_tiles[kMaxTiles];
FwdTile h_queue[kMaxTiles];
int32_t h_cost[kMaxTiles];
int32_t h_order[kMaxTiles];
int32_t h_tmp[kMaxTiles];
int32_t h_seg[kMaxSms + 1];
int32_t h_fill[kMaxSms];
std::mutex g_mutex;

gdpa_status setup_device(int dev, DeviceSlot** out) {
    if (dev < 0 || dev >= kMaxDevices) return GDPA_ERR_UNSUPPORTED;
    DeviceSlot& s = g_slots[dev];
    if (!s.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return GDPA_ERR_CUDA;
        if (cudaEventCreateWithFlags(&s.uploaded, cudaEventDisableTiming) != cudaSuccess)
            return GDPA_ERR_CUDA;
        s.scratch = (unsigned char*)p;
        s.ready = true;
    }
    *out = &s;
    return GDPA_OK;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Stable sort of h_order[0..n) by h_cost descending (bottom-up merge sort
// on the static buffers).
void sort_by_cost(int n) {
    int32_t* a = h_order;
    int32_t* b = h_tmp;
    for (int w = 1; w < n; w *= 2) {
        for (int lo = 0; lo < n; lo += 2 * w) {
            const int mid = lo + w < n ? lo + w : n;
            const int hi = lo + 2 * w < n ? lo + 2 * w : n;
            int i = lo, j = mid, k = lo;
            while (i < mid && j < hi) b[k++] = (h_cost[a[j]] > h_cost[a[i]]) ? a[j++] : a[i++];
            while (i < mid) b[k++] = a[i++];
            while (j < hi) b[k++] = a[j++];
        }
        int32_t* t = a;
        a = b;
        b = t;
    }
    if (a != h_order)
        for (int i = 0; i < n; ++i) h_order[i] = a[i];
}

// The library's forward plan (same rules as gdpa_plan_create, zigzag, no
// key splitting) into the static staging; returns the tile count or -1 if it
// exceeds kMaxTiles, -2 for bad offsets.
int plan_static(const int32_t* q_off, const int32_t* kv_off, int B, int H, int mask, int window,
                int S) {
    if (q_off[0] != 0 || kv_off[0] != 0) return -2;
    int n = 0;
    for (int b = 0; b < B; ++b) {
        if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) return -2;
        const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
        for (int h = 0; h < H; ++h) {
            for (int64_t m = 0; m < cdiv(lq, kBM); ++m) {
                if (n >= kMaxTiles) return -1;
                const int64_t r0 = m * kBM, r1 = r0 + kBM < lq ? r0 + kBM : lq;
                int64_t lo = 0, hi = lkv;
                if (mask == GDPA_MASK_CAUSAL_WINDOW) {
                    lo = r0 - window + 1 > 0 ? r0 - window + 1 : 0;
                    hi = lkv < r1 ? lkv : r1;
                }
                int64_t k0 = 0, k1 = 0;
                if (lo < hi) {
                    k0 = lo / kBN;
                    k1 = cdiv(hi, kBN);
                }
                FwdTile& t = h_tiles[n];
                t.qt0 = (int32_t)(q_off[b] + r0);
                t.nq = (int32_t)(r1 - r0);
                t.kvt0 = kv_off[b];
                t.lkv = (int32_t)lkv;
                t.h = h;
                t.kb0 = (int32_t)k0;
                t.kb1 = (int32_t)k1;
                t.i0 = (int32_t)r0;
                h_cost[n] = (int32_t)(k1 - k0);
                h_order[n] = n;
                ++n;
            }
        }
    }
    sort_by_cost(n);
    for (int s = 0; s <= S; ++s) h_seg[s] = 0;
    for (int r = 0; r < n; ++r) {
        int p = r % S;
        if ((r / S) & 1) p = S - 1 - p;
        h_seg[p + 1]++;
    }
    for (int s = 0; s < S; ++s) h_seg[s + 1] += h_seg[s];
    for (int s = 0; s < S; ++s) h_fill[s] = h_seg[s];
    for (int r = 0; r < n; ++r) {
        int p = r % S;
        if ((r / S) & 1) p = S - 1 - p;
        h_queue[h_fill[p]++] = h_tiles[h_order[r]];
    }
    return n;
}

}  // namespace
}  // namespace gdpa

using namespace gdpa;

extern "C" gdpa_status gdpa_fwd_noalloc(const int32_t* q_off_host, const int32_t* kv_off_host,
                                        int B, int H, int d, gdpa_mask mask, int window,
                                        const void* q, const void* k, const void* v, void* o,
                                        float alpha, gdpa_act act, void* stream) {
    if (!q_off_host || !kv_off_host || B < 0 || H < 1) return GDPA_ERR_INVALID_ARG;
    if (mask != GDPA_MASK_NONE && mask != GDPA_MASK_CAUSAL_WINDOW) return GDPA_ERR_INVALID_ARG;
    if (mask == GDPA_MASK_CAUSAL_WINDOW && window < 1) return GDPA_ERR_INVALID_ARG;
    if (act < GDPA_ACT_GELU_ERF || act > GDPA_ACT_SOFTMAX) return GDPA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GDPA_ERR_UNSUPPORTED;
    const int64_t Tq = q_off_host[B], Tkv = kv_off_host[B];
    if (Tq > 0 && (!q || !o)) return GDPA_ERR_INVALID_ARG;
    if (Tkv > 0 && (!k || !v)) return GDPA_ERR_INVALID_ARG;
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)o) & 15u) return GDPA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int dev = 0, S = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&S, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GDPA_ERR_CUDA;
    if (S > kMaxSms) S = kMaxSms;

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceSlot* slot = nullptr;
    gdpa_status s = setup_device(dev, &slot);
    if (s != GDPA_OK) return s;
    // the staging buffers may still feed the previous call's upload (on any
    // device: the host staging is shared); a failed wait is reported once and
    // does not hold back later calls
    for (int i = 0; i < kMaxDevices; ++i) {
        if (g_slots[i].pending) {
            const cudaError_t e = cudaEventSynchronize(g_slots[i].uploaded);
            g_slots[i].pending = false;
            if (e != cudaSuccess) return GDPA_ERR_CUDA;
        }
    }
    const int n = plan_static(q_off_host, kv_off_host, B, H, mask, window, S);
    if (n == -2) return GDPA_ERR_INVALID_ARG;
    if (n < 0) return GDPA_ERR_SCRATCH_LIMIT;
    if (n == 0) return GDPA_OK;
    int32_t* d_err = (int32_t*)(slot->scratch + kOffErr);
    int32_t* d_seg = (int32_t*)(slot->scratch + kOffSeg);
    FwdTile* d_tiles = (FwdTile*)(slot->scratch + kOffTiles);
    if (cudaMemsetAsync(d_err, 0, 4 * sizeof(int32_t), st) != cudaSuccess ||
        cudaMemcpyAsync(d_seg, h_seg, sizeof(int32_t) * (S + 1), cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaMemcpyAsync(d_tiles, h_queue, sizeof(FwdTile) * n, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaEventRecord(slot->uploaded, st) != cudaSuccess)
        return GDPA_ERR_CUDA;
    slot->pending = true;
    return launch_tc_fwd_raw(d_tiles, d_seg, S, d_err, nullptr, nullptr, H, d, Tq, Tkv, mask,
                             window, q, Tq, 0, k, v, o, nullptr, nullptr, alpha, act, st);
}
