/*
 * gdpa.h - C ABI of the GB300 (sm_103a) GDPA library.
 *
 * GDPA (Generalized Dot-Product Attention) is defined on the page
 * "범용 내적 어텐션(GDPA): 실제 추천 시스템 학습 부하를 위한 커널 최적화"
 * (aitrends.kr), summary ("핵심 요약") and first paragraph of "섹션별 상세":
 * attention in which the softmax is replaced by an element-wise activation
 * such as GELU or SiLU.  For every sample b of a jagged batch and every head:
 *
 *     O_b = act(alpha * Q_b K_b^T) V_b
 *
 * with no row normalisation.  The same section describes host-side
 * precomputation of the valid tiles of a jagged batch and their zigzag
 * assignment to SMs (gdpa_plan_create), and the ALU-only 6th-order Taylor
 * GELU (GDPA_ACT_GELU_TAYLOR6).
 *
 * Conventions shared by every call:
 *   - Offsets are int32 exclusive prefix sums of the per-sample lengths:
 *     q_off[0] = 0, q_off[b+1] - q_off[b] = Lq_b, likewise kv_off; B samples.
 *   - Tensors are token-major with heads interleaved, row-major, contiguous:
 *     Q, O, dO are [q_off[B]][H][d]; K, V are [kv_off[B]][H][d];
 *     dQ is [q_off[B]][H][d] float32; dK, dV are [kv_off[B]][H][d] float32.
 *     Q, K, V, O, dO share one element type (gdpa_dtype).  Device pointers
 *     must be 16-byte aligned.
 *   - Query i of sample b is row q_off[b] + i; with the causal window W, key
 *     j of the same sample is valid for query i iff i - W < j <= i.  Pairs
 *     that are not valid contribute exactly zero; a row with no valid key
 *     gets a zero output (and zero dQ).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  gdpa_fwd / gdpa_bwd only enqueue work and never synchronise.
 *   - Every call returns a gdpa_status and never aborts.  Device-side
 *     failures (an expired wait in a kernel) are reported by gdpa_check.
 *   - The caller owns all tensors and streams; a plan owns its host and
 *     device buffers and is freed by gdpa_plan_destroy.
 *   - A plan belongs to the device that was current when it was created;
 *     every call that launches work on it or reads its device state
 *     (gdpa_fwd, gdpa_bwd, gdpa_softmax_fwd, gdpa_softmax_bwd, gdpa_fwd_mx,
 *     gdpa_bwd_mx, gdpa_check, gdpa_sm_times) must be made with that device
 *     current and returns
 *     INVALID_ARG, before touching the device, otherwise.
 */
#ifndef GDPA_H
#define GDPA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDPA_OK = 0,
    GDPA_ERR_INVALID_ARG = 1,   /* bad pointer, offsets, sizes or enum value */
    GDPA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head dim) */
    GDPA_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    GDPA_ERR_ALLOC = 4,         /* host or device allocation failed */
    GDPA_ERR_TIMEOUT = 5,       /* a kernel gave up waiting on a barrier */
    GDPA_ERR_DEVICE = 6,        /* a kernel flagged an internal inconsistency */
    GDPA_ERR_SCRATCH_LIMIT = 7  /* more tiles than gdpa_fwd_noalloc's static scratch holds */
} gdpa_status;

/* Element-wise activation applied to x = alpha * q.k (GDPA page, summary
 * and the SFU paragraph with its Taylor code figure). */
typedef enum {
    GDPA_ACT_GELU_ERF = 0,      /* x * Phi(x) = x/2 (1 + erf(x / sqrt 2)) */
    GDPA_ACT_GELU_TANH = 1,     /* x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
    GDPA_ACT_SILU = 2,          /* x / (1 + exp(-x)) */
    GDPA_ACT_GELU_TAYLOR6 = 3,  /* x/2 + (x^2 - x^4/6 + x^6/40) / sqrt(2 pi) */
    GDPA_ACT_IDENTITY = 4,      /* x (for tests of the linear algebra) */
    /* Softmax variant: O_i = sum_j softmax_j(alpha q_i.k_j) V_j over the row's
     * valid keys (0 for a row without one), i.e. Jagged Flash Attention, the
     * softmax kernel the GEM page ("GEM 트레이닝: Meta가 LLM 규모의 광고
     * 파운데이션 모델 효율성을 두 배로 높인 방법", techlist.io, section "GPU
     * 연산 효율을 높인 맞춤형 커널과 정밀도", its kernel list) names beside
     * GDPA.  gdpa_fwd, gdpa_fwd_noalloc and gdpa_softmax_fwd; its gradients
     * come from gdpa_softmax_bwd (gdpa_bwd returns UNSUPPORTED);
     * gdpa_act_eval returns INVALID_ARG. */
    GDPA_ACT_SOFTMAX = 5
} gdpa_act;

typedef enum {
    GDPA_MASK_NONE = 0,            /* every (query, key) pair of a sample */
    GDPA_MASK_CAUSAL_WINDOW = 1    /* i - window < j <= i */
} gdpa_mask;

/* Tile-to-SM assignment (GDPA page, zigzag scheduling paragraph and diagram).
 *
 * ZIGZAG costs a forward tile by its key blocks and a backward unit by its
 * query tiles.  ZIGZAG_TIMED deals the same way (stable sort by cost, snake
 * order) but costs a backward unit with an integer time model, in units of
 * 50 ns, fitted to the tensor-core backward's measured times on GB300:
 *   36 + 22 nkv16 / 128 + sum over its query tiles of
 *   (40 + 34 nq32 / 128 + 24 nkv16 / 128)          (a zero unit: 1)
 * where nq32 is a query tile's rows rounded up to 32 and nkv16 the unit's
 * keys rounded up to 16 (integer divisions): a unit carries a fixed cost
 * (loading its K and V, storing dK and dV) and each query tile a cost that
 * grows with the keys, which counting query tiles alone does not see.
 * Forward tiles keep the key-block cost: equal-cost tiles keep their
 * enumeration order, so the tiles of one sample run at the same time and
 * share its K and V in L2 (costing them by time scattered them and was
 * measured slower). */
typedef enum {
    GDPA_SCHED_ZIGZAG = 0,       /* sort by cost, deal in snake order */
    GDPA_SCHED_ROUND_ROBIN = 1,  /* enumeration order, tile r to SM r % S */
    GDPA_SCHED_ZIGZAG_TIMED = 2  /* sort by the time model, deal in snake order */
} gdpa_sched;

typedef enum { GDPA_BF16 = 0, GDPA_F32 = 1 } gdpa_dtype;

/* Which kernels a plan launches.  AUTO: tensor-core (tcgen05) kernels for
 * bf16 with d in {64, 128}, CUDA-core kernels otherwise (float32 always
 * runs on CUDA cores so that it keeps full float32 products). */
typedef enum { GDPA_KERNEL_AUTO = 0, GDPA_KERNEL_TCGEN05 = 1, GDPA_KERNEL_SIMT = 2 } gdpa_kernel;

typedef struct gdpa_plan_s* gdpa_plan;   /* opaque, owned by the library */

/* Tile sizes of every plan: 128 query rows x 128 key rows. */
#define GDPA_BLOCK_M 128
#define GDPA_BLOCK_N 128
/* max_kv_blocks_per_tile value that lets the planner choose the key split */
#define GDPA_KV_SPLIT_AUTO (-1)

/*
 * Build the tile plan of a jagged batch on the host and upload it on
 * `stream` (GDPA page: the CPU precomputes the valid tiles from the jagged
 * lengths and assigns them to SMs in zigzag order).
 *
 *   q_off_host, kv_off_host  host int32 [B+1]; read only during this call.
 *   B >= 0 samples; H >= 1 heads; d = head dim (a multiple of 4, <= 128;
 *     the tcgen05 kernels need 64 or 128).
 *   mask, window             window >= 1 when mask is CAUSAL_WINDOW.
 *   sched                    dealing policy.
 *   num_sms                  S, the number of persistent CTAs (0 = the
 *                            current device's SM count).
 *   max_kv_blocks_per_tile   0 = one forward tile per query tile; > 0 cuts
 *                            longer key ranges into chunks of at most this
 *                            many 128-row key blocks, each its own tile
 *                            (spreads few-query, many-key samples over more
 *                            SMs).  The forward of such a plan adds float32
 *                            partial sums of O into a plan-owned workspace
 *                            ([Tq][H][d] float, allocated on first use and
 *                            cleared on every call) and rounds it into O with
 *                            a second kernel: on the tensor cores for d =
 *                            128, on the CUDA-core kernels otherwise (float32
 *                            inputs, other head dims; with GDPA_KERNEL_AUTO
 *                            also bf16 d = 64, which GDPA_KERNEL_TCGEN05
 *                            refuses with UNSUPPORTED).  The softmax
 *                            variant's forward refuses split plans
 *                            (UNSUPPORTED: its chunks would need a max/sum
 *                            merge).  The backward takes split plans on
 *                            every path (the CUDA-core dQ kernel then adds
 *                            each chunk's share atomically into a cleared
 *                            dQ).
 *                            GDPA_KV_SPLIT_AUTO (-1): the planner picks
 *                            chunks of 2 key blocks when some query tile
 *                            reaches 8 or more key blocks (the fastest
 *                            setting measured for 32-query samples against
 *                            up to 8192 keys), else no split; such a plan
 *                            may therefore be split, with the limits above.
 *                            Values below -1 are INVALID_ARG.
 *   out                      receives the plan; *out is NULL on failure.
 *
 * Forward tiles: one per (sample, head, 128-row query tile), with the range
 * of 128-row key blocks that hold a valid pair (a zero tile, kb0 = kb1 = 0,
 * when none does); cost = number of key blocks.  Backward units: one per
 * (sample, head, key block), with the range of query tiles that hold a valid
 * pair; cost = number of query tiles.  Zigzag: stable sort by cost
 * descending; the r-th tile goes to SM r % S on even rounds r / S and to
 * S - 1 - r % S on odd rounds.
 *
 * Errors: INVALID_ARG for NULL pointers, negative sizes, offsets that do not
 * start at 0 or decrease, window < 1 with the window mask; UNSUPPORTED for
 * d > 128 or d % 4 != 0; ALLOC / CUDA for allocation or copy failures.
 *
 * The plan's device buffers come from the stream-ordered allocator and its
 * upload is enqueued on `stream`; the call does not wait for it.  Launches on
 * the plan, on any stream, are ordered after the upload by an event.
 *
 * Concurrency: calls on one plan may be enqueued on different streams only
 * if their GPU work does not overlap when they use a plan-owned workspace
 * (the forward of a key-split plan, the softmax variant's backward) or the
 * plan's device error word; use one plan per concurrent stream otherwise.
 */
gdpa_status gdpa_plan_create(const int32_t* q_off_host, const int32_t* kv_off_host, int B,
                             int H, int d, gdpa_mask mask, int window, gdpa_sched sched,
                             int num_sms, int max_kv_blocks_per_tile, void* stream,
                             gdpa_plan* out);

/*
 * Same planning on the host only, with no device and no upload: num_sms must
 * be > 0.  The plan can be exported and destroyed but not launched
 * (gdpa_fwd / gdpa_bwd return INVALID_ARG).  Useful to inspect a plan on a
 * machine without a GPU.
 */
gdpa_status gdpa_plan_create_host(const int32_t* q_off_host, const int32_t* kv_off_host, int B,
                                  int H, int d, gdpa_mask mask, int window, gdpa_sched sched,
                                  int num_sms, int max_kv_blocks_per_tile, gdpa_plan* out);

/* Number of forward tiles, backward units and SMs (S) of a plan. */
gdpa_status gdpa_plan_sizes(gdpa_plan plan, int64_t* n_fwd, int64_t* n_bwd, int* num_sms);

/*
 * Copy the forward tile list to host memory in queue order (SM 0's queue
 * first).  tiles_out: int32 [cap][6] rows (b, h, m, kb0, kb1, sm);
 * seg_start_out: int32 [S+1] first row of each SM's queue (may be NULL).
 * Returns INVALID_ARG if cap is smaller than the tile count (*n_out still
 * receives the count).
 */
gdpa_status gdpa_plan_export(gdpa_plan plan, int32_t* tiles_out, int64_t cap, int64_t* n_out,
                             int32_t* seg_start_out);

/*
 * Same for the backward units: int32 [cap][7] rows (b, h, j, m0, m1, flags,
 * sm); flags bit 0 = this sample's dQ is accumulated with atomic adds.
 * *zero_dq_out (may be NULL) is 1 when gdpa_bwd clears dQ before its kernels.
 */
gdpa_status gdpa_plan_export_bwd(gdpa_plan plan, int32_t* units_out, int64_t cap,
                                 int64_t* n_out, int32_t* seg_start_out, int* zero_dq_out);

/*
 * Deal the samples of one batch to num_ranks GPUs (one process per GPU), so
 * that each rank runs the samples given to it as a batch of its own with no
 * exchange (samples and heads are independent; GDPA page, the jagged-input
 * and zigzag-scheduling paragraph, applied one level up; GEM page "GEM
 * 트레이닝: Meta가 LLM 규모의 광고 파운데이션 모델 효율성을 두 배로 높인 방법",
 * techlist.io, section on scaling to thousands of GPUs: variable lengths
 * make stragglers).  A sample's work is H times the key blocks of its
 * 128-row query tiles (with the causal window: of the window's hull), the
 * forward tile cost of gdpa_plan_create summed over the sample.  Samples are
 * sorted by work, descending and stable, and dealt in snake order: the r-th
 * goes to rank r % R on even rounds r / R and R - 1 - r % R on odd ones.
 *
 *   q_off, kv_off  host int32 [B+1] offsets (as gdpa_plan_create).
 *   rank_out       host int32 [B]: the rank of each sample.
 *   work_out       host int64 [num_ranks] (may be NULL): each rank's work.
 *
 * INVALID_ARG for NULL pointers, B < 0, H < 1, num_ranks < 1, bad offsets
 * or a window < 1 with the window mask.  Host only; no device is touched.
 */
gdpa_status gdpa_shard_batch(const int32_t* q_off, const int32_t* kv_off, int B, int H,
                             gdpa_mask mask, int window, int num_ranks, int32_t* rank_out,
                             int64_t* work_out);

/* Choose the kernel family (default AUTO); INVALID_ARG for unknown values. */
gdpa_status gdpa_plan_set_kernel(gdpa_plan plan, gdpa_kernel kernel);

/*
 * Shared-query mode, for pooling attention (PMA: a fixed set of learned seed
 * queries attends to each sample's history, compressing it into short
 * queries against long keys; GEM page "GEM 트레이닝: Meta가 LLM 규모의 광고
 * 파운데이션 모델 효율성을 두 배로 높인 방법", techlist.io, section on the
 * asymmetric attention shapes; the GDPA page's diagram of self-attention,
 * PMA and pFFN sharing one kernel).  n_seeds > 0: the q of gdpa_fwd,
 * gdpa_bwd, gdpa_softmax_fwd and gdpa_softmax_bwd on this plan is a
 * [n_seeds][H][d] tensor of seed rows shared by every sample, sample b's
 * queries being seeds 0 .. Lq_b - 1, so Q is never replicated per sample;
 * O, dO and lse keep their per-token layout.  The backward's dq is then
 * [n_seeds][H][d] float32, each seed's gradient summed over the samples
 * (cleared by the call, then accumulated with atomic adds).  INVALID_ARG if
 * some sample has more than n_seeds queries.  Every kernel path supports
 * it.  n_seeds = 0 restores per-token queries.
 * gdpa_fwd_noalloc has no such mode.
 */
gdpa_status gdpa_plan_set_shared_q(gdpa_plan plan, int n_seeds);

/*
 * Fused RMSNorm prologue (the GDPA page: RMSNorm keeps the activation's
 * inputs in range, the caption under its Taylor code; GEM page, section on
 * why GPU utilisation is hard for recommendation models: normalisation is a
 * memory-bound pass of its own).  gain > 0: the q and k given to gdpa_fwd,
 * gdpa_bwd, gdpa_softmax_fwd and gdpa_softmax_bwd on this plan are the raw
 * rows, and every (token, head) row of Q and K is normalised inside the
 * kernels,
 *     y = gain x / sqrt(mean(x^2) + eps),
 * before it enters the attention; V is used as given.  The backward's dq and
 * dk are then the gradients with respect to the raw rows,
 *     dL/dx = (gain / r) (dy - x (x . dy) / (d r^2)),  r = sqrt(mean(x^2) + eps).
 * Each launch first normalises the keys in one pass over K (c = gain / r of
 * every key row into a plan-owned [H][Tkv + 128] float workspace, the rows
 * c k rounded to bf16 into a plan-owned [Tkv][H][d] workspace; both
 * allocated on first use and kept until gdpa_plan_destroy); the attention
 * kernels read those keys, compute each query row's c from its tile and
 * fold it into alpha (x = alpha c_i q_i . k_hat_j), and apply the norm's
 * Jacobian to dq and dk as they drain them.  The queries are never written
 * normalised.  Tensor-core kernels only (bf16, d = 64 or 128): the CUDA-core path
 * returns UNSUPPORTED while it is on; gdpa_fwd_noalloc has no such mode.
 * gain = 0 turns it off.  INVALID_ARG for a negative or NaN gain or eps, or
 * eps = 0 with gain > 0 (an all-zero row would divide by zero).
 */
gdpa_status gdpa_plan_set_qk_norm(gdpa_plan plan, float gain, float eps);

/* Record per-CTA start/end times (%globaltimer, ns) and SM ids on the next
 * launches (enable != 0), readable with gdpa_sm_times. */
gdpa_status gdpa_plan_set_timing(gdpa_plan plan, int enable);

/*
 * Forward: O = act(alpha Q K^T) V per sample and head (GDPA page, summary).
 * q, k, v, o: device pointers, layouts above, element type `dtype`.  Every
 * row of O is written (rows with no valid key become zero).  Enqueued on
 * `stream`; returns INVALID_ARG / UNSUPPORTED before any launch when the
 * arguments do not fit the plan.
 */
gdpa_status gdpa_fwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                     const void* v, void* o, float alpha, gdpa_act act, void* stream);

/*
 * Backward: given dO, the float32 gradients
 *   dV_j = sum_i act(x_ij) dO_i,  dQ_i = alpha sum_j g_ij K_j,
 *   dK_j = alpha sum_i g_ij Q_i,  g_ij = (dO_i . V_j) act'(x_ij),
 * with x_ij = alpha q_i . k_j over valid pairs.  dq, dk, dv are device
 * float32 buffers that this call overwrites entirely (no prior clearing
 * needed).  Enqueued on `stream`.
 */
gdpa_status gdpa_bwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                     const void* v, const void* d_o, float* dq, float* dk, float* dv,
                     float alpha, gdpa_act act, void* stream);

/*
 * Wait for this plan's launches (on every stream they were enqueued on) and
 * for `stream`, and report device-side failures of the plan's launches since
 * the last check: TIMEOUT if a kernel abandoned a barrier wait (its outputs
 * are then incomplete; the kernel has returned and the device stays usable),
 * DEVICE for other flagged errors, CUDA for an asynchronous CUDA error.
 * Clears the flags.
 */
gdpa_status gdpa_check(gdpa_plan plan, void* stream);

/*
 * Where the last failure that gdpa_check reported for this plan came from
 * (host-side copy, no device access): detail = int32 [4], the device error
 * code (1 = an abandoned barrier wait), the site (a number naming the wait
 * in the kernel source: 1-16 forward, 21-50 backward), the CTA that gave up
 * first, and a code-specific word.  All zero if gdpa_check has reported no
 * failure for this plan.  Errors: INVALID_ARG for a NULL plan or detail.
 */
gdpa_status gdpa_error_detail(gdpa_plan plan, int32_t* detail);

/*
 * Per-CTA timing of the last timed tensor-core launch (which = 0 forward,
 * 1 backward): start_end: uint64 [S][2] globaltimer ns; smid: int32 [S].
 * Waits for this plan's launches only (not the whole device) and reads on the
 * stream of the timed launch, which must still exist.  INVALID_ARG if timing
 * was not enabled or nothing was recorded.
 */
gdpa_status gdpa_sm_times(gdpa_plan plan, int which, uint64_t* start_end, int32_t* smid);

/* Number of kernel launches this plan has issued since creation. */
int64_t gdpa_plan_launches(gdpa_plan plan);

/* Frees the plan (NULL is a no-op).  Does not wait on the host: the plan's
 * device buffers are returned to the stream-ordered allocator on a private
 * stream that first waits (on the device) for every launch made on the plan,
 * so work still queued may keep reading them until it has run.  Other work
 * on the device is not waited for. */
void gdpa_plan_destroy(gdpa_plan plan);

/*
 * Failure-path test hook (the pages have no counterpart; it exists so that
 * tests can exercise the kernels' bounded waits without a GPU fault).
 *
 *   limit_us   > 0: the tensor-core kernels' barrier waits on this plan give
 *              up after limit_us microseconds instead of 2 s; 0 restores the
 *              default.
 *   stall      != 0: on the next tensor-core launches, CTA 0's loader skips
 *              its first query-tile load, so a wait for it expires: the
 *              kernel records a timeout, every role unwinds (waits, bounded,
 *              for its own copies and MMAs in flight, frees TMEM) and returns.
 *              gdpa_check then reports GDPA_ERR_TIMEOUT and the outputs of
 *              that launch are incomplete.  0 restores normal launches.
 *
 * INVALID_ARG for a NULL plan or limit_us < 0.  Host-side only.
 */
gdpa_status gdpa_plan_set_wait_test(gdpa_plan plan, int limit_us, int stall);

/*
 * Forward pass that allocates nothing (the GDPA page has no counterpart of
 * this call; it exists for callers of this library).
 *
 * Some callers cannot call cudaMalloc: code running inside a custom device
 * allocator or memory pool (which would recurse into itself), plugins that
 * are handed one fixed device arena, and processes that must reserve all of
 * their device memory up front.  They cannot create a gdpa_plan, whose tile
 * queue and error word are allocated on the device.  This call computes the same
 * O = act(alpha Q K^T) V as gdpa_fwd with a zigzag plan over the current
 * device's SMs, on the tensor-core kernel (bf16, d = 64 or 128), without
 * allocating: the plan is built in static host buffers and its tile queue
 * is uploaded into a static device array of GDPA_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library keeps until the process exits.  The caller
 * still owns q, k, v, o (device, layout as above) and the stream.
 *
 *   - Returns GDPA_ERR_SCRATCH_LIMIT, before any work, when the batch has
 *     more than GDPA_NOALLOC_MAX_TILES forward tiles (one per sample, head
 *     and 128-row query tile); UNSUPPORTED for other head dims; INVALID_ARG
 *     for bad offsets or pointers.
 *   - The first call on a device sets up that device (looks up the array's
 *     device address, creates one event); make it before any stream capture.
 *   - Every call shares the one array and overwrites it: calls whose work
 *     overlaps on the GPU (e.g. on two streams) race.  Host threads are
 *     serialised internally.  A call waits for the previous call's upload
 *     (not its kernel) before reusing the host staging buffers.
 *   - The kernel's barrier-timeout word lives in the array and is cleared by
 *     every call; it is not reported (use a gdpa_plan and gdpa_check for
 *     that).
 */
#define GDPA_NOALLOC_MAX_TILES 32768
#define GDPA_NOALLOC_SCRATCH_BYTES 1056768
gdpa_status gdpa_fwd_noalloc(const int32_t* q_off_host, const int32_t* kv_off_host, int B, int H,
                             int d, gdpa_mask mask, int window, const void* q, const void* k,
                             const void* v, void* o, float alpha, gdpa_act act, void* stream);

/* Softmax variant (Jagged Flash Attention) with its row statistics.
 *
 * As gdpa_fwd with act = GDPA_ACT_SOFTMAX, and also writes
 *   lse[t][h] = log sum_j exp(alpha q_t.k_j)   (natural log; over the row's
 *               valid keys; -inf for a row without one),
 * device float32 [Tq][H] (caller-owned; required when Tq > 0), which the
 * backward needs.  Same dtypes, shapes, errors and kernels as gdpa_fwd.
 */
gdpa_status gdpa_softmax_fwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                             const void* v, void* o, float* lse, float alpha, void* stream);

/* Gradients of the softmax variant.
 *
 * With P_tj = exp(alpha q_t.k_j - lse_t) over the valid pairs, dP_tj =
 * dO_t.V_j and D_t = dO_t.O_t:
 *   dV_j = sum_t P_tj dO_t,   dS_tj = P_tj (dP_tj - D_t),
 *   dQ_t = alpha sum_j dS_tj K_j,   dK_j = alpha sum_t dS_tj Q_t.
 * o and lse are gdpa_softmax_fwd's outputs for the same q, k, v, plan and
 * alpha; d_o has o's dtype and shape; dq, dk, dv as gdpa_bwd (float32, fully
 * written).  D goes to a [Tq][H] float32 workspace the plan allocates on the
 * first call (ALLOC on failure) and keeps until gdpa_plan_destroy.  Errors
 * as gdpa_bwd, plus INVALID_ARG for a NULL or misaligned o or a NULL lse.
 */
gdpa_status gdpa_softmax_bwd(gdpa_plan plan, gdpa_dtype dtype, const void* q, const void* k,
                             const void* v, const void* o, const void* d_o, const float* lse,
                             float* dq, float* dk, float* dv, float alpha, void* stream);

/*
 * MXFP8 encoding of Q and K.  The GEM page ("GEM 트레이닝: Meta가 LLM 규모의
 * 광고 파운데이션 모델 효율성을 두 배로 높인 방법", techlist.io, section "GPU
 * 연산 효율을 높인 맞춤형 커널과 정밀도") trains attention in mixed precision
 * that includes MXFP8; the format is OCP Microscaling: blocks of 32
 * consecutive values share one power-of-two scale 2^E (E8M0), and each value
 * is an FP8 E4M3 element (bias 7, largest finite 448, subnormals, no
 * infinities).  For a block whose largest magnitude is a > 0,
 * E = floor(log2 a) - 8, clamped to [-127, 127]; an all-zero block has
 * E = -127.  Element = x / 2^E rounded to the nearest E4M3 value, ties to
 * the even mantissa, saturated at +-448.  The block stands for element * 2^E.
 *
 * Storage: `elements` holds one E4M3 code per value in the value's position
 * (uint8, 16-byte aligned device memory); `scales` holds E + 127 as one byte
 * per block, block i covering values [32 i, 32 i + 32).  For a [T][H][d]
 * tensor (d a multiple of 32) that is elements [T][H][d] and scales
 * [T][H][d / 32].
 */

/* x: n bf16 values (device, 16-byte aligned) -> elements [n], scales [n / 32].
 * INVALID_ARG for n < 0, n not a multiple of 32, NULL or misaligned
 * pointers; CUDA if the launch fails.  Asynchronous on `stream`. */
gdpa_status gdpa_mx_quantise(const void* x, int64_t n, uint8_t* elements, uint8_t* scales,
                             void* stream);

/* elements [n], scales [n / 32] -> x: n bf16 values, each element * 2^E
 * rounded to bf16 (exact unless the value is below bf16's smallest
 * subnormal).  Errors and stream as gdpa_mx_quantise. */
gdpa_status gdpa_mx_dequantise(const uint8_t* elements, const uint8_t* scales, int64_t n, void* x,
                               void* stream);

/*
 * GDPA with Q and K given in MXFP8 (blocks along d; d = 32, 64 or 128), V in
 * bf16: the forward and backward of gdpa_fwd / gdpa_bwd (and the softmax
 * variant's forward with act = GDPA_ACT_SOFTMAX) on the values the MXFP8
 * tensors stand for.  The gradients dq, dk are with respect to those values
 * (float32, as gdpa_bwd).  q_el / q_sc hold Q's rows (Tq rows, or the seed
 * rows in shared-query mode), k_el / k_sc K's Tkv rows.  The call expands Q
 * and K to bf16 in a plan-owned device workspace ((Q rows + Tkv) H d bf16,
 * allocated on the stream on first use, kept until gdpa_plan_destroy; ALLOC
 * on failure) and runs the bf16 kernels the plan selects; the fused
 * RMSNorm, when on, normalises the expanded rows.  With all four of q_el,
 * q_sc, k_el, k_sc NULL the call reuses the expansion the plan's previous
 * gdpa_fwd_mx / gdpa_bwd_mx made (e.g. the backward of a forward on the same
 * Q and K, saving the second expansion); the caller orders the two calls
 * (same stream, or an event) and INVALID_ARG is returned if there is no
 * such expansion.  Errors as gdpa_fwd / gdpa_bwd, plus INVALID_ARG for NULL
 * or misaligned element pointers (other than the reuse form) or
 * d % 32 != 0.
 */
gdpa_status gdpa_fwd_mx(gdpa_plan plan, const uint8_t* q_el, const uint8_t* q_sc,
                        const uint8_t* k_el, const uint8_t* k_sc, const void* v, void* o,
                        float alpha, gdpa_act act, void* stream);
gdpa_status gdpa_bwd_mx(gdpa_plan plan, const uint8_t* q_el, const uint8_t* q_sc,
                        const uint8_t* k_el, const uint8_t* k_sc, const void* v, const void* d_o,
                        float* dq, float* dk, float* dv, float alpha, gdpa_act act, void* stream);

/* Activation test hook.
 *
 * Evaluates act(x) and act'(x) element-wise with the same device functions
 * the kernels use: fast == 1 selects the tensor-core kernels' flavour (the
 * one P and dS are computed with on the bf16 path) one element at a time,
 * fast == 2 the same flavour in the two-at-a-time (f32x2) form the
 * tensor-core kernels evaluate it in (elements 2k and 2k + 1 together; an
 * odd last element with a copy of itself), fast == 0 the CUDA-core float32
 * path's.  Forms 1 and 2 are meant to agree bit for bit.  The activations are those of the GDPA page ("범용 내적
 * 어텐션(GDPA)", aitrends.kr: GELU, SiLU and the Taylor-6 GELU replacing
 * softmax), plus identity.  It exists so that tests can check those
 * functions against reference values directly.
 *
 *   x, y, dy   device float32 arrays of n elements (caller-owned); y = act(x),
 *              dy = act'(x).
 *   n          >= 0; n == 0 does nothing.
 *   stream     cudaStream_t; asynchronous.
 *
 * Errors: INVALID_ARG for an unknown act, fast outside 0..2, n < 0 or NULL
 * arrays; CUDA if the launch fails.
 */
gdpa_status gdpa_act_eval(gdpa_act act, int fast, const float* x, float* y, float* dy, int64_t n,
                          void* stream);

const char* gdpa_status_str(gdpa_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDPA_H */
