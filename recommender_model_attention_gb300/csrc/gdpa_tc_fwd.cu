// Persistent tcgen05 GDPA forward kernel (bf16 in, fp32 accumulate, bf16 out).
//
// GDPA ("범용 내적 어텐션(GDPA)", aitrends.kr) computes O = act(alpha Q K^T) V
// per sample with the softmax replaced by an element-wise activation; the
// page's design notes drop the softmax correction (no running max, row sum
// or rescaling of O), pipeline across the outer loop for short K/V, flatten
// the (query tile, key block) loops, and walk a host-planned tile list dealt
// to SMs in zigzag order.  This kernel is the GB300 rendering of that:
//
//  * grid = one CTA per planned SM queue; CTA s walks tiles seg[s]..seg[s+1].
//  * warp 0 (one lane): TMA producer.  Q tile [128 x d] per tile through a
//    3-stage ring, K and V blocks [128 x d] per (tile, key block) item
//    through 2-stage rings; a K stage is handed back once its item's S has
//    read it and a V stage once its P V has, and the producer loads K one
//    item ahead of V, so the next items' scores never wait for a P V.  The
//    next tile's Q is prefetched into L2 while its stage is still busy.
//  * warps 1 and 18: tcgen05.mma issuers (the whole warp runs the issue
//    code, one elected lane issues).  Warp 1 issues S = Q K^T of each tile's
//    first item as soon as its Q and K are loaded and its slot's previous
//    P V is done; warp 18 issues P V of every item as soon as its P is in
//    TMEM, then S of the tile's next item.  So the tensor core computes the
//    next tile's scores while this tile's activation runs, and a tile's P V
//    never waits for the next tile's loads (software pipelining across tile
//    boundaries on one flattened loop).  Within an item, S and P V run in
//    two key halves with their own barriers: the activation starts on keys
//    [0, 64) while the tensor core computes keys [64, 128), and their P V
//    while the activation finishes the rest.
//  * warps 2-17: four activation/epilogue warpgroups.  Tiles alternate
//    between two slots, each with its own TMEM S (128 columns) and O (128
//    columns) accumulators, and two warpgroups share a slot: part h takes
//    the 16-column key steps h, h + 2, ... of S (the softmax variant the
//    32-column chunks h and h + 2) and the O columns [h d/2, (h + 1) d/2).
//    They read S with tcgen05.ld, apply alpha, the activation and the
//    jagged / window mask (masked pairs become exactly 0 after the
//    activation), and write P as packed bf16 into the first half of each
//    S step (chunk) they have read (tcgen05.st); P V then takes P
//    straight from TMEM (A operand in TMEM, one address per K = 16 step).
//    After the last key block they read O from TMEM and stage it (bf16) in
//    the tile's consumed Q buffer; each warp writes its 32 rows with one TMA
//    bulk store (the warp at a tile's ragged end with plain stores of its
//    valid rows).  Zero tiles (no valid key) are written as zeros directly.
//  * O accumulates P V over key blocks with no rescaling.
//  * Every barrier wait is bounded; a timeout sets the plan's error word and
//    the CTA unwinds (waits for its TMA loads and MMAs, frees TMEM, returns).
#include <algorithm>
#include <cuda_bf16.h>

#include "act.cuh"
#include "tc_common.cuh"
#include "tc_drain.cuh"

namespace gdpa {
namespace {

using namespace tc;

constexpr int kNumWG = 2;                       // tile slots (TMEM S/P + O each)
constexpr int kParts = 2;                       // warpgroups sharing one slot
// producer, S issuer, warpgroups, P V issuer
constexpr int kThreads = 64 + 128 * kNumWG * kParts + 32;
constexpr int kPvWarp = 2 + 4 * kNumWG * kParts;
constexpr int kHalfBytes = 128 * 128;           // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kTmemCols = 512;

template <int D>
struct FwdCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kNQ = 3;
    static constexpr int kNKV = 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kNQ * kTileBytes;
    static constexpr int kOffV = kOffK + kNKV * kTileBytes;
    static constexpr int kOffBar = kOffV + kNKV * kTileBytes;
    // q_full, q_empty, k_full, v_full, k_empty, v_empty,
    // s_full, p_full, o_full, o_free, stage (per warpgroup), mma_done
    static constexpr int kBarQFull = 0;
    static constexpr int kBarQEmpty = kBarQFull + kNQ;
    static constexpr int kBarKFull = kBarQEmpty + kNQ;
    static constexpr int kBarVFull = kBarKFull + kNKV;
    static constexpr int kBarKEmpty = kBarVFull + kNKV;   // the item's S has read K
    static constexpr int kBarVEmpty = kBarKEmpty + kNKV;  // the item's P V has read V
    static constexpr int kBarSFull = kBarVEmpty + kNKV;    // per slot and key half
    static constexpr int kBarPFull = kBarSFull + 2 * kNumWG;   // per slot and key half
    static constexpr int kBarOFull = kBarPFull + 2 * kNumWG;
    static constexpr int kBarOFree = kBarOFull + kNumWG;
    static constexpr int kBarStage = kBarOFree + kNumWG;             // per warpgroup
    static constexpr int kBarMmaDone = kBarStage + kNumWG * kParts;   // S issuer, P V issuer
    static constexpr int kBarXchg = kBarMmaDone + 2;   // per slot: softmax part exchange
    static constexpr int kNumBars = kBarXchg + kNumWG;
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
};

struct FwdParams {
    const FwdTile* tiles;
    const int32_t* seg;
    __nv_bfloat16* O;
    float* lse;   // softmax variant: row log-sum-exp [Tq][H] out, or NULL
    float* W;     // key-split plans: float32 [Tq][H][D] partial-sum target, or NULL
    int shared_q; // Q holds seed rows shared by all samples: a tile's Q rows
                  // start at its position in the sample, not at its token row
    int H;
    float alpha;
    int mask;
    int window;
    int32_t* err;
    unsigned long long* times;
    int32_t* smid;
    int timing;
    uint64_t wait_ns;   // bounded-wait limit
    int stall;          // test hook: CTA 0 skips its first Q load
    // fused RMSNorm (qk_gain > 0): the keys arrive normalised; each query
    // row's scale g / rms is computed from its tile and folded into alpha
    float qk_gain, qk_eps;
};

// Bounded wait for a shared-memory counter that other warps raise to reach
// `v` (false, with the error recorded, if it does not in time or the CTA is
// aborting).  Every lane of the calling warp reads it.
__device__ __forceinline__ bool counter_wait(const volatile int* c, int v, const Abort& ab,
                                             int32_t where) {
    if (*c >= v) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1; *c < v; ++it) {
        if ((it & 31u) == 0) {
            if (*ab.flag) return false;
            if (globaltimer() - t0 > ab.limit_ns || it > kWaitLimitIters) {
                raise_error(ab, kDevTimeout, where);
                return false;
            }
        }
    }
    return true;
}

// Hint: bring the line holding p into L1 (no register result, no wait).
__device__ __forceinline__ void prefetch_l1(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ FwdTile load_tile(const FwdTile* p) {
    const int4* q = reinterpret_cast<const int4*>(p);
    const int4 a = __ldg(q), b = __ldg(q + 1);
    FwdTile t;
    t.qt0 = a.x; t.nq = a.y; t.kvt0 = a.z; t.lkv = a.w;
    t.h = b.x; t.kb0 = b.y; t.kb1 = b.z; t.i0 = b.w;
    return t;
}

// Items of a tile: one per key block.  The softmax variant makes two passes
// over a tile with more than one key block: the row maxima first (S only),
// then the weights and P V; with one key block both come from one S.
template <bool SM>
__device__ __forceinline__ int tile_items(const FwdTile& t) {
    const int nb = t.kb1 - t.kb0;
    return (SM && nb > 1) ? 2 * nb : nb;
}

template <bool SM>
__device__ __forceinline__ int item_block(const FwdTile& t, int it) {
    const int nb = t.kb1 - t.kb0;
    return t.kb0 + ((SM && nb > 1) ? it % nb : it);
}

// does the item carry a P V product (and, for the softmax variant, weights)?
template <bool SM>
__device__ __forceinline__ bool item_pv(const FwdTile& t, int it) {
    const int nb = t.kb1 - t.kb0;
    return !SM || nb == 1 || it >= nb;
}

template <int D, bool SM>
__device__ void fwd_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                             const FwdParams& prm, uint8_t* smem, uint64_t* bars, int seg0,
                             int seg1, const Abort& ab) {
    using C = FwdCfg<D>;
    const uint64_t pol_q = policy_evict_first();
    const uint64_t pol_kv = policy_evict_last();
    int32_t q_armed[C::kNQ], k_armed[C::kNKV], v_armed[C::kNKV];
    for (int s = 0; s < C::kNQ; ++s) q_armed[s] = -1;
    for (int s = 0; s < C::kNKV; ++s) k_armed[s] = v_armed[s] = -1;
    // K runs ahead of V: a K stage is free once its item's S has read it, a
    // V stage only once its P V has, so within a tile item i's K goes in as
    // soon as item i - kNKV's S is done, and item i - 1's V after it; a
    // tile's last V goes in before the next tile's Q (whose stage waits for
    // an epilogue).  Either way item i's V precedes item i + 2's K.
    int pend_y = -1, pend_h = 0;   // the item whose V is still to load
    uint32_t pend_i = 0;
    auto load_v = [&]() -> bool {
        const uint32_t vs = pend_i % C::kNKV, vph = (pend_i / C::kNKV) & 1;
        if (!mbar_wait(&bars[C::kBarVEmpty + vs], vph ^ 1, ab, 2)) return false;
        mbar_arrive_expect_tx(&bars[C::kBarVFull + vs], C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
            tma_load_2d(tmV, &bars[C::kBarVFull + vs],
                        smem + C::kOffV + vs * C::kTileBytes + hf * kHalfBytes,
                        pend_h * D + hf * 64, pend_y, pol_kv);
        v_armed[vs] = (int32_t)vph;
        pend_y = -1;
        return true;
    };
    uint32_t a = 0, i = 0;
    for (int t = seg0; t < seg1; ++t) {
        // (the descriptor line 4 tiles ahead, so that this warp's next
        // descriptor loads hit in L1)
        if (t + 4 < seg1) prefetch_l1(prm.tiles + t + 4);
        const FwdTile tile = load_tile(prm.tiles + t);
        if (tile.kb1 <= tile.kb0) continue;
        if (pend_y >= 0 && !load_v()) goto unwind;   // the previous tile's last V
        const uint32_t qs = a % C::kNQ, qph = (a / C::kNQ) & 1;
        if (!mbar_wait(&bars[C::kBarQEmpty + qs], qph ^ 1, ab, 1)) goto unwind;
        // failure-path test hook: CTA 0 never loads its first Q tile, so the
        // S issuer's bounded wait for it expires
        if (!(prm.stall && blockIdx.x == 0 && a == 0)) {
            mbar_arrive_expect_tx(&bars[C::kBarQFull + qs], C::kTileBytes);
            q_armed[qs] = (int32_t)qph;
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_2d(tmQ, &bars[C::kBarQFull + qs],
                            smem + C::kOffQ + qs * C::kTileBytes + hf * kHalfBytes,
                            tile.h * D + hf * 64, prm.shared_q ? tile.i0 : tile.qt0, pol_q);
        }
        const int nit = tile_items<SM>(tile);
        for (int it = 0; it < nit; ++it, ++i) {
            const uint32_t ks = i % C::kNKV, kph = (i / C::kNKV) & 1;
            if (!mbar_wait(&bars[C::kBarKEmpty + ks], kph ^ 1, ab, 2)) goto unwind;
            const int y = tile.kvt0 + item_block<SM>(tile, it) * kBN;
            mbar_arrive_expect_tx(&bars[C::kBarKFull + ks], C::kTileBytes);
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_2d(tmK, &bars[C::kBarKFull + ks],
                            smem + C::kOffK + ks * C::kTileBytes + hf * kHalfBytes,
                            tile.h * D + hf * 64, y, pol_kv);
            k_armed[ks] = (int32_t)kph;
            if (pend_y >= 0 && !load_v()) goto unwind;   // the item before's V
            pend_y = y;
            pend_h = tile.h;
            pend_i = i;
        }
        // the next tile's Q box into L2 once this tile's loads are issued:
        // its ring load waits for an epilogue to free a stage, and then
        // finds Q in L2 instead of starting the HBM read (a shared Q is
        // read by every tile and stays in L2 anyway).  Prefetched as
        // evict-last, so that it is still there when the load (evict-first)
        // takes it.
        if (!prm.shared_q && t + 1 < seg1) {
            const FwdTile tn = load_tile(prm.tiles + t + 1);
            if (tn.kb1 > tn.kb0) {
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf)
                    tma_prefetch_2d(tmQ, tn.h * D + hf * 64, tn.qt0, pol_kv);
            }
        }
        ++a;
    }
    if (pend_y >= 0) load_v();
unwind:
    // never leave the CTA with a TMA write still in flight
    for (int s = 0; s < C::kNQ; ++s)
        if (q_armed[s] >= 0) mbar_wait_teardown(&bars[C::kBarQFull + s], (uint32_t)q_armed[s]);
    for (int s = 0; s < C::kNKV; ++s) {
        if (k_armed[s] >= 0) mbar_wait_teardown(&bars[C::kBarKFull + s], (uint32_t)k_armed[s]);
        if (v_armed[s] >= 0) mbar_wait_teardown(&bars[C::kBarVFull + s], (uint32_t)v_armed[s]);
    }
}

// S = Q K^T of one item into slot w's S columns (K-major Q and K tiles) in
// two key halves, [0, 64) and [64, 128), each N = its valid keys rounded up
// to 16 and each committing its own S-full, so that the activation starts
// on the first half while the tensor core computes the second.  An item of
// at most 64 keys has no second half: nothing is issued or committed for it,
// and no one waits for it (every role decides this from the tile alone).
template <int D>
__device__ __forceinline__ void issue_s(uint8_t* smem, uint64_t* bars, uint32_t tmem, uint32_t w,
                                        uint32_t qs, uint32_t ks, int nvalid) {
    using C = FwdCfg<D>;
    const uint32_t n16 = (uint32_t)((nvalid + 15) & ~15);
    const uint64_t qdesc = smem_desc_sw128(smem_u32(smem + C::kOffQ + qs * C::kTileBytes), 16, 1024);
    const uint64_t kdesc = smem_desc_sw128(smem_u32(smem + C::kOffK + ks * C::kTileBytes), 16, 1024);
    const uint32_t na = n16 < 64u ? n16 : 64u;
    const uint32_t idesc_a = idesc_bf16(128, na, false, false);
#pragma unroll
    for (int k = 0; k < D / 16; ++k)
        mma_ss(tmem + w * 256, qdesc + kmajor_step(k), kdesc + kmajor_step(k), idesc_a,
               k > 0 ? 1u : 0u);
    mma_commit(&bars[C::kBarSFull + 2 * w]);
    if (n16 > 64u) {
        // keys 64..127: K rows 64.. start 64 x 128 bytes into each 128-byte-
        // swizzled box (a whole number of 1024-byte swizzle atoms)
        const uint32_t idesc_b = idesc_bf16(128, n16 - 64u, false, false);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
            mma_ss(tmem + w * 256 + 64, qdesc + kmajor_step(k), kdesc + (8192 >> 4) + kmajor_step(k),
                   idesc_b, k > 0 ? 1u : 0u);
        mma_commit(&bars[C::kBarSFull + 2 * w + 1]);
    }
}

// S issuer (warp 1, the whole warp; one elected lane issues): S of each
// tile's first item, as soon as its Q and K are loaded and the slot's
// previous item has had its P V complete (its S columns hold that item's P;
// P V runs on another warp, whose commit of the item's V-empty arrival this
// waits for).  S of a tile's later items follows the P V of the item before
// it on the P V warp, in issue order.  Each S commits its K stage's
// K-empty arrival.  Its waits on barriers that other warps also consume are
// kept within one phase: a K-full only after the K kNKV items back has been
// seen to land (a shared counter the two MMA warps raise), and the slot's
// previous P V only while that V-empty phase is current.
template <int D, bool SM>
__device__ void fwd_mma_s(const FwdParams& prm, uint8_t* smem, uint64_t* bars, uint32_t tmem,
                          volatile int* k_seen, int seg0, int seg1, const Abort& ab) {
    const int lane = threadIdx.x & 31;
    using C = FwdCfg<D>;
    static_assert(kNumWG == 2, "slot bookkeeping below is written for two slots");
    int64_t last0 = -1, last1 = -1;   // each slot's last item so far
    uint32_t a = 0, i = 0;
    for (int t = seg0; t < seg1; ++t) {
        // (the descriptor line 4 tiles ahead, so that this warp's next
        // descriptor loads hit in L1)
        if (t + 4 < seg1) prefetch_l1(prm.tiles + t + 4);
        const FwdTile tile = load_tile(prm.tiles + t);
        if (tile.kb1 <= tile.kb0) continue;
        const uint32_t wg = a % kNumWG;
        const uint32_t qs = a % C::kNQ, qph = (a / C::kNQ) & 1;
        const uint32_t ks = i % C::kNKV, kph = (i / C::kNKV) & 1;
        int64_t& last = wg ? last1 : last0;
        // (the producer loads the V of every item before a tile's first
        // item ahead of that item's K, so once item i >= last + kNKV + 1
        // has its K, the V stage of `last` has been refilled, which took
        // its P V's completion: no wait, and its V-empty phase could be
        // stale.  For i <= last + kNKV the phase after `last`'s completion,
        // the P V of item last + kNKV, cannot have completed: that item is
        // this one or a later one, which needs this S.)
        if (last >= 0 && last + C::kNKV >= (int64_t)i) {
            const uint32_t ls = (uint32_t)(last % C::kNKV), lph = (uint32_t)((last / C::kNKV) & 1);
            if (!wg_wait(&bars[C::kBarVEmpty + ls], lph, ab, 13)) goto drain;
        }
        // K-full of this stage says "item i's K is in" only once the load of
        // item i - kNKV into it has been seen to land (by this warp or the
        // P V warp, which raise k_seen as they see each K-full)
        if (!__all_sync(0xffffffffu, counter_wait(k_seen, (int)i - C::kNKV, ab, 16)) ||
            !wg_wait(&bars[C::kBarQFull + qs], qph, ab, 3) ||
            !wg_wait(&bars[C::kBarKFull + ks], kph, ab, 4))
            goto drain;
        if (lane == 0) atomicMax((int*)k_seen, (int)i);
        tc_fence_after();
        issue_s<D>(smem, bars, tmem, wg, qs, ks, min(kBN, tile.lkv - tile.kb0 * kBN));
        mma_commit(&bars[C::kBarKEmpty + ks]);
        i += (uint32_t)tile_items<SM>(tile);
        last = (int64_t)i - 1;
        ++a;
    }
drain:
    // all MMAs issued by this warp complete before TMEM is released
    mma_commit(&bars[C::kBarMmaDone]);
    mbar_wait_teardown(&bars[C::kBarMmaDone], 0);
}

// P V issuer (its own warp; one elected lane issues): O[slot] (+)= P V of
// every item in queue order as soon as the warpgroups have put P in TMEM, so
// it never waits for the next tile's loads; then S of the tile's next item,
// which overwrites the P just read (in issue order on this thread).  P comes
// from the slot's S columns (keys [16k, 16k + 16) in the first 8 columns of
// step k; softmax variant: in 32-column chunk k/2's first 16 columns, half
// k%2), V MN-major from shared memory.
template <int D, bool SM>
__device__ void fwd_mma_pv(const FwdParams& prm, uint8_t* smem, uint64_t* bars, uint32_t tmem,
                           volatile int* k_seen, int seg0, int seg1, const Abort& ab) {
    const int lane = threadIdx.x & 31;
    using C = FwdCfg<D>;
    uint32_t p_use0 = 0, p_use1 = 0, pb_use0 = 0, pb_use1 = 0, o_use0 = 0, o_use1 = 0;
    uint32_t a = 0, i = 0;
    for (int t = seg0; t < seg1; ++t) {
        // (the descriptor line 4 tiles ahead, so that this warp's next
        // descriptor loads hit in L1)
        if (t + 4 < seg1) prefetch_l1(prm.tiles + t + 4);
        const FwdTile tile = load_tile(prm.tiles + t);
        if (tile.kb1 <= tile.kb0) continue;
        const uint32_t wg = a % kNumWG;
        const uint32_t qs = a % C::kNQ;
        uint32_t& p_use = wg ? p_use1 : p_use0;
        uint32_t& pb_use = wg ? pb_use1 : pb_use0;   // second key halves
        uint32_t& o_use = wg ? o_use1 : o_use0;
        const int nit = tile_items<SM>(tile);
        for (int it = 0; it < nit; ++it, ++i) {
            const uint32_t ks = i % C::kNKV, kph = (i / C::kNKV) & 1;
            const int kb = item_block<SM>(tile, it);
            const bool pv = item_pv<SM>(tile, it);
            const bool first = pv && (it == 0 || !item_pv<SM>(tile, it - 1));
            const bool last = it == nit - 1;
            if (!wg_wait(&bars[C::kBarPFull + 2 * wg], p_use & 1, ab, 11)) goto drain;
            // (also for an item without P V: its V load must have landed
            // before the stage goes back to the producer)
            if (!wg_wait(&bars[C::kBarVFull + ks], kph, ab, 10)) goto drain;
            if (first && !wg_wait(&bars[C::kBarOFree + wg], (o_use & 1) ^ 1, ab, 12)) goto drain;
            {
                const int nvalid = min(kBN, tile.lkv - kb * kBN);
                const int nsteps = pv ? (nvalid + 15) >> 4 : 0;
                constexpr uint32_t idesc = idesc_bf16(128, D, false, true);
                const uint32_t p_tmem = tmem + wg * 256;
                const uint32_t d_o = tmem + wg * 256 + 128;
                const uint64_t vdesc =
                    smem_desc_sw128(smem_u32(smem + C::kOffV + ks * C::kTileBytes), kHalfBytes, 1024);
                // keys [0, 64) as soon as their P is in, keys [64, 128) once
                // the rest is
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    if (hlf == 1) {
                        if (nvalid <= 64) break;
                        if (!wg_wait(&bars[C::kBarPFull + 2 * wg + 1], pb_use & 1, ab, 11)) goto drain;
                        pb_use++;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int k = 4 * hlf; k < 4 * hlf + 4; ++k)
                        if (k < nsteps)
                            mma_ts(d_o, p_tmem + (SM ? (k >> 1) * 32 + (k & 1) * 8 : k * 16),
                                   vdesc + mnmajor_step(k), idesc, (first && k == 0) ? 0u : 1u);
                }
            }
            p_use++;
            mma_commit(&bars[C::kBarVEmpty + ks]);
            if (last) {
                mma_commit(&bars[C::kBarOFull + wg]);
                o_use++;
            } else {
                const uint32_t ks1 = (i + 1) % C::kNKV, kph1 = ((i + 1) / C::kNKV) & 1;
                // (item i - 1's K, kNKV back in this stage, has landed: its
                // S preceded this item's P V)
                if (!wg_wait(&bars[C::kBarKFull + ks1], kph1, ab, 4)) goto drain;
                if (lane == 0) atomicMax((int*)k_seen, (int)(i + 1));
                tc_fence_after();
                issue_s<D>(smem, bars, tmem, wg, qs, ks1,
                           min(kBN, tile.lkv - item_block<SM>(tile, it + 1) * kBN));
                mma_commit(&bars[C::kBarKEmpty + ks1]);
            }
        }
        ++a;
    }
drain:
    mma_commit(&bars[C::kBarMmaDone + 1]);
    mbar_wait_teardown(&bars[C::kBarMmaDone + 1], 0);
}

template <int D>
__device__ __forceinline__ void store_zero_rows(const FwdTile& tile, const FwdParams& prm, int tid) {
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const int64_t rs = (int64_t)prm.H * D;
    for (int idx = tid; idx < tile.nq * kChunks; idx += 128) {
        const int row = idx / kChunks, ch = idx % kChunks;
        *reinterpret_cast<uint4*>(prm.O + (int64_t)(tile.qt0 + row) * rs + tile.h * D + ch * 8) =
            make_uint4(0, 0, 0, 0);
    }
}

// Softmax variant (Jagged Flash Attention), one tile, one thread = one row
// of this part's key columns.  With t = alpha log2(e) s, the row maximum m
// of t over every valid key (a first pass over the key blocks when there are
// several), then P = 2^(t - m) (exactly zero for invalid pairs) into TMEM as
// for GDPA, and the row sum l.  The slot's two parts combine m, then l,
// through a TMEM column that no one else reads at that point: the first
// column of this part's O share before the tile's first P V (for m), the
// 17th column of this part's first S chunk, already read, before the last
// P is released (for l), meeting at the slot's exchange barrier (all 256
// threads, a bounded wait like every other).
// Returns 1 / l for the epilogue (0 for a row without a valid key), or a
// negative value if a wait gave up.
template <int D>
__device__ float softmax_tile(const FwdTile& tile, const FwdParams& prm, uint64_t* bars,
                              uint32_t& s_use, uint32_t& sb_use, uint32_t& x_use, uint32_t s_tmem,
                              uint32_t o_tmem_part0, int wg, int part, int r, bool warp_rows,
                              float alpha, const Abort& ab) {
    using C = FwdCfg<D>;
    const float c2 = alpha * 1.44269504088896340736f;   // alpha log2(e)
    const int ipos = tile.i0 + r;
    const int nit = tile_items<true>(tile);
    float m = -INFINITY, l = 0.0f;
    // write v to my column, meet the other part, read its value
    auto exchange = [&](uint32_t mine, uint32_t theirs, float v, float& out) -> bool {
        tmem_st1(mine, __float_as_uint(v));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[C::kBarXchg + wg]);
        if (!wg_wait(&bars[C::kBarXchg + wg], x_use & 1, ab, 14)) return false;
        x_use++;
        tc_fence_after();
        out = __uint_as_float(tmem_ld1(theirs));
        tmem_ld_wait();
        return true;
    };
    for (int it = 0; it < nit; ++it) {
        const int kb = item_block<true>(tile, it);
        const bool pv = item_pv<true>(tile, it);
        const bool single = tile.kb1 - tile.kb0 == 1;
        const int nvalid = min(kBN, tile.lkv - kb * kBN);
        const int nch = (nvalid + 31) >> 5;
        const int jbase = kb * kBN;
        if (!wg_wait(&bars[C::kBarSFull + 2 * wg], s_use & 1, ab, 6)) return -1.0f;
        s_use++;
        if (nvalid > 64) {
            if (!wg_wait(&bars[C::kBarSFull + 2 * wg + 1], sb_use & 1, ab, 6)) return -1.0f;
            sb_use++;
        }
        tc_fence_after();
        auto valid_at = [&](int col) {
            const int jpos = jbase + col;
            bool v = col < nvalid;
            if (prm.mask == GDPA_MASK_CAUSAL_WINDOW)
                v = v && jpos <= ipos && jpos > ipos - prm.window;
            return v;
        };
        if (!pv || single) {   // row maxima
            if (warp_rows) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = part + 2 * cc;
                    if (c < nch) {
#pragma unroll 1
                        for (int hh = 0; hh < 2; ++hh) {
                            const int col0 = c * 32 + hh * 16;
                            if (col0 >= nvalid) break;
                            uint32_t sv[16];
                            tmem_ld16(s_tmem + col0, sv);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float t = c2 * __uint_as_float(sv[e]);
                                m = valid_at(col0 + e) ? fmaxf(m, t) : m;
                            }
                        }
                    }
                }
            }
            if (single || it == nit / 2 - 1) {   // the maxima are complete: combine the parts
                float mo;
                if (!exchange(o_tmem_part0 + (uint32_t)(part * (D / 2)),
                              o_tmem_part0 + (uint32_t)((1 - part) * (D / 2)), m, mo))
                    return -1.0f;
                m = fmaxf(m, mo);
                if (m == -INFINITY) m = 0.0f;   // no valid key: every P is zero
            }
        }
        if (pv) {   // P = 2^(t - m), row sums
            if (warp_rows) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = part + 2 * cc;
                    if (c < nch) {
#pragma unroll 1
                        for (int hh = 0; hh < 2; ++hh) {
                            const int col0 = c * 32 + hh * 16;
                            if (col0 >= nvalid) break;
                            uint32_t sv[16], pk[8];
                            tmem_ld16(s_tmem + col0, sv);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                float pv2[2];
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const float w = ex2_approx(fmaf(c2, __uint_as_float(sv[e + u]), -m));
                                    pv2[u] = valid_at(col0 + e + u) ? w : 0.0f;
                                    l += pv2[u];
                                }
                                pk[e >> 1] = pack_bf16x2(pv2[0], pv2[1]);
                            }
                            tmem_st8(s_tmem + c * 32 + hh * 8, pk);
                        }
                    }
                }
                tmem_st_wait();
            }
            if (it == nit - 1) {   // the sums are complete: combine the parts
                float lo;
                if (!exchange(s_tmem + (uint32_t)(32 * part + 16),
                              s_tmem + (uint32_t)(32 * (1 - part) + 16), l, lo))
                    return -1.0f;
                l += lo;
            }
        }
        tc_fence_before();
        mbar_arrive(&bars[C::kBarPFull + 2 * wg]);
        if (nvalid > 64) mbar_arrive(&bars[C::kBarPFull + 2 * wg + 1]);
    }
    if (prm.lse && part == 0 && r < tile.nq)   // natural log of the row's sum of exp(alpha s)
        prm.lse[(int64_t)(tile.qt0 + r) * prm.H + tile.h] =
            l > 0.0f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    return l > 0.0f ? 1.0f / l : 0.0f;
}

template <int D, int ACT, bool SPLIT, bool NORM>
__device__ void fwd_compute(const FwdParams& prm, const CUtensorMap* tmO, const CUtensorMap* tmW,
                            uint8_t* smem,
                            uint64_t* bars, uint32_t tmem, int seg0, int seg1, const Abort& ab) {
    using C = FwdCfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = (warp - 2) >> 2;                 // warpgroup 0..3
    const uint32_t wg = (uint32_t)(grp % kNumWG);    // tile slot
    const int part = grp / kNumWG;                   // column share within the slot
    const int quarter = warp & 3;                    // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;               // tile row of this thread
    const int tid = (int)threadIdx.x - 64 - 128 * grp;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + wg * 256 + lane_addr;
    const uint32_t o_tmem = tmem + wg * 256 + 128 + lane_addr + part * (D / 2);
    ActScale ksc = act_scale<ACT>(prm.alpha);
    uint32_t a = 0, s_use = 0, sb_use = 0, o_use = 0, x_use = 0;
    for (int t = seg0; t < seg1; ++t) {
        // (the descriptor line 4 tiles ahead, so that this warp's next
        // descriptor loads hit in L1)
        if (t + 4 < seg1) prefetch_l1(prm.tiles + t + 4);
        const FwdTile tile = load_tile(prm.tiles + t);
        if (tile.kb1 <= tile.kb0) {
            if (!SPLIT && (t - seg0) % (kNumWG * kParts) == grp) store_zero_rows<D>(tile, prm, tid);
            continue;
        }
        if (a % kNumWG != wg) {
            ++a;
            continue;
        }
        const uint32_t qs = a % C::kNQ;
        const bool warp_rows = quarter * 32 < tile.nq;
        const int ipos = tile.i0 + r;
        // fused RMSNorm: the keys are normalised; this row's scale c, from
        // the tile's raw Q, joins alpha (x = alpha c q . k_hat)
        float alpha_row = prm.alpha;
        if constexpr (NORM) {
            if (!wg_wait(&bars[C::kBarQFull + qs], (a / C::kNQ) & 1, ab, 15)) return;
            alpha_row *= row_scale<D>(smem + C::kOffQ + qs * C::kTileBytes, r, prm.qk_gain,
                                      prm.qk_eps);
            ksc = act_scale<ACT>(alpha_row);
        }
        float oscale = 1.0f;   // the softmax variant's 1 / (row sum)
        if constexpr (ACT == kSoftmax) {
            oscale = softmax_tile<D>(tile, prm, bars, s_use, sb_use, x_use, s_tmem,
                                     tmem + wg * 256 + 128 + lane_addr, (int)wg, part, r, warp_rows,
                                     alpha_row, ab);
            if (__any_sync(0xffffffffu, oscale < 0.0f)) return;
        } else
        for (int kb = tile.kb0; kb < tile.kb1; ++kb) {
            const int nvalid = min(kBN, tile.lkv - kb * kBN);
            const int jbase = kb * kBN;
            // S -> registers 16 columns at a time; alpha, activation and mask;
            // P (bf16 pairs) back into the first 8 columns of the same
            // 16-column step, which only this warpgroup reads and has read.
            // Part h takes the steps h, h + 2, ...; the keys [0, 64) as soon
            // as their half of S is in, releasing their P to the P V issuer,
            // then the keys [64, 128)
#pragma unroll 1
            for (int hlf = 0; hlf < (nvalid > 64 ? 2 : 1); ++hlf) {
                if (!wg_wait(&bars[C::kBarSFull + 2 * wg + hlf], (hlf ? sb_use : s_use) & 1, ab, 6))
                    return;
                tc_fence_after();
                if (warp_rows) {
#pragma unroll 1
                    for (int k = 2 * hlf; k < 2 * hlf + 2; ++k) {
                        const int col0 = (part + 2 * k) * 16;
                        if (col0 >= nvalid) break;   // GEMMs stop at 16-column granularity
                        uint32_t sv[16], pk[8];
                        tmem_ld16(s_tmem + col0, sv);
                        tmem_ld_wait();
                        // the step's keys against the window of this warp's 32
                        // rows (warp-uniform): all valid, none valid, or mixed
                        // (per-pair masks)
                        const int jlo = jbase + col0, jhi = jlo + 15;
                        bool all_valid = col0 + 16 <= nvalid, none_valid = false;
                        if (prm.mask == GDPA_MASK_CAUSAL_WINDOW) {
                            const int ilo = tile.i0 + quarter * 32, ihi = ilo + 31;
                            all_valid = all_valid && jhi <= ilo && jlo > ihi - prm.window;
                            none_valid = jlo > ihi || jhi <= ilo - prm.window;
                        }
                        if (none_valid) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) pk[e] = 0u;
                        } else if (all_valid) {
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                float a0, a1;
                                act_s2<ACT>(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), ksc,
                                            a0, a1);
                                pk[e >> 1] = pack_bf16x2(a0, a1);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                float pv[2];
                                act_s2<ACT>(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), ksc,
                                            pv[0], pv[1]);
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const int col = col0 + e + u;
                                    const int jpos = jbase + col;
                                    bool valid = col < nvalid;
                                    if (prm.mask == GDPA_MASK_CAUSAL_WINDOW)
                                        valid = valid && jpos <= ipos && jpos > ipos - prm.window;
                                    pv[u] = valid ? pv[u] : 0.0f;
                                }
                                pk[e >> 1] = pack_bf16x2(pv[0], pv[1]);
                            }
                        }
                        tmem_st8(s_tmem + col0, pk);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(&bars[C::kBarPFull + 2 * wg + hlf]);
            }
            s_use++;
            if (nvalid > 64) sb_use++;
        }
        // epilogue: this part's O columns (TMEM) -> bf16 -> this part's half of
        // the tile's (consumed) Q buffer -> global
        if (!wg_wait(&bars[C::kBarOFull + wg], o_use & 1, ab, 8)) return;
        o_use++;
        tc_fence_after();
        if constexpr (SPLIT) {
            {
                // key-split plan: this tile holds a partial sum of its rows' O;
                // add it (float32, TMA bulk reduce-add) into the workspace that
                // a second kernel converts once every tile has landed
                static_assert(D == 128 && ACT != kSoftmax, "key split: d = 128 GDPA only");
                const int64_t rs = (int64_t)prm.H * D;
                drain_warp16_inl(tmem + wg * 256 + lane_addr, 128 + part * (D / 2), D / 2,
                           smem + C::kOffQ + qs * C::kTileBytes + part * (C::kTileBytes / 2), tmW,
                           tile.h * D + part * (D / 2), tile.qt0,
                           prm.W + (int64_t)tile.qt0 * rs + tile.h * D + part * (D / 2), rs,
                           tile.nq, true, 1.0f, quarter, lane, &bars[C::kBarOFree + wg]);
                staging_release_wait(lane);
                fence_proxy_async_smem();
                mbar_arrive(&bars[C::kBarQEmpty + qs]);
                ++a;
                continue;
            }
        }
        constexpr int kRowBytes = D;                 // D/2 bf16 per row and part
        constexpr int kChunks = kRowBytes / 16;      // 16-byte chunks per row
        constexpr int kSwz = kChunks - 1 < 7 ? kChunks - 1 : 7;
        uint8_t* stage = smem + C::kOffQ + qs * C::kTileBytes + part * (C::kTileBytes / 2);
        if (warp_rows) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t ov[32];
                tmem_ld32(o_tmem + c * 32, ov);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int chunk = (c * 4 + u) ^ (r & kSwz);
                    uint4 w;
                    w.x = pack_bf16x2(oscale * __uint_as_float(ov[8 * u + 0]), oscale * __uint_as_float(ov[8 * u + 1]));
                    w.y = pack_bf16x2(oscale * __uint_as_float(ov[8 * u + 2]), oscale * __uint_as_float(ov[8 * u + 3]));
                    w.z = pack_bf16x2(oscale * __uint_as_float(ov[8 * u + 4]), oscale * __uint_as_float(ov[8 * u + 5]));
                    w.w = pack_bf16x2(oscale * __uint_as_float(ov[8 * u + 6]), oscale * __uint_as_float(ov[8 * u + 7]));
                    *reinterpret_cast<uint4*>(stage + r * kRowBytes + chunk * 16) = w;
                }
            }
        }
        tc_fence_before();
        mbar_arrive(&bars[C::kBarOFree + wg]);
        if constexpr (D == 128) {
            // each warp writes its own 32 rows: one TMA bulk store of the
            // [32 x 64] box it staged (128-byte rows, 128-byte swizzle), or
            // plain stores of the valid rows for the tile's ragged warp
            const int row0 = quarter * 32;
            fence_proxy_async_smem();
            __syncwarp();
            if (row0 + 32 <= tile.nq) {
                if (lane == 0) {
                    tma_store_2d(tmO, stage + quarter * 4096, tile.h * D + part * (D / 2),
                                 tile.qt0 + row0);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                __syncwarp();
            } else if (row0 < tile.nq) {
                const int64_t rs = (int64_t)prm.H * D;
                __nv_bfloat16* obase = prm.O + (int64_t)tile.qt0 * rs + tile.h * D + part * (D / 2);
                for (int idx = lane; idx < (tile.nq - row0) * kChunks; idx += 32) {
                    const int row = row0 + idx / kChunks, ch = idx % kChunks;
                    const uint4 w = *reinterpret_cast<const uint4*>(stage + row * kRowBytes +
                                                                    ((ch ^ (row & kSwz)) * 16));
                    *reinterpret_cast<uint4*>(obase + (int64_t)row * rs + ch * 8) = w;
                }
            }
        } else {
            // the whole warpgroup's staging writes before anyone reads them back
            mbar_arrive(&bars[C::kBarStage + grp]);
            if (!wg_wait(&bars[C::kBarStage + grp], (o_use - 1) & 1, ab, 9)) return;
            const int64_t rs = (int64_t)prm.H * D;
            __nv_bfloat16* obase = prm.O + (int64_t)tile.qt0 * rs + tile.h * D + part * (D / 2);
            for (int idx = tid; idx < tile.nq * kChunks; idx += 128) {
                const int row = idx / kChunks, ch = idx % kChunks;
                const uint4 w = *reinterpret_cast<const uint4*>(stage + row * kRowBytes +
                                                                ((ch ^ (row & kSwz)) * 16));
                *reinterpret_cast<uint4*>(obase + (int64_t)row * rs + ch * 8) = w;
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[C::kBarQEmpty + qs]);
        ++a;
    }
}

template <int D, int ACT, bool SPLIT, bool NORM>
__global__ void __launch_bounds__(kThreads, 1)
tc_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const __grid_constant__ CUtensorMap tmW, const FwdParams prm) {
    using C = FwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // the highest item whose K-full the MMA warps have seen (the S issuer's
    // guard against reading a K-full phase two completions short)
    volatile int* k_seen = reinterpret_cast<volatile int*>(tmem_slot + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg0 = prm.seg[blockIdx.x], seg1 = prm.seg[blockIdx.x + 1];
    uint64_t t_start = 0;
    if (threadIdx.x == 0) {
        t_start = globaltimer();
        for (int s = 0; s < C::kNQ; ++s) {
            mbar_init(&bars[C::kBarQFull + s], 1);
            mbar_init(&bars[C::kBarQEmpty + s], 128 * kParts);
        }
        for (int s = 0; s < C::kNKV; ++s) {
            mbar_init(&bars[C::kBarKFull + s], 1);
            mbar_init(&bars[C::kBarVFull + s], 1);
            mbar_init(&bars[C::kBarKEmpty + s], 1);
            mbar_init(&bars[C::kBarVEmpty + s], 1);
        }
        for (int w = 0; w < 2 * kNumWG; ++w) {
            mbar_init(&bars[C::kBarSFull + w], 1);
            mbar_init(&bars[C::kBarPFull + w], 128 * kParts);
        }
        for (int w = 0; w < kNumWG; ++w) {
            mbar_init(&bars[C::kBarOFull + w], 1);
            mbar_init(&bars[C::kBarOFree + w], 128 * kParts);
        }
        for (int g = 0; g < kNumWG * kParts; ++g) mbar_init(&bars[C::kBarStage + g], 128);
        mbar_init(&bars[C::kBarMmaDone], 1);
        mbar_init(&bars[C::kBarMmaDone + 1], 1);
        for (int w = 0; w < kNumWG; ++w) mbar_init(&bars[C::kBarXchg + w], 128 * kParts);
        *abort_flag = 0;
        *k_seen = -1;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
        if (SPLIT) tma_prefetch_desc(&tmW);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, prm.err, prm.wait_ns};

    if (warp == 0) {
        if (lane == 0) fwd_producer<D, ACT == kSoftmax>(&tmQ, &tmK, &tmV, prm, smem, bars, seg0, seg1, ab);
        __syncwarp();
    } else if (warp == 1) {
        fwd_mma_s<D, ACT == kSoftmax>(prm, smem, bars, tmem, k_seen, seg0, seg1, ab);
        __syncwarp();
    } else if (warp == kPvWarp) {
        fwd_mma_pv<D, ACT == kSoftmax>(prm, smem, bars, tmem, k_seen, seg0, seg1, ab);
        __syncwarp();
    } else {
        fwd_compute<D, ACT, SPLIT, NORM>(prm, &tmO, &tmW, smem, bars, tmem, seg0, seg1, ab);
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && prm.timing) {
        prm.times[2 * blockIdx.x] = t_start;
        prm.times[2 * blockIdx.x + 1] = globaltimer();
        prm.smid[blockIdx.x] = (int32_t)smid();
    }
}

template <int D, int ACT, bool SPLIT, bool NORM>
gdpa_status launch1(int S, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                    const CUtensorMap& mo, const CUtensorMap& mw, const FwdParams& prm,
                    cudaStream_t st) {
    using C = FwdCfg<D>;
    auto kern = tc_fwd_kernel<D, ACT, SPLIT, NORM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return GDPA_ERR_CUDA;
    kern<<<S, kThreads, C::kSmemBytes, st>>>(mq, mk, mv, mo, mw, prm);
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

// the fused RMSNorm is a separate instantiation, so that the plain kernels
// carry none of its work
template <int D, int ACT, bool SPLIT = false>
gdpa_status launch(int S, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                   const CUtensorMap& mo, const CUtensorMap& mw, const FwdParams& prm,
                   cudaStream_t st) {
    return prm.qk_gain > 0.0f ? launch1<D, ACT, SPLIT, true>(S, mq, mk, mv, mo, mw, prm, st)
                              : launch1<D, ACT, SPLIT, false>(S, mq, mk, mv, mo, mw, prm, st);
}

// Key-split plans: O = bf16(W), four elements per thread and step.
__global__ void __launch_bounds__(256) split_finalize_kernel(const float4* __restrict__ w,
                                                             uint2* __restrict__ o, int64_t n4) {
    for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < n4; i += (int64_t)gridDim.x * 256) {
        const float4 x = w[i];
        o[i] = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
    }
}

}  // namespace

gdpa_status launch_tc_fwd_raw(const FwdTile* tiles, const int32_t* seg, int S, int32_t* err,
                              unsigned long long* times, int32_t* smid, int H, int d, int64_t Tq,
                              int64_t Tkv, int mask, int window, const void* q, int64_t q_rows,
                              int shared_q, const void* k, const void* v, void* o, float* lse,
                              float* w, float alpha, int act, cudaStream_t st,
                              uint32_t wait_limit_us, int stall, float qk_gain, float qk_eps) {
    if (d != 64 && d != 128) return GDPA_ERR_UNSUPPORTED;
    if (w && (d != 128 || act == kSoftmax)) return GDPA_ERR_UNSUPPORTED;
    if (Tq == 0) return GDPA_OK;
    CUtensorMap mq, mk, mv, mo, mw;
    const uint64_t row = (uint64_t)H * d;
    const uint64_t kv_rows = Tkv > 0 ? (uint64_t)Tkv : 1;
    const void* kp = Tkv > 0 ? k : q;
    const void* vp = Tkv > 0 ? v : q;
    if (q_rows < 1) return GDPA_ERR_INVALID_ARG;
    if (!tc::make_tmap_bf16(&mq, q, (uint64_t)q_rows, row, 128) ||
        !tc::make_tmap_bf16(&mk, kp, kv_rows, row, 128) ||
        !tc::make_tmap_bf16(&mv, vp, kv_rows, row, 128) ||
        !tc::make_tmap_bf16(&mo, o, (uint64_t)Tq, row, 32))
        return GDPA_ERR_CUDA;
    if (w) {
        if (!tc::make_tmap_f32(&mw, w, (uint64_t)Tq, row, 32, 16)) return GDPA_ERR_CUDA;
    } else {
        mw = mo;   // not read
    }
    FwdParams prm;
    prm.tiles = tiles;
    prm.seg = seg;
    prm.O = (__nv_bfloat16*)o;
    prm.lse = lse;
    prm.W = w;
    prm.shared_q = shared_q;
    prm.H = H;
    prm.alpha = alpha;
    prm.mask = mask;
    prm.window = window;
    prm.err = err;
    prm.times = times;
    prm.smid = smid;
    prm.timing = times != nullptr && smid != nullptr;
    prm.wait_ns = tc::wait_limit_ns(wait_limit_us);
    prm.stall = stall;
    prm.qk_gain = qk_gain;
    prm.qk_eps = qk_eps;
    gdpa_status s = GDPA_OK;
    if (w) {
        GDPA_DISPATCH_ACT(act, A, s = launch<128, A, true>(S, mq, mk, mv, mo, mw, prm, st))
    } else if (d == 128) {
        if (act == kSoftmax)
            s = launch<128, kSoftmax>(S, mq, mk, mv, mo, mw, prm, st);
        else
            GDPA_DISPATCH_ACT(act, A, s = launch<128, A>(S, mq, mk, mv, mo, mw, prm, st))
    } else {
        if (act == kSoftmax)
            s = launch<64, kSoftmax>(S, mq, mk, mv, mo, mw, prm, st);
        else
            GDPA_DISPATCH_ACT(act, A, s = launch<64, A>(S, mq, mk, mv, mo, mw, prm, st))
    }
    return s;
}

gdpa_status launch_tc_fwd(Plan& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, float alpha, int act, cudaStream_t st) {
    if (p.n_fwd == 0) return GDPA_OK;
    float* w = nullptr;
    if (p.fwd_split) {
        // key-split plan: the tiles of one query tile add float32 partial sums
        // into a zeroed workspace; a second kernel rounds it into O
        if (p.d != 128 || act == kSoftmax) return GDPA_ERR_UNSUPPORTED;
        const size_t bytes = (size_t)p.Tq * p.H * p.d * sizeof(float);
        if (!p.d_wsplit && cudaMallocAsync((void**)&p.d_wsplit, bytes, st) != cudaSuccess) {
            p.d_wsplit = nullptr;
            return GDPA_ERR_ALLOC;
        }
        if (cudaMemsetAsync(p.d_wsplit, 0, bytes, st) != cudaSuccess) return GDPA_ERR_CUDA;
        w = p.d_wsplit;
    }
    if (p.timing) p.timed[0] = 1;
    if (p.qk_gain > 0.0f) {   // fused RMSNorm: the normalised keys first
        gdpa_status ks;
        k = plan_key_norm(p, k, st, &ks);
        if (ks != GDPA_OK) return ks;
    }
    gdpa_status s = launch_tc_fwd_raw(
        p.d_fwd, p.d_fwd_seg, p.S, p.d_err, p.timing ? p.d_times : nullptr,
        p.timing ? p.d_smid : nullptr, p.H, p.d, p.Tq, p.Tkv, p.mask, p.window, q,
        p.shared_q > 0 ? (int64_t)p.shared_q : p.Tq, p.shared_q > 0, k, v, o, lse, w, alpha, act,
        st, p.wait_limit_us, p.stall, p.qk_gain, p.qk_eps);
    if (s == GDPA_OK) p.launches += 1;
    if (s == GDPA_OK && w) {
        const int64_t n4 = p.Tq * p.H * p.d / 4;
        const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, 152 * 8);
        split_finalize_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(w),
                                                      reinterpret_cast<uint2*>(o), n4);
        s = cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
        if (s == GDPA_OK) p.launches += 1;
    }
    return s;
}

}  // namespace gdpa
