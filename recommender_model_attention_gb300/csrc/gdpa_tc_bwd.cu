// Persistent tcgen05 GDPA backward kernel (bf16 inputs, fp32 gradients).
//
// With x = alpha q.k over the valid pairs of a sample, P = act(x) and
// dS = (dO V^T) * act'(x) (the derivative of O = act(alpha Q K^T) V, the GDPA
// of "범용 내적 어텐션(GDPA)", aitrends.kr, which has no softmax and so no
// row-sum term):
//     dV = P^T dO,   dK = alpha dS^T Q,   dQ = alpha dS K.
//
// Work unit = one 128-row key block of one (sample, head) with the range of
// 128-row query tiles that see it (host plan, zigzag-dealt like the forward
// tiles).  The unit's dK and dV accumulate in TMEM over its query tiles and
// are stored once; each query tile's dQ is complete when the sample has a
// single key block (stored directly) and is otherwise added atomically into
// a cleared dQ.
//
// Roles: warp 0 TMA producer (K, V once per unit; Q and dO per query tile
// through 2-stage rings, the next tile's and the next unit's boxes
// prefetched into L2); warp 1 tcgen05.mma issuer (the whole warp runs
// the issue code, one elected lane issues); warps 2-9 two
// warpgroups that turn S and dP (TMEM) into dS and P (bf16, shared memory),
// warpgroup j taking the 16-column key steps j, j + 2, ..., and drain dQ (j:
// d columns [64j, 64j + 64)), dV (j = 0) and dK (j = 1) from TMEM.  Per
// query tile:
//     S  = Q K^T   -> TMEM [0, 128)      dP = dO V^T -> TMEM [128, 256)
//     dS           -> the 32 KB shared [query x key] buffer, and packed into
//                     the first half of each 16-column step of S's own
//                     columns (already read)
//     dK += dS^T Q -> TMEM [384, 512), dS^T from the buffer
//     dQ  = dS K   -> TMEM [128, 256) (dP's columns, already read), dS from
//                     TMEM
//     P            -> the same buffer, once dK has read dS
//     dV += P^T dO -> TMEM [256, 384), while the warpgroups drain dQ through
//                     the tile's Q buffer (its MMAs are done)
// The next tile's S is issued as soon as both warpgroups have read S, its dP
// once dQ is drained; dV stays off the warpgroups' critical path.  P^T and
// dS^T are the MN-major reading of the [query x key] buffer, and Q, dO, K
// are the MN-major reading of their [row x d] tiles, so nothing is
// transposed in memory.  Every wait is bounded (timeouts set the plan's
// error word; the CTA unwinds, frees TMEM and returns).
#include <cuda_bf16.h>

#include "act.cuh"
#include "tc_common.cuh"
#include "tc_drain.cuh"

namespace gdpa {
namespace {

using namespace tc;

constexpr int kThreads = 64 + 256;
constexpr int kHalfBytes = 128 * 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

template <int D>
struct BwdCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kTileBytes = 128 * D * 2;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;          // 2 stages
    static constexpr int kOffDO = kOffQ + 2 * kTileBytes;     // 2 stages
    static constexpr int kOffPS = kOffDO + 2 * kTileBytes;    // P / dS / staging
    static constexpr int kOffDot = kOffPS + 128 * 128 * 2;    // fused RMSNorm: [2][128] f32
    static constexpr int kOffBar = kOffDot + 2 * 128 * 4;
    enum {
        kKVFull = 0, kKVEmpty, kQFull, kQFull1, kQEmpty, kQEmpty1, kDOFull, kDOFull1, kDOEmpty,
        kDOEmpty1, kSDFull, kSFree, kDQFree, kPFull, kPVDone, kDSFull, kDKDone, kAccFull,
        kAccFree, kStage, kStage1, kPSFree, kMmaDone, kDQDone, kDotFull, kNumBars
    };
    static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
};

struct BwdParams {
    const BwdUnit* units;
    const int32_t* seg;
    float* dQ;
    float* dK;
    float* dV;
    const float* lse;     // softmax variant: row log-sum-exp [Tq][H]
    const float* delta;   // softmax variant: dO . O per row [Tq][H]
    int shared_q;         // Q and dQ hold seed rows shared by all samples
    int H;
    float alpha;
    int mask;
    int window;
    int32_t* err;
    unsigned long long* times;
    int32_t* smid;
    int timing;
    uint64_t wait_ns;     // bounded-wait limit
    int stall;            // test hook: CTA 0 skips its first Q load
    // fused RMSNorm (or NULL): the keys arrive normalised and kscale holds
    // each key row's g / rms, [H][ld] floats; each query row's scale is
    // computed from its tile (gain, eps) and folded into alpha
    const float* kscale;
    int64_t kscale_ld;
    float qk_gain, qk_eps;
};

__device__ __forceinline__ BwdUnit load_unit(const BwdUnit* p) {
    const int4* q = reinterpret_cast<const int4*>(p);
    const int4 a = __ldg(q), b = __ldg(q + 1);
    BwdUnit u;
    u.kvt0 = a.x; u.nkv = a.y; u.qt0 = a.z; u.lq = a.w;
    u.hf = b.x; u.m0 = b.y; u.m1 = b.z; u.c0 = b.w;
    return u;
}

template <int D>
__device__ void bwd_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                             const CUtensorMap* tmDO, const BwdParams& prm, uint8_t* smem,
                             uint64_t* bars, int seg0, int seg1, const Abort& ab) {
    using C = BwdCfg<D>;
    const uint64_t pol_stream = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int32_t kv_armed = -1, q_armed[2] = {-1, -1}, do_armed[2] = {-1, -1};
    uint32_t nu = 0, i = 0;
    for (int t = seg0; t < seg1; ++t) {
        const BwdUnit u = load_unit(prm.units + t);
        if (u.m1 <= u.m0) continue;
        const int h = u.hf & 0xffff;
        if (!mbar_wait(&bars[C::kKVEmpty], (nu & 1) ^ 1, ab, 21)) goto unwind;
        mbar_arrive_expect_tx(&bars[C::kKVFull], 2 * C::kTileBytes);
        kv_armed = (int32_t)(nu & 1);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
            tma_load_2d(tmK, &bars[C::kKVFull], smem + C::kOffK + hf * kHalfBytes, h * D + hf * 64,
                        u.kvt0, pol_keep);
            tma_load_2d(tmV, &bars[C::kKVFull], smem + C::kOffV + hf * kHalfBytes, h * D + hf * 64,
                        u.kvt0, pol_keep);
        }
        for (int m = u.m0; m < u.m1; ++m, ++i) {
            const uint32_t s = i & 1, ph = (i >> 1) & 1;
            const int y = u.qt0 + m * kBM;   // dO rows
            const int yq = prm.shared_q ? m * kBM : y;
            if (!mbar_wait(&bars[C::kQEmpty + s], ph ^ 1, ab, 22)) goto unwind;
            // failure-path test hook: CTA 0 never loads its first Q tile, so
            // the MMA warp's bounded wait for it expires
            if (!(prm.stall && blockIdx.x == 0 && i == 0)) {
                mbar_arrive_expect_tx(&bars[C::kQFull + s], C::kTileBytes);
                q_armed[s] = (int32_t)ph;
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf)
                    tma_load_2d(tmQ, &bars[C::kQFull + s],
                                smem + C::kOffQ + s * C::kTileBytes + hf * kHalfBytes,
                                h * D + hf * 64, yq, pol_stream);
            }
            if (!mbar_wait(&bars[C::kDOEmpty + s], ph ^ 1, ab, 23)) goto unwind;
            mbar_arrive_expect_tx(&bars[C::kDOFull + s], C::kTileBytes);
            do_armed[s] = (int32_t)ph;
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf)
                tma_load_2d(tmDO, &bars[C::kDOFull + s],
                            smem + C::kOffDO + s * C::kTileBytes + hf * kHalfBytes, h * D + hf * 64,
                            y, pol_stream);
            if (!prm.kscale && m + 1 < u.m1) {
                // the next query tile's Q and dO boxes into L2 (evict-last,
                // so that they stay until their loads take them): their ring
                // loads wait for this tile's stages to free and then find
                // them there (a shared Q stays in L2 anyway).  The fused
                // RMSNorm kernel, bound by its arithmetic, runs faster
                // without.
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    if (!prm.shared_q) tma_prefetch_2d(tmQ, h * D + hf * 64, y + kBM, pol_keep);
                    tma_prefetch_2d(tmDO, h * D + hf * 64, y + kBM, pol_keep);
                }
            }
            if (m == u.m0) {
                // the next unit's K and V into L2 now, so that its loads at
                // the unit boundary need not come from HBM
                for (int t1 = t + 1; t1 < seg1; ++t1) {
                    const BwdUnit u1 = load_unit(prm.units + t1);
                    if (u1.m1 <= u1.m0) continue;
                    const int h1 = u1.hf & 0xffff;
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf) {
                        tma_prefetch_2d(tmK, h1 * D + hf * 64, u1.kvt0, pol_keep);
                        tma_prefetch_2d(tmV, h1 * D + hf * 64, u1.kvt0, pol_keep);
                    }
                    break;
                }
            }
        }
        ++nu;
    }
unwind:
    if (kv_armed >= 0) mbar_wait_teardown(&bars[C::kKVFull], (uint32_t)kv_armed);
    for (int s = 0; s < 2; ++s) {
        if (q_armed[s] >= 0) mbar_wait_teardown(&bars[C::kQFull + s], (uint32_t)q_armed[s]);
        if (do_armed[s] >= 0) mbar_wait_teardown(&bars[C::kDOFull + s], (uint32_t)do_armed[s]);
    }
}

template <int D>
__device__ void bwd_mma(const BwdParams& prm, uint8_t* smem, uint64_t* bars, uint32_t tmem,
                        int seg0, int seg1, const Abort& ab) {
    using C = BwdCfg<D>;
    const uint32_t kbase = smem_u32(smem + C::kOffK);
    const uint32_t vbase = smem_u32(smem + C::kOffV);
    const uint32_t psbase = smem_u32(smem + C::kOffPS);
    constexpr uint32_t idesc_acc = idesc_bf16(128, D, true, true);   // P^T dO, dS^T Q
    constexpr uint32_t idesc_dq = idesc_bf16(128, D, false, true);   // dS K
    // K-major descriptors of the resident K and V tiles
    const uint64_t kd_k = smem_desc_sw128(kbase, 16, 1024);
    const uint64_t vd_k = smem_desc_sw128(vbase, 16, 1024);

    uint32_t nu = 0, i = 0;
    for (int t = seg0; t < seg1; ++t) {
        const BwdUnit u = load_unit(prm.units + t);
        if (u.m1 <= u.m0) continue;
        const uint32_t nkv16 = (uint32_t)((u.nkv + 15) & ~15);
        const uint32_t idesc_s = idesc_bf16(128, nkv16, false, false);
        // S = Q K^T of item j (after the warpgroups have read item j-1's S)
        auto issue_s = [&](uint32_t j) -> bool {
            const uint32_t st = j & 1, ph = (j >> 1) & 1;
            if (!wg_wait(&bars[C::kQFull + st], ph, ab, 32)) return false;
            if (!wg_wait(&bars[C::kSFree], (j & 1) ^ 1, ab, 33)) return false;
            tc_fence_after();
            const uint32_t qb = smem_u32(smem + C::kOffQ + st * C::kTileBytes);
            const uint64_t qd = smem_desc_sw128(qb, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_ss(tmem + kColS, qd + kmajor_step(k), kd_k + kmajor_step(k), idesc_s, k > 0);
            return true;
        };
        // dP = dO V^T of item j (into the columns item j-1's dQ used)
        auto issue_dp = [&](uint32_t j) -> bool {
            const uint32_t st = j & 1, ph = (j >> 1) & 1;
            if (!wg_wait(&bars[C::kDOFull + st], ph, ab, 34)) return false;
            if (!wg_wait(&bars[C::kDQFree], (j & 1) ^ 1, ab, 35)) return false;
            tc_fence_after();
            const uint32_t dob = smem_u32(smem + C::kOffDO + st * C::kTileBytes);
            const uint64_t dd = smem_desc_sw128(dob, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                mma_ss(tmem + kColDP, dd + kmajor_step(k), vd_k + kmajor_step(k), idesc_s, k > 0);
            mma_commit(&bars[C::kSDFull]);
            return true;
        };
        if (!wg_wait(&bars[C::kKVFull], nu & 1, ab, 31)) goto drain;
        if (!issue_s(i) || !issue_dp(i)) goto drain;
        for (int m = u.m0; m < u.m1; ++m, ++i) {
            const uint32_t s = i & 1;
            const bool first = m == u.m0, last = m == u.m1 - 1;
            const int nq = min(kBM, u.lq - m * kBM);
            const uint32_t nq32 = (uint32_t)((nq + 31) & ~31);
            const uint32_t qb = smem_u32(smem + C::kOffQ + s * C::kTileBytes);
            const uint32_t dob = smem_u32(smem + C::kOffDO + s * C::kTileBytes);
            // dK += dS^T Q (dS^T from the shared buffer), then dQ = dS K into
            // dP's columns (already read), dS from TMEM: the warpgroups may
            // replace dS by P in the buffer as soon as dK is done
            if (!wg_wait(&bars[C::kDSFull], i & 1, ab, 38)) goto drain;
            if (first && !wg_wait(&bars[C::kAccFree], (nu & 1) ^ 1, ab, 37)) goto drain;
            tc_fence_after();
            for (uint32_t k = 0; k < nq32 / 16; ++k)
                mma_ss(tmem + kColDK, smem_desc_sw128(psbase + k * 2048, kHalfBytes, 1024),
                       smem_desc_sw128(qb + k * 2048, kHalfBytes, 1024), idesc_acc,
                       (first && k == 0) ? 0u : 1u);
            mma_commit(&bars[C::kDKDone]);
            for (uint32_t k = 0; k < nkv16 / 16; ++k)
                mma_ts(tmem + kColDP, tmem + kColS + k * 16,
                       smem_desc_sw128(kbase + k * 2048, kHalfBytes, 1024), idesc_dq, k > 0);
            mma_commit(&bars[C::kDQDone]);
            // the unit's last reader of K and V (dV reads P and dO): the
            // stage goes back to the producer (the fused RMSNorm's dK drain
            // still reads K: warpgroup 1 hands it back then)
            if (last && !prm.kscale) mma_commit(&bars[C::kKVEmpty]);
            // the next tile's scores (the warpgroups have read this tile's S)
            if (!last && !issue_s(i + 1)) goto drain;
            // dV += P^T dO once P has replaced dS in shared memory
            if (!wg_wait(&bars[C::kPFull], i & 1, ab, 36)) goto drain;
            tc_fence_after();
            for (uint32_t k = 0; k < nq32 / 16; ++k)
                mma_ss(tmem + kColDV, smem_desc_sw128(psbase + k * 2048, kHalfBytes, 1024),
                       smem_desc_sw128(dob + k * 2048, kHalfBytes, 1024), idesc_acc,
                       (first && k == 0) ? 0u : 1u);
            mma_commit(&bars[C::kPVDone]);
            mma_commit(&bars[C::kDOEmpty + s]);
            if (last) {
                mma_commit(&bars[C::kAccFull]);
            } else if (!issue_dp(i + 1)) {   // once this tile's dQ is drained
                goto drain;
            }
        }
        ++nu;
    }
drain:
    mma_commit(&bars[C::kMmaDone]);
    mbar_wait_teardown(&bars[C::kMmaDone], 0);
}

template <int D>
__device__ __forceinline__ void zero_rows(float* dst, int64_t rs, int nrows, int tid) {
    constexpr int kChunks = D / 4;
    for (int idx = tid; idx < nrows * kChunks; idx += 128) {
        const int row = idx / kChunks, ch = idx % kChunks;
        *reinterpret_cast<float4*>(dst + (int64_t)row * rs + ch * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// 16 columns (half hh of 32-column chunk c) of P or dS into the [query x key]
// SW128 buffer
__device__ __forceinline__ void store_half_chunk(uint8_t* ps, int c, int hh, int r,
                                                 const uint32_t (&v)[8]) {
    uint8_t* rowp = ps + (c >> 1) * kHalfBytes + r * 128;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const int chunk = ((c & 1) * 4 + hh * 2 + w) ^ (r & 7);
        *reinterpret_cast<uint4*>(rowp + chunk * 16) =
            make_uint4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
    }
}

// Fused RMSNorm: the drain of a row's gradient with respect to the
// normalised row, dy = TMEM value (times alpha for dQ and dK), into the
// gradient with respect to the raw row x,
//     dx = c (dy - x (x . dy) c^2 / (d g^2)),   c = g / rms(x),
// i.e. out = sc (v - kappa x) with sc = alpha c and kappa = (x . v) c^2 /
// (d g^2) (or, in terms of the normalised row x_hat = c x, kappa = (x_hat .
// v) / (d g^2) with x_hat in place of x).  Columns [col, col + 16 P) of this
// warp's 32 lanes, 16 at a time; xw(step, x8) gives the 8 packed bf16 words
// of x for columns col + 16 step ..; staging and stores as drain_warp, the
// plain (not reduce-add) stores marked evict-first in L2.
template <int P, typename XW>
__device__ __forceinline__ void drain_warp_norm(uint32_t trow, uint32_t col, uint8_t* stage,
                                                const CUtensorMap* map, int x0, int y0, float* dst,
                                                int64_t rs, int nrows, bool atomic, float sc,
                                                float kappa, XW xw, int quarter, int lane,
                                                uint64_t* release) {
    const int row0 = quarter * 32;
    const bool any = row0 < nrows;
    const bool full = row0 + 32 <= nrows;
    uint8_t* wst = stage + quarter * 4096;
#pragma unroll
    for (int pass = 0; pass < P; ++pass) {
        uint32_t v[16];
        if (any) {
            tmem_ld16(trow + col + pass * 16, v);
            tmem_ld_wait();
        }
        if (pass == P - 1 && release) {
            tc_fence_before();
            mbar_arrive(release);
        }
        if (!any) continue;
        uint32_t x8[8];
        xw(pass, x8);
        float o[16];
        const uint64_t nk2 = f2_make(-kappa, -kappa), sc2 = f2_make(sc, sc);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 r2 = f2_split(f2_mul(
                sc2, f2_fma(nk2, f2_bf16x2(x8[e]),
                            f2_make(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])))));
            o[2 * e] = r2.x;
            o[2 * e + 1] = r2.y;
        }
        if (full) {
            uint8_t* buf = wst + (pass & 1) * 2048;
            if (pass >= 2) {
                if (lane == 0) bulk_wait_read_but1();
                __syncwarp();
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<float4*>(buf + stage_off64(lane, c)) =
                    make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (atomic)
                    tma_reduce_add_2d(map, buf, x0 + pass * 16, y0 + row0);
                else   // (evict-first: 6.28 -> 6.10 ms for this kernel's backward,
                       // where the same hint slows the plain kernels' stores)
                    tma_store_2d_hint(map, buf, x0 + pass * 16, y0 + row0, policy_evict_first());
                bulk_commit();
            }
        } else if (row0 + lane < nrows) {
            float* d = dst + (int64_t)(row0 + lane) * rs + pass * 16;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 w = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                if (atomic)
                    atomicAdd(reinterpret_cast<float4*>(d + 4 * c), w);
                else
                    *reinterpret_cast<float4*>(d + 4 * c) = w;
            }
        }
    }
}

// 8 packed bf16 words: columns [c0, c0 + 16) of row r of a [128 x D] bf16
// tile in shared memory (128-byte-swizzled halves of 64 columns)
__device__ __forceinline__ void load_row16(const uint8_t* tile, int r, int c0, uint32_t (&x)[8]) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int c = c0 / 8 + q;
        const uint4 v = *reinterpret_cast<const uint4*>(tile + (c >> 3) * 16384 + r * 128 +
                                                        (((c & 7) ^ (r & 7)) << 4));
        x[4 * q] = v.x;
        x[4 * q + 1] = v.y;
        x[4 * q + 2] = v.z;
        x[4 * q + 3] = v.w;
    }
}

// The dQ tile's drain with the RMSNorm Jacobian.  The keys are normalised
// (k_hat) and x = alpha c q . k_hat, so the TMEM tile T = dS K_hat gives the
// gradient alpha T for the normalised row, and its dot with the raw row is
// q . (alpha T) = alpha sum_j dS_j s_j, the row's `dot` over all keys (the
// warpgroups' shares added): dq = alpha c (T - q dot c^2 / (d g^2)).  The
// raw row's columns [64 wg, 64 wg + 64) come from the tile's Q stage, all
// read before the drain's first staging write goes over them.
template <int D>
static __device__ __noinline__ void drain_dq_norm(uint32_t trow, int wg, int r, const uint8_t* qtile,
                                                  float dot, uint8_t* stage, const CUtensorMap* map,
                                                  int x0, int y0, float* dst, int64_t rs, int nrows,
                                                  bool atomic, float alpha, float ci, float gain,
                                                  int quarter, int lane, uint64_t* release) {
    uint32_t xq[32];
    load_row_bf16<2>(qtile, r, 64 * wg, xq);
    __syncwarp();   // every lane's row is read before any staging write lands on it
    const float kappa = dot * ci * ci / ((float)D * gain * gain);
    drain_warp_norm<4>(
        trow, kColDP + 64 * wg, stage, map, x0, y0, dst, rs, nrows, atomic, alpha * ci, kappa,
        [&](int step, uint32_t (&x8)[8]) {
#pragma unroll
            for (int e = 0; e < 8; ++e) x8[e] = xq[8 * step + e];
        },
        quarter, lane, release);
}

// The unit's dK drain with the RMSNorm Jacobian (warpgroup 1).  In terms of
// the normalised key row k_hat (the K stage holds it) and the TMEM row U
// (the gradient for k_hat is alpha U): dk = alpha c (U - k_hat (k_hat . U)
// / (d g^2)).  The K stage goes back to the producer (`kv_empty`) after the
// drain's last read of it.
template <int D>
static __device__ __noinline__ void drain_dk_norm(uint32_t trow, int r, const uint8_t* ktile,
                                                  uint8_t* stage, const CUtensorMap* map, int x0,
                                                  int y0, float* dst, int64_t rs, int nrows,
                                                  float alpha, float cj, float gain, int quarter,
                                                  int lane, uint64_t* kv_empty, uint64_t* release) {
    float dot = 0.0f;
    if (quarter * 32 < nrows) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t v[16], x8[8];
            tmem_ld16(trow + kColDK + c0, v);
            load_row16(ktile, r, c0, x8);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                dot = fmaf(bf16_lo(x8[e]), __uint_as_float(v[2 * e]), dot);
                dot = fmaf(bf16_hi(x8[e]), __uint_as_float(v[2 * e + 1]), dot);
            }
        }
    }
    const float kappa = dot / ((float)D * gain * gain);
    drain_warp_norm<D / 16>(
        trow, kColDK, stage, map, x0, y0, dst, rs, nrows, false, alpha * cj, kappa,
        [&](int step, uint32_t (&x8)[8]) { load_row16(ktile, r, 16 * step, x8); },
        quarter, lane, release);
    mbar_arrive(kv_empty);
}

// P and dS of one pair from its score s and dP: GDPA, P = act(alpha s) and
// dS = dP act'(alpha s); the softmax variant, P = exp(alpha s - lse) (in base
// 2 with lse2 = lse log2 e) and dS = P (dP - D), lse2 and D being the row's.
template <int ACT>
__device__ __forceinline__ void bwd_p_ds(float s, float dp, const ActScale& k, float lse2,
                                         float drow, float& p, float& ds) {
    if constexpr (ACT == kSoftmax) {
        p = ex2_approx(fmaf(s, k.c0, -lse2));
        ds = p * (dp - drow);
    } else {
        float da;
        act_dact_s<ACT>(s, k, p, da);
        ds = dp * da;
    }
}

// bwd_p_ds of two pairs at once (f32x2 arithmetic for the GDPA activations;
// the same results)
template <int ACT>
__device__ __forceinline__ void bwd_p_ds2(float s0, float s1, float dp0, float dp1,
                                          const ActScale& k, float lse2, float drow, float& p0,
                                          float& p1, float& ds0, float& ds1) {
    if constexpr (ACT == kSoftmax) {
        bwd_p_ds<ACT>(s0, dp0, k, lse2, drow, p0, ds0);
        bwd_p_ds<ACT>(s1, dp1, k, lse2, drow, p1, ds1);
    } else {
        float da0, da1;
        act_dact_s2<ACT>(s0, s1, k, p0, p1, da0, da1);
        const float2 d = f2_split(f2_mul(f2_make(dp0, dp1), f2_make(da0, da1)));
        ds0 = d.x;
        ds1 = d.y;
    }
}

template <int D, int ACT, bool NORM>
__device__ void bwd_compute(const BwdParams& prm, const CUtensorMap* tmDQ, const CUtensorMap* tmDK,
                            const CUtensorMap* tmDV, uint8_t* smem, uint64_t* bars, uint32_t tmem,
                            int seg0, int seg1, const Abort& ab) {
    using C = BwdCfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = (warp - 2) >> 2;      // key chunks c = wg, wg + 2
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // TMEM lane = row of this thread
    const int tid = (int)threadIdx.x - 64 - 128 * wg;
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* ps = smem + C::kOffPS;
    uint8_t* stage = ps + wg * kHalfBytes;
    const int64_t rs = (int64_t)prm.H * D;
    ActScale ksc = act_scale<ACT>(prm.alpha);
    uint32_t nu = 0, i = 0;
    int pending_q = -1;   // Q stage still read by this warp's last dQ stores
    for (int t = seg0; t < seg1; ++t) {
        const BwdUnit u = load_unit(prm.units + t);
        const int h = u.hf & 0xffff;
        // shared seeds: every sample adds its dQ into the same seed rows
        const bool atomic_dq = prm.shared_q || ((u.hf >> 16) & kUnitAtomicDQ);
        const int dq_row0 = prm.shared_q ? 0 : u.qt0;   // dQ row of the sample's query 0
        if (u.m1 <= u.m0) {
            float* base = (wg == 0 ? prm.dK : prm.dV) + (int64_t)u.kvt0 * rs + h * D;
            zero_rows<D>(base, rs, u.nkv, tid);
            continue;
        }
        const int nh = (u.nkv + 15) >> 4;   // 16-column key steps; this warpgroup: s = wg + 2k
        // softmax variant: the row statistics of query tile m, loaded one tile
        // ahead so that their latency hides behind the previous tile
        auto row_stats = [&](int m, float& l_out, float& d_out) {
            l_out = -INFINITY;
            d_out = 0.0f;
            if (m * kBM + r < u.lq) {
                const int64_t ri = (int64_t)(u.qt0 + m * kBM + r) * prm.H + h;
                l_out = prm.lse[ri];
                d_out = prm.delta[ri];
            }
        };
        float lse_next = 0.0f, d_next = 0.0f;
        if constexpr (ACT == kSoftmax) row_stats(u.m0, lse_next, d_next);
        for (int m = u.m0; m < u.m1; ++m, ++i) {
            const int nq = min(kBM, u.lq - m * kBM);
            const bool warp_rows = quarter * 32 < nq;
            const int ipos = m * kBM + r;        // query position in the sample
            const bool row_ok = r < nq;
            const bool windowed = prm.mask == GDPA_MASK_CAUSAL_WINDOW;
            float lse2 = 0.0f, drow = 0.0f;   // softmax variant: this row's statistics
            if constexpr (ACT == kSoftmax) {
                lse2 = lse_next == -INFINITY ? INFINITY : lse_next * kLog2e;   // no key: P = 0
                drow = d_next;
                if (m + 1 < u.m1) row_stats(m + 1, lse_next, d_next);
            }
            // fused RMSNorm: the keys are normalised; this row's scale c,
            // from the tile's raw Q, joins alpha (x = alpha c q . k_hat);
            // computed while S and dP are on the tensor core (their Q is in)
            float ci = 1.0f;
            if constexpr (NORM) {
                if (!wg_wait(&bars[C::kQFull + (i & 1)], (i >> 1) & 1, ab, 42)) return;
                ci = row_scale<D>(smem + C::kOffQ + (i & 1) * C::kTileBytes, r, prm.qk_gain,
                                  prm.qk_eps);
                ksc = act_scale<ACT>(prm.alpha * ci);
            }
            if (!wg_wait(&bars[C::kSDFull], i & 1, ab, 43)) return;
            // the previous tile's dQ bulk stores have long been issued: once
            // they have read their staging, its Q stage goes back to the
            // producer
            if (pending_q >= 0) {
                staging_release_wait(lane);
                mbar_arrive(&bars[C::kQEmpty + pending_q]);
                pending_q = -1;
            }
            // the shared buffer must be clear of the previous unit's dK, dV
            // drain by both warpgroups and of the previous tile's P (read by
            // its dV MMA) before dS goes in
            if (m == u.m0 && nu > 0 && !wg_wait(&bars[C::kPSFree], (nu - 1) & 1, ab, 47)) return;
            if (!wg_wait(&bars[C::kPVDone], (i & 1) ^ 1, ab, 44)) return;
            tc_fence_after();
            uint64_t gdot2 = f2_make(0.0f, 0.0f);   // sum_j dS_j s_j over this warpgroup's keys
            uint32_t pp[4][8];
            if (warp_rows) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int sidx = wg + 2 * k;
                    if (sidx < nh) {
                        const int col0 = sidx * 16;
                        // pd: dS (TMEM, the A operand of dQ = dS K); pq:
                        // dS for dK = dS^T Q, times the row's c when fused
                        // RMSNorm gives dK for the normalised keys
                        uint32_t sv[16], dv[16], pd[8], pq[8];
                        tmem_ld16(trow + kColS + col0, sv);
                        tmem_ld16(trow + kColDP + col0, dv);
                        tmem_ld_wait();
                        const bool full = !windowed && col0 + 16 <= u.nkv;
                        if (!row_ok) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) pp[k][e] = pd[e] = pq[e] = 0u;
                        } else {
                            // one body for whole and ragged steps: the masks
                            // only where the step is not entirely valid
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                float p2[2], d2[2];
                                bwd_p_ds2<ACT>(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1]),
                                               __uint_as_float(dv[e]), __uint_as_float(dv[e + 1]),
                                               ksc, lse2, drow, p2[0], p2[1], d2[0], d2[1]);
                                if (!full) {
#pragma unroll
                                    for (int w = 0; w < 2; ++w) {
                                        const int col = col0 + e + w;
                                        const int jpos = u.c0 + col;
                                        bool valid = col < u.nkv;
                                        if (windowed)
                                            valid = valid && jpos <= ipos && jpos > ipos - prm.window;
                                        p2[w] = valid ? p2[w] : 0.0f;
                                        d2[w] = valid ? d2[w] : 0.0f;
                                    }
                                }
                                pp[k][e >> 1] = pack_bf16x2(p2[0], p2[1]);
                                pd[e >> 1] = pack_bf16x2(d2[0], d2[1]);
                                if constexpr (NORM) {
                                    const uint64_t dd = f2_make(d2[0], d2[1]);
                                    const float2 q2 = f2_split(f2_mul(dd, f2_make(ci, ci)));
                                    pq[e >> 1] = pack_bf16x2(q2.x, q2.y);
                                    gdot2 = f2_fma(dd,
                                                   f2_make(__uint_as_float(sv[e]),
                                                           __uint_as_float(sv[e + 1])),
                                                   gdot2);
                                }
                            }
                        }
                        if constexpr (NORM) {
                            store_half_chunk(ps, sidx >> 1, sidx & 1, r, pq);
                            tmem_st8(trow + kColS + col0, pd);
                        } else {
                            store_half_chunk(ps, sidx >> 1, sidx & 1, r, pd);
                            // and packed into the step's own S columns
                            // (already read), the A operand of dQ = dS K
                            tmem_st8(trow + kColS + col0, pd);
                        }
                    }
                }
                tmem_st_wait();
            }
            if constexpr (NORM) {   // this warpgroup's share of the row dot
                const float2 g2 = f2_split(gdot2);
                reinterpret_cast<float*>(smem + C::kOffDot)[wg * 128 + r] = g2.x + g2.y;
                mbar_arrive(&bars[C::kDotFull]);
            }
            tc_fence_before();
            mbar_arrive(&bars[C::kSFree]);
            fence_proxy_async_smem();
            mbar_arrive(&bars[C::kDSFull]);
            // P -> shared once dK += dS^T Q has read dS
            if (!wg_wait(&bars[C::kDKDone], i & 1, ab, 45)) return;
            if (warp_rows) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int sidx = wg + 2 * k;
                    if (sidx < nh) store_half_chunk(ps, sidx >> 1, sidx & 1, r, pp[k]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[C::kPFull]);
            // dQ tile, d columns [64 wg, 64 wg + 64): TMEM -> this warpgroup's
            // half of the tile's Q buffer (its MMAs are done) -> global
            if (!wg_wait(&bars[C::kDQDone], i & 1, ab, 48)) return;
            tc_fence_after();
            float* dq = prm.dQ + (int64_t)(dq_row0 + m * kBM) * rs + h * D;
            uint8_t* dq_stage = smem + C::kOffQ + (i & 1) * C::kTileBytes + wg * kHalfBytes;
            if constexpr (NORM) {
                if (D == 128 || wg == 0) {
                    if (!wg_wait(&bars[C::kDotFull], i & 1, ab, 49)) return;
                    const float* dotx = reinterpret_cast<const float*>(smem + C::kOffDot);
                    drain_dq_norm<D>(trow, wg, r, smem + C::kOffQ + (i & 1) * C::kTileBytes,
                                     dotx[r] + dotx[128 + r], dq_stage, tmDQ,
                                     h * D + 64 * wg, dq_row0 + m * kBM, dq + 64 * wg, rs, nq,
                                     atomic_dq, prm.alpha, ci, prm.qk_gain, quarter, lane,
                                     &bars[C::kDQFree]);
                } else {
                    tc_fence_before();
                    mbar_arrive(&bars[C::kDQFree]);
                }
            } else if (D == 128 || wg == 0) {
                drain_warp(trow, kColDP + 64 * wg, 64, dq_stage, tmDQ, h * D + 64 * wg,
                           dq_row0 + m * kBM, dq + 64 * wg, rs, nq, atomic_dq, prm.alpha, quarter,
                           lane, &bars[C::kDQFree]);
            } else {
                tc_fence_before();
                mbar_arrive(&bars[C::kDQFree]);
            }
            pending_q = (int)(i & 1);
        }
        // the unit's dV (warpgroup 0) and dK (warpgroup 1)
        if (!wg_wait(&bars[C::kAccFull], nu & 1, ab, 46)) return;
        tc_fence_after();
        if (pending_q >= 0) {
            staging_release_wait(lane);
            mbar_arrive(&bars[C::kQEmpty + pending_q]);
            pending_q = -1;
        }
        {
            float* dst = (wg == 0 ? prm.dV : prm.dK) + (int64_t)u.kvt0 * rs + h * D;
            if (NORM && wg == 1) {
                const float cj = r < u.nkv ? __ldg(prm.kscale + (int64_t)h * prm.kscale_ld + u.kvt0 + r)
                                           : 0.0f;
                drain_dk_norm<D>(trow, r, smem + C::kOffK, stage, tmDK, h * D, u.kvt0, dst, rs,
                                 u.nkv, prm.alpha, cj, prm.qk_gain, quarter, lane,
                                 &bars[C::kKVEmpty], &bars[C::kAccFree]);
            } else if (NORM) {   // dV, with the norm's 16-column tensor maps
                drain_warp16(trow, kColDV, D, stage, tmDV, h * D, u.kvt0, dst, rs, u.nkv, false,
                             1.0f, quarter, lane, &bars[C::kAccFree]);
            } else {
                drain_warp(trow, wg == 0 ? kColDV : kColDK, D, stage, wg == 0 ? tmDV : tmDK, h * D,
                           u.kvt0, dst, rs, u.nkv, false, wg == 0 ? 1.0f : prm.alpha, quarter,
                           lane, &bars[C::kAccFree]);
            }
            staging_release_wait(lane);
            mbar_arrive(&bars[C::kPSFree]);
        }
        ++nu;
    }
}

template <int D, int ACT, bool NORM>
__global__ void __launch_bounds__(kThreads, 1)
tc_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
              const __grid_constant__ CUtensorMap tmDV, const BwdParams prm) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg0 = prm.seg[blockIdx.x], seg1 = prm.seg[blockIdx.x + 1];
    uint64_t t_start = 0;
    if (threadIdx.x == 0) {
        t_start = globaltimer();
        const uint32_t counts[C::kNumBars] = {
            1, NORM ? 128u : 1u,  // kv full / empty (fused RMSNorm: warpgroup 1 after dK)
            1, 1, 256, 256,       // q full x2, q empty x2 (warpgroups, after dQ staging)
            1, 1, 1, 1,           // dO full x2, dO empty x2
            1, 256, 256,          // sd full, s free, dq free
            256, 1, 256, 1,       // p full, pv done, ds full, dk done
            1, 256, 128, 128,     // acc full, acc free, stage x2
            256, 1,               // ps free, mma done
            1, 256                // dq done, row dots written (fused RMSNorm)
        };
        for (int b = 0; b < C::kNumBars; ++b) mbar_init(&bars[b], counts[b]);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO);
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, prm.err, prm.wait_ns};

    if (warp == 0) {
        if (lane == 0) bwd_producer<D>(&tmQ, &tmK, &tmV, &tmDO, prm, smem, bars, seg0, seg1, ab);
        __syncwarp();
    } else if (warp == 1) {
        bwd_mma<D>(prm, smem, bars, tmem, seg0, seg1, ab);   // the whole warp
        __syncwarp();
    } else {
        bwd_compute<D, ACT, NORM>(prm, &tmDQ, &tmDK, &tmDV, smem, bars, tmem, seg0, seg1, ab);
        // every bulk store of this warp has landed before the CTA retires
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
        prm.times[2 * (gridDim.x + blockIdx.x)] = t_start;
        prm.times[2 * (gridDim.x + blockIdx.x) + 1] = globaltimer();
        prm.smid[gridDim.x + blockIdx.x] = (int32_t)smid();
    }
}

template <int D, int ACT, bool NORM>
gdpa_status launch1(Plan& p, const CUtensorMap* maps, const BwdParams& prm, cudaStream_t st) {
    using C = BwdCfg<D>;
    auto kern = tc_bwd_kernel<D, ACT, NORM>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
        return GDPA_ERR_CUDA;
    kern<<<p.S, kThreads, C::kSmemBytes, st>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                maps[5], maps[6], prm);
    p.launches += 1;
    return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

template <int D, int ACT>
gdpa_status launch(Plan& p, const CUtensorMap* maps, const BwdParams& prm, cudaStream_t st) {
    return prm.kscale ? launch1<D, ACT, true>(p, maps, prm, st)
                      : launch1<D, ACT, false>(p, maps, prm, st);
}

}  // namespace

gdpa_status launch_tc_bwd(Plan& p, const void* q, const void* k, const void* v, const void* d_o,
                          float* dq, float* dk, float* dv, float alpha, int act, const float* lse,
                          const float* delta, cudaStream_t st) {
    if (p.d != 64 && p.d != 128) return GDPA_ERR_UNSUPPORTED;
    const uint64_t row = (uint64_t)p.H * p.d;
    const bool shared = p.shared_q > 0;
    // dQ rows: the tokens', or the shared seeds' (a sum over samples)
    const int64_t dq_rows = shared ? p.shared_q : p.Tq;
    if ((p.zero_dq || shared) && dq_rows > 0) {
        if (cudaMemsetAsync(dq, 0, (size_t)dq_rows * row * sizeof(float), st) != cudaSuccess)
            return GDPA_ERR_CUDA;
    }
    if (p.n_bwd == 0) return GDPA_OK;
    if (p.qk_gain > 0.0f) {   // fused RMSNorm: the normalised keys first
        gdpa_status ks;
        k = plan_key_norm(p, k, st, &ks);
        if (ks != GDPA_OK) return ks;
    }
    CUtensorMap maps[7];
    // the fused RMSNorm's drains stage 16 columns at a time
    const uint32_t norm_cols = p.qk_gain > 0.0f ? 16 : 32;
    const uint64_t q_rows = p.Tq > 0 ? (uint64_t)p.Tq : 1;
    const uint64_t qt_rows = dq_rows > 0 ? (uint64_t)dq_rows : 1;   // Q and dQ tensors
    const void* qp = p.Tq > 0 ? q : k;
    const void* dop = p.Tq > 0 ? d_o : k;
    if (!tc::make_tmap_bf16(&maps[0], qp, qt_rows, row, 128) ||
        !tc::make_tmap_bf16(&maps[1], k, (uint64_t)p.Tkv, row, 128) ||
        !tc::make_tmap_bf16(&maps[2], v, (uint64_t)p.Tkv, row, 128) ||
        !tc::make_tmap_bf16(&maps[3], dop, q_rows, row, 128) ||
        !tc::make_tmap_f32(&maps[4], p.Tq > 0 ? (const void*)dq : (const void*)dk, qt_rows, row, 32,
                           norm_cols) ||
        !tc::make_tmap_f32(&maps[5], dk, (uint64_t)p.Tkv, row, 32, norm_cols) ||
        !tc::make_tmap_f32(&maps[6], dv, (uint64_t)p.Tkv, row, 32, norm_cols))
        return GDPA_ERR_CUDA;
    BwdParams prm;
    prm.units = p.d_bwd;
    prm.seg = p.d_bwd_seg;
    prm.dQ = dq;
    prm.dK = dk;
    prm.dV = dv;
    prm.lse = lse;
    prm.delta = delta;
    prm.shared_q = shared ? 1 : 0;
    prm.H = p.H;
    prm.alpha = alpha;
    prm.mask = p.mask;
    prm.window = p.window;
    prm.err = p.d_err;
    prm.times = p.d_times;
    prm.smid = p.d_smid;
    prm.timing = p.timing;
    prm.wait_ns = tc::wait_limit_ns(p.wait_limit_us);
    prm.stall = p.stall;
    prm.kscale = p.qk_gain > 0.0f ? p.d_kscale : nullptr;
    prm.kscale_ld = p.Tkv + 128;
    prm.qk_gain = p.qk_gain;
    prm.qk_eps = p.qk_eps;
    if (p.timing) p.timed[1] = 1;
    gdpa_status s = GDPA_OK;
    if (p.d == 128) {
        if (act == kSoftmax)
            s = launch<128, kSoftmax>(p, maps, prm, st);
        else
            GDPA_DISPATCH_ACT(act, A, s = launch<128, A>(p, maps, prm, st))
    } else {
        if (act == kSoftmax)
            s = launch<64, kSoftmax>(p, maps, prm, st);
        else
            GDPA_DISPATCH_ACT(act, A, s = launch<64, A>(p, maps, prm, st))
    }
    return s;
}

}  // namespace gdpa
