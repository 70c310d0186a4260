// TMEM -> global drain of fp32 accumulators, shared by the tensor-core
// kernels (the backward's dQ, dK, dV; the forward's partial O of key-split
// tiles).
#pragma once

#include "tc_common.cuh"

namespace gdpa {
namespace tc {

// four accumulator words times `sc2` (the scale in both halves), in pairs
__device__ __forceinline__ float4 scaled4(const uint32_t* v, uint64_t sc2) {
    const float2 lo = f2_split(f2_mul(sc2, f2_make(__uint_as_float(v[0]), __uint_as_float(v[1]))));
    const float2 hi = f2_split(f2_mul(sc2, f2_make(__uint_as_float(v[2]), __uint_as_float(v[3]))));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Drain TMEM columns [col, col + ncols) (a multiple of 32) of this warp's
// 32 lanes (block rows 32 * quarter + lane) into rows [0, nrows) of a block
// of a [rows][H * d] fp32 tensor whose first element has tensor-map
// coordinates (x0, y0) and address `dst` (row stride `rs` floats), scaled by
// `scale`.  A warp whose 32 rows are all inside the block stages 32 columns
// at a time in its own 4 KB of `stage` (128-byte rows, 16-byte chunks
// swizzled by row, the layout of a 128-byte-swizzled TMA box: the tensor
// map's box is [32][32]) and writes them with one TMA bulk store, or a bulk
// reduce-add when `atomic`; the warp
// holding the block's ragged end writes its valid rows from registers.
// `release` (if any) is arrived by every thread after its last TMEM read.
// On return the last bulk store may still be reading the staging area: call
// staging_release_wait before it is reused.
__device__ __forceinline__ void drain_warp_inl(uint32_t trow, uint32_t col, int ncols,
                                               uint8_t* stage, const CUtensorMap* map, int x0,
                                               int y0, float* dst, int64_t rs, int nrows,
                                               bool atomic, float scale, int quarter, int lane,
                                               uint64_t* release) {
    const int row0 = quarter * 32;
    const bool any = row0 < nrows;
    const bool full = row0 + 32 <= nrows;
    uint8_t* wst = stage + quarter * 4096;
    const uint64_t sc2 = f2_make(scale, scale);
    for (int pass = 0; pass < ncols / 32; ++pass) {
        uint32_t v[32];
        if (any) {
            tmem_ld32(trow + col + pass * 32, v);
            tmem_ld_wait();
        }
        if (pass == ncols / 32 - 1 && release) {
            tc_fence_before();
            mbar_arrive(release);
        }
        if (!any) continue;
        if (full) {
            if (pass > 0) {
                if (lane == 0) bulk_wait_read_all();
                __syncwarp();
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<float4*>(wst + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                    scaled4(v + 4 * c, sc2);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (atomic)
                    tma_reduce_add_2d(map, wst, x0 + pass * 32, y0 + row0);
                else
                    tma_store_2d(map, wst, x0 + pass * 32, y0 + row0);
                bulk_commit();
            }
        } else if (row0 + lane < nrows) {
            float* d = dst + (int64_t)(row0 + lane) * rs + pass * 32;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 w = scaled4(v + 4 * c, sc2);
                if (atomic)
                    atomicAdd(reinterpret_cast<float4*>(d + 4 * c), w);
                else
                    *reinterpret_cast<float4*>(d + 4 * c) = w;
            }
        }
    }
}

// Byte offset of 16-byte chunk c of staging row `lane` in the 64-byte-
// swizzled layout of a [32][16] fp32 TMA box (2 KB, 512-byte aligned).
__device__ __forceinline__ uint32_t stage_off64(int lane, int c) {
    return (uint32_t)(lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
}

// drain_warp_inl in steps of 16 columns (ncols a multiple of 16): a full
// warp stages each step in one of the two 2 KB halves of its 4 KB of
// `stage`, alternately, with the [32][16] box of a 64-byte-swizzled tensor
// map, rewriting a half only once the store issued from it two steps
// earlier has read it, so that no step waits for the one before.  More bulk
// operations than drain_warp_inl, fewer registers; otherwise the same.
__device__ __forceinline__ void drain_warp16_inl(uint32_t trow, uint32_t col, int ncols,
                                               uint8_t* stage, const CUtensorMap* map, int x0,
                                               int y0, float* dst, int64_t rs, int nrows,
                                               bool atomic, float scale, int quarter, int lane,
                                               uint64_t* release) {
    const int row0 = quarter * 32;
    const bool any = row0 < nrows;
    const bool full = row0 + 32 <= nrows;
    uint8_t* wst = stage + quarter * 4096;
    const uint64_t sc2 = f2_make(scale, scale);
    for (int pass = 0; pass < ncols / 16; ++pass) {
        uint32_t v[16];
        if (any) {
            tmem_ld16(trow + col + pass * 16, v);
            tmem_ld_wait();
        }
        if (pass == ncols / 16 - 1 && release) {
            tc_fence_before();
            mbar_arrive(release);
        }
        if (!any) continue;
        if (full) {
            uint8_t* buf = wst + (pass & 1) * 2048;
            if (pass >= 2) {
                if (lane == 0) bulk_wait_read_but1();
                __syncwarp();
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<float4*>(buf + stage_off64(lane, c)) =
                    scaled4(v + 4 * c, sc2);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (atomic)
                    tma_reduce_add_2d(map, buf, x0 + pass * 16, y0 + row0);
                else
                    tma_store_2d(map, buf, x0 + pass * 16, y0 + row0);
                bulk_commit();
            }
        } else if (row0 + lane < nrows) {
            float* d = dst + (int64_t)(row0 + lane) * rs + pass * 16;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 w = scaled4(v + 4 * c, sc2);
                if (atomic)
                    atomicAdd(reinterpret_cast<float4*>(d + 4 * c), w);
                else
                    *reinterpret_cast<float4*>(d + 4 * c) = w;
            }
        }
    }
}

// Out-of-line form, for kernels that drain from several places.
static __device__ __noinline__ void drain_warp(uint32_t trow, uint32_t col, int ncols, uint8_t* stage,
                                           const CUtensorMap* map, int x0, int y0, float* dst,
                                           int64_t rs, int nrows, bool atomic, float scale,
                                           int quarter, int lane, uint64_t* release) {
    drain_warp_inl(trow, col, ncols, stage, map, x0, y0, dst, rs, nrows, atomic, scale, quarter,
                   lane, release);
}

static __device__ __noinline__ void drain_warp16(uint32_t trow, uint32_t col, int ncols,
                                             uint8_t* stage, const CUtensorMap* map, int x0,
                                             int y0, float* dst, int64_t rs, int nrows,
                                             bool atomic, float scale, int quarter, int lane,
                                             uint64_t* release) {
    drain_warp16_inl(trow, col, ncols, stage, map, x0, y0, dst, rs, nrows, atomic, scale, quarter,
                     lane, release);
}

// The calling warp's bulk stores have read their staging: the area may be
// reused or handed back.
__device__ __forceinline__ void staging_release_wait(int lane) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
}

}  // namespace tc
}  // namespace gdpa
