// Blackwell (sm_100-family, built for sm_103a) primitives used by the GDPA
// tensor-core kernels, as inline PTX: mbarriers with bounded waits, TMA 2-D
// tile loads, tcgen05 TMEM allocation / MMA / commit / load, and the shared
// memory and instruction descriptors of tcgen05.mma kind::f16.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "f2.cuh"
#include "gdpa_internal.h"

namespace gdpa {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smid() {
    uint32_t s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Every wait of the tensor-core kernels is bounded: after the CTA's limit
// (kWaitLimitNs unless the plan's failure-path test hook set a shorter one)
// or kWaitLimitIters polls it records a timeout in the plan's error word,
// raises the CTA's abort flag and returns false; the caller then unwinds.
// A raised abort flag (another role gave up) also ends the wait.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitLimitIters = 1u << 30;

struct Abort {
    volatile int* flag;   // shared memory, per CTA
    int32_t* err;         // global error word (code, where, cta, detail)
    uint64_t limit_ns;    // wait limit
};

// The wait limit of a launch: `limit_us` > 0 from the test hook, else the
// default.
__host__ __device__ constexpr uint64_t wait_limit_ns(uint32_t limit_us) {
    return limit_us > 0 ? (uint64_t)limit_us * 1000ull : kWaitLimitNs;
}

__device__ __forceinline__ void raise_error(const Abort& ab, int32_t code, int32_t where) {
    if (atomicCAS(ab.err, 0, code) == 0) {
        ab.err[1] = where;
        ab.err[2] = (int32_t)blockIdx.x;
    }
    *ab.flag = 1;
}

__device__ __forceinline__ bool mbar_wait_slow_inl(uint64_t* bar, uint32_t parity, const Abort& ab,
                                                  int32_t where) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*ab.flag) return false;
            if (globaltimer() - t0 > ab.limit_ns || it > kWaitLimitIters) {
                raise_error(ab, kDevTimeout, where);
                return false;
            }
        }
    }
}

// Out-of-line form: smaller code where registers are not scarce.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const Abort& ab,
                                                   int32_t where) {
    return mbar_wait_slow_inl(bar, parity, ab, where);
}

// kInline: the slow path inlined (no call, so no registers saved around it;
// for kernels that hold many live values across their waits).
template <bool kInline = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Abort& ab,
                                          int32_t where) {
    if (mbar_try_wait(bar, parity)) return true;
    if constexpr (kInline)
        return mbar_wait_slow_inl(bar, parity, ab, where);
    else
        return mbar_wait_slow(bar, parity, ab, where);
}

// bounded wait used while unwinding (ignores the abort flag)
__device__ __forceinline__ bool mbar_wait_teardown(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0; it < kWaitLimitIters; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 31u && globaltimer() - t0 > kWaitLimitNs / 4) return false;
    }
    return false;
}

// ---------------------------------------------------------------- fences

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tile load global -> shared, completion counted in bytes on `bar`.
// x (innermost, elements) * sizeof(element) must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2-D tile prefetch global -> L2 (no shared memory written, no completion to
// wait for): a later tma_load_2d of the same box hits in L2.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y,
                                                uint64_t policy) {
    asm volatile(
        "cp.async.bulk.prefetch.tensor.2d.L2.global.tile.L2::cache_hint [%0, {%1, %2}], %3;" ::"l"(map),
        "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// 2-D tile store shared -> global (bulk-group completion); x * 4 bytes (fp32)
// must be a multiple of 16 and no coordinate may be negative.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            map),
        "r"(x), "r"(y), "r"(smem_u32(src))
        : "memory");
}

// Same with an L2 eviction-priority hint for the written lines.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, const void* src,
                                                  int32_t x, int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
        " [%0, {%1, %2}], [%3], %4;" ::"l"(map),
        "r"(x), "r"(y), "r"(smem_u32(src)), "l"(policy)
        : "memory");
}

// Same, adding into global memory element-wise (f32 add, atomic per element).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src,
                                                  int32_t x, int32_t y) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%1, %2}], [%3];" ::"l"(map),
        "r"(x), "r"(y), "r"(smem_u32(src))
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ... all but the most recent group
__device__ __forceinline__ void bulk_wait_read_but1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// this thread's bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- tcgen05

// Allocate `ncols` TMEM columns (whole warp); the address lands in *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// The MMA and commit wrappers below are warp-wide: every lane of the warp
// calls them, converged, and one elected lane (the lowest) issues the
// instruction.  Running the issue code on the whole warp keeps its operands
// warp-uniform; issuing from a one-lane branch instead was measured several
// times slower while other warps kept the scheduler busy.

// D[tmem] (+)= A[smem] * B[smem], kind::f16, one CTA.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16, one CTA.  A is K-major in
// TMEM: row m in lane m, two 16-bit elements per 32-bit column (lower half =
// lower k), so a K = 16 step reads 8 columns from `a_tmem`.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation the elected lane issued
// so far has completed (the same lane that issues the MMAs above).
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t gets lane (base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns from registers (thread t -> lane
// base + t).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
    uint32_t v;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr) : "memory");
    return v;
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1, swizzle mode 2
// (128-byte swizzle).
//   K-major SW128 (rows of 64 bf16 = 128 B, 8-row groups of 1024 B):
//     LBO unused (1), SBO = 1024.
//   MN-major SW128 (rows are K, 64 N-elements per 128 B row):
//     LBO = byte distance between 64-element N chunks, SBO = 1024.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // version
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}

// Advance of a descriptor's start-address field (16-byte units) for K step
// k (16 elements) of a 128-byte-swizzled tile stored as 64-element halves of
// 128 rows: K-major (k-th 32 bytes of the row, next half after 4 steps) and
// MN-major (16 rows of 128 bytes per step).  Adding it to a descriptor built
// for the tile's base keeps the other fields (addresses stay below 256 KB).
__host__ __device__ constexpr uint64_t kmajor_step(int k) {
    return (uint64_t)(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t mnmajor_step(int k) { return (uint64_t)((k * 2048) >> 4); }

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A MN-major, 16 B MN-major, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// A wait taken by every thread of a warp(group); warp-uniform result so
// that the .sync.aligned tcgen05 instructions after it run with whole warps.
template <bool kInline = false>
__device__ __forceinline__ bool wg_wait(uint64_t* bar, uint32_t parity, const Abort& ab,
                                        int32_t where) {
    return __all_sync(0xffffffffu, mbar_wait<kInline>(bar, parity, ab, where));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------- fused RMSNorm

// Fused RMSNorm: c = g / rms of row r of a [128 x D] bf16 tile of raw rows
// in shared memory (128-byte-swizzled halves of 64 columns, 16 KB each); the
// kernels fold it into alpha, x = alpha c q . k_hat with normalised keys.
template <int D>
__device__ __forceinline__ float row_scale(const uint8_t* tile, int r, float gain, float eps) {
    uint64_t ss2 = f2_make(0.0f, 0.0f);
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v =
                *reinterpret_cast<const uint4*>(tile + hf * 16384 + r * 128 + ((c ^ (r & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint64_t x2 = f2_bf16x2(w[u]);
                ss2 = f2_fma(x2, x2, ss2);
            }
        }
    }
    const float2 ss = f2_split(ss2);
    return gain / sqrtf((ss.x + ss.y) / (float)D + eps);
}

// Columns [c0, c0 + 32 n) of row r of the same tile layout, as packed bf16
// pairs (16 n words).
template <int N>
__device__ __forceinline__ void load_row_bf16(const uint8_t* tile, int r, int c0, uint32_t (&x)[16 * N]) {
#pragma unroll
    for (int q = 0; q < 4 * N; ++q) {
        const int c = c0 / 8 + q;   // 16-byte chunk (8 columns) within the row
        const uint4 v = *reinterpret_cast<const uint4*>(tile + (c >> 3) * 16384 + r * 128 +
                                                        (((c & 7) ^ (r & 7)) << 4));
        x[4 * q] = v.x;
        x[4 * q + 1] = v.y;
        x[4 * q + 2] = v.z;
        x[4 * q + 3] = v.w;
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }


// ---------------------------------------------------------------- host side

// Build a 2-D bf16 tensor map over a [rows][row_elems] row-major tensor with
// a [box_rows][64] box and 128-byte swizzle.  Returns false on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                    uint32_t box_rows);

// Same for fp32 with a [box_rows][box_cols] box: box_cols = 32 (128-byte
// rows, 128-byte swizzle: 16-byte chunk c of row r at position c ^ (r & 7))
// or 16 (64-byte rows, 64-byte swizzle: chunk c of row r at position
// c ^ ((r >> 1) & 3)); staging buffers 1024-byte aligned.
bool make_tmap_f32(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_elems,
                   uint32_t box_rows, uint32_t box_cols);

}  // namespace tc
}  // namespace gdpa
