// pkv_device.cuh -- device helpers shared by the library's kernels:
// mbarrier / TMA / bulk-copy wrappers (inline PTX for sm_103a), bf16 and
// int8 unpacking, the device error word and bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr unsigned FULL_MASK = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// Set bits in the device error word (PKV_DEV_*); its address is a kernel
// parameter (the word itself lives in pkv_abi.cu).
__device__ __forceinline__ void record_error(unsigned int *err, unsigned bits)
{
    atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA).
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// try_wait with a suspend-time hint: a waiting thread sleeps (up to the
// hint, 20 us) until the phase completes instead of spinning, which leaves
// issue slots to the warps that have work.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Non-blocking probe: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete.  Bounded: after
// about `limit_ns` nanoseconds the wait gives up, records PKV_DEV_TIMEOUT
// and returns false so that the caller can drain and exit.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned int *err,
                                          uint64_t limit_ns = 2000000000ull)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) {
            record_error(err, PKV_DEV_TIMEOUT);
            return false;
        }
    }
}

// Spinning variant of mbar_wait for the roles on a pipeline's critical path:
// try_wait without a suspend-time hint returns after a short, system-defined
// interval, so a completed phase is seen within that interval instead of
// after a wake-up from a longer sleep.  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_try_wait_short(uint64_t *bar, uint32_t parity)
{
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

__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity, unsigned int *err,
                                               uint64_t limit_ns = 2000000000ull)
{
    // the common case, a phase already complete, costs no timer read
    if (mbar_try_wait_short(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_short(bar, parity))
            return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) {
            record_error(err, PKV_DEV_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------ flags between CTAs
__device__ __forceinline__ void st_release_gpu(int *addr, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *addr)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

// Order this thread's completed async-proxy (bulk copy) global writes before
// its later generic accesses.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------- programmatic dependent launch
// Let the next kernel in the stream (launched with programmatic stream
// serialisation) start its prologue now.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the preceding kernel has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- TMA loads
// 3-D tiled tensor load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// 2-D tiled tensor load global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Untiled bulk copy shared -> global (16-byte aligned, size multiple of 16),
// tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the committed bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until the committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Untiled bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policy for data read exactly once per launch (the KV stream).
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for data read by every CTA of a group (kept in L2 if possible).
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------ exp2 approx
// ex2.approx.ftz.f32: hardware 2^x (relative error ~2^-22); ex2(-inf) = +0.
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ unpacking
// Two bf16 packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Four int8 packed in a 32-bit word -> floats (exact).
__device__ __forceinline__ void int8x4_to_float(uint32_t w, float *f)
{
    f[0] = static_cast<float>(static_cast<int8_t>(w & 0xff));
    f[1] = static_cast<float>(static_cast<int8_t>((w >> 8) & 0xff));
    f[2] = static_cast<float>(static_cast<int8_t>((w >> 16) & 0xff));
    f[3] = static_cast<float>(static_cast<int8_t>(w >> 24));
}

// Load N consecutive elements (bf16 or int8) from shared memory as floats.
// N*elem bytes is 2..16 and the address is aligned to that size.
template <int N, bool INT8>
__device__ __forceinline__ void load_row_chunk(const uint8_t *p, float (&f)[N])
{
    if constexpr (!INT8) {
        static_assert(N == 2 || N == 4 || N == 8, "bf16 chunk");
        if constexpr (N == 8) {
            uint4 w = *reinterpret_cast<const uint4 *>(p);
            f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
            f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
        } else if constexpr (N == 4) {
            uint2 w = *reinterpret_cast<const uint2 *>(p);
            f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
        } else {
            uint32_t w = *reinterpret_cast<const uint32_t *>(p);
            f[0] = bf16lo(w); f[1] = bf16hi(w);
        }
    } else {
        static_assert(N == 2 || N == 4 || N == 8, "int8 chunk");
        if constexpr (N == 8) {
            uint2 w = *reinterpret_cast<const uint2 *>(p);
            int8x4_to_float(w.x, f);
            int8x4_to_float(w.y, f + 4);
        } else if constexpr (N == 4) {
            uint32_t w = *reinterpret_cast<const uint32_t *>(p);
            int8x4_to_float(w, f);
        } else {
            uint16_t w = *reinterpret_cast<const uint16_t *>(p);
            f[0] = static_cast<float>(static_cast<int8_t>(w & 0xff));
            f[1] = static_cast<float>(static_cast<int8_t>(w >> 8));
        }
    }
}

}  // namespace pkv

namespace pkv {

// ------------------------------------------------------------ tcgen05
// Shared-memory matrix descriptor for tcgen05.mma (sm_100 family):
// start address, leading and stride byte offsets (all >> 4), descriptor
// version 1 at bits 46-47, swizzle mode at bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// The same with the 32-byte swizzle (mode 6): 16-byte chunk bit 4 of the
// address XOR address bit 7, i.e. rows of 32 bytes in 256-byte atoms.
__device__ __forceinline__ uint64_t umma_smem_desc_sw32(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 6ull << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16 with bf16 A and B and an
// fp32 accumulator: D format at bits 4-5 (1 = f32), A/B formats at bits
// 7-9 / 10-12 (1 = bf16), A/B major at bits 15/16 (1 = MN-major), N >> 3 at
// bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn_major,
                                                       bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
           ((static_cast<uint32_t>(M) >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The same with A read from TMEM (M rows = TMEM lanes, two 16-bit elements
// of consecutive K per 32-bit column; a_tmem = the first of K / 2 columns).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Arrive (once) on an mbarrier when all previously issued tcgen05.mma of
// this thread have completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// N consecutive fp32 columns (N = 2, 4, 8) of this thread's TMEM lane.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N])
{
    uint32_t r[N];
    if constexpr (N == 2) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1])
                     : "r"(taddr)
                     : "memory");
    } else if constexpr (N == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr)
                     : "memory");
    } else {
        static_assert(N == 8, "columns");
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
                     "tcgen05.wait::ld.sync.aligned;"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                       "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    }
#pragma unroll
    for (int i = 0; i < N; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Store N consecutive fp32 columns (N = 2, 4, 8 or 16) of this thread's
// TMEM lane and wait until the stores are done.
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const float (&v)[N])
{
    uint32_t r[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        r[i] = __float_as_uint(v[i]);
    if constexpr (N == 2) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};\n\t"
                     "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(r[0]), "r"(r[1])
                     : "memory");
    } else if constexpr (N == 4) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n\t"
                     "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                     "r"(r[2]), "r"(r[3])
                     : "memory");
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
                     "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                     "r"(r[7])
                     : "memory");
    } else {
        static_assert(N == 16, "columns");
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
            "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
            "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
            "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
            "r"(r[15])
            : "memory");
    }
}

// 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    // load and wait in one statement: the registers are not valid before
    // tcgen05.wait::ld, so nothing may read them in between
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

}  // namespace pkv

namespace pkv {

// Block-table entries of logical blocks first, first+1, ... of one
// sequence, read 32 at a time by a whole warp: lane j holds the entry of
// block first + base + j of the current chunk, the next chunk is fetched
// ahead, and entry i is shuffled out, so no iteration waits on a global
// load.  With a ring of `ring` blocks, logical block x lives in table entry
// x % ring (position t in slot t mod (ring * 16)); ring 0 is the paged
// layout, entry x.
struct TableCursor {
    const int32_t *row;
    int first, n, ring, cur, nxt;
    __device__ __forceinline__ int load(int i) const
    {
        int x = first + i;
        if (ring > 0)
            x %= ring;
        return __ldg(row + x);
    }
    __device__ __forceinline__ void init(const int32_t *r, int first_block, int count, int ring_blocks,
                                         int lane)
    {
        row = r;
        first = first_block;
        n = count;
        ring = ring_blocks;
        cur = lane < n ? load(lane) : -1;
        nxt = 32 + lane < n ? load(32 + lane) : -1;
    }
    // entry i (all lanes call with the same i, in increasing order)
    __device__ __forceinline__ int get(int i, int lane)
    {
        if ((i & 31) == 0 && i > 0) {
            cur = nxt;
            nxt = i + 32 + lane < n ? load(i + 32 + lane) : -1;
        }
        return __shfl_sync(FULL_MASK, cur, i & 31);
    }
};

}  // namespace pkv
