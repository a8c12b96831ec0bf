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

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
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
