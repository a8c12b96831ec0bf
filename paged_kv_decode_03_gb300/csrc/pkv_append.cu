// pkv_append.cu -- write the step's new K/V rows into their pool slots,
// copying bf16 or quantising to int8.
//
// Sources (page title, section): "CS336 · 第 10 课", KV-cache section (each
// decode step appends the new token's K/V) and int8 section
// (scale = max|x| / 127, x_q = round(x / scale)); "推理优化与 AI Infra",
// section 2 (pool [block][slot][head][dim]), section 5 (per_token or
// per_head scales) and section 8 (slot ids as a static step buffer).
//
// One CTA per token.  The token's row for all kv heads is contiguous in the
// pool ([slot][H_kv][D] with slot = block * 16 + offset), so the write is a
// straight vectorised copy.  Quantisation follows the fp32 formula exactly:
// IEEE division for the scale and for every element (no reciprocal),
// round-half-to-even, saturation to [-127, 127], zero scale -> zero codes.
#include <cuda_bf16.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int APPEND_THREADS = 128;

// Code of x under scale: round half to even, saturated to [-127, 127]; a
// zero scale gives 0, and so does a quotient that is not a number (a NaN
// input, or inf / inf when the token's scale is infinite).
__device__ __forceinline__ int8_t quantize_one(float x, float scale)
{
    if (scale == 0.f)
        return 0;
    const float y = __fdiv_rn(x, scale);
    if (y != y)
        return 0;
    int r = __float2int_rn(y);
    r = max(-127, min(127, r));
    return static_cast<int8_t>(r);
}

__device__ __forceinline__ void unpack8(const uint4 w, float *f)
{
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

__device__ __forceinline__ uint2 pack8(const int8_t *q)
{
    uint2 r;
    r.x = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) |
          ((uint32_t)(uint8_t)q[2] << 16) | ((uint32_t)(uint8_t)q[3] << 24);
    r.y = (uint32_t)(uint8_t)q[4] | ((uint32_t)(uint8_t)q[5] << 8) |
          ((uint32_t)(uint8_t)q[6] << 16) | ((uint32_t)(uint8_t)q[7] << 24);
    return r;
}

// Block-wide max of non-negative values; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float *red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, off));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        red[warp] = v;
    __syncthreads();
    float r = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
        r = fmaxf(r, red[w]);
    __syncthreads();
    return r;
}

template <bool INT8>
__global__ void __launch_bounds__(APPEND_THREADS) append_kernel(const AppendParams p)
{
    __shared__ float red[APPEND_THREADS / 32];
    const int t = blockIdx.x;
    const int64_t slot = p.slot_mapping[t];
    if (slot < 0)
        return;
    if (slot >= p.num_slots) {
        if (threadIdx.x == 0)
            record_error(p.err, PKV_DEV_BAD_SLOT);
        return;
    }
    const int nvec = p.row / 8;  // 8 elements per vector
    for (int which = 0; which < (p.alias ? 1 : 2); ++which) {
        const uint4 *src =
            reinterpret_cast<const uint4 *>((which ? p.v : p.k) + static_cast<int64_t>(t) * p.row);
        if constexpr (!INT8) {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(which ? p.pool_v : p.pool_k) +
                                                   slot * p.row);
            for (int i = threadIdx.x; i < nvec; i += blockDim.x)
                dst[i] = src[i];
        } else {
            uint2 *dst = reinterpret_cast<uint2 *>(static_cast<int8_t *>(which ? p.pool_v : p.pool_k) +
                                                   slot * p.row);
            float *tbl = which ? p.v_scale : p.k_scale;
            float scale = 0.f;
            if (p.scale_mode == PKV_SCALE_PER_TOKEN) {
                float amax = 0.f;
                for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
                    float f[8];
                    unpack8(src[i], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        amax = fmaxf(amax, fabsf(f[e]));
                }
                amax = block_max(amax, red);
                scale = __fdiv_rn(amax, 127.f);
                if (threadIdx.x == 0)
                    tbl[slot] = scale;
            }
            for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
                float f[8];
                unpack8(src[i], f);
                const float s = p.scale_mode == PKV_SCALE_PER_TOKEN ? scale : tbl[(i * 8) / p.head_dim];
                int8_t q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    q[e] = quantize_one(f[e], s);
                dst[i] = pack8(q);
            }
        }
    }
}

cudaError_t launch_append(const AppendParams &p, int int8, cudaStream_t s)
{
    if (p.num_tokens <= 0)
        return cudaSuccess;
    if (int8)
        append_kernel<true><<<p.num_tokens, APPEND_THREADS, 0, s>>>(p);
    else
        append_kernel<false><<<p.num_tokens, APPEND_THREADS, 0, s>>>(p);
    note_launch();
    return cudaGetLastError();
}

// Slot of each token under the pool's layout: entry pos / 16 of the
// sequence's table row (paged) or entry (pos mod W) / 16 of its ring
// (W = ring_blocks * 16), offset pos % 16; -1 for padding (negative
// position) or a table entry that names no block of the pool (reported).
__global__ void slot_mapping_kernel(const int32_t *block_table, int max_blocks, int ring_blocks,
                                    int num_blocks, const int32_t *seq_ids,
                                    const int64_t *positions, int num_tokens, int64_t *slots,
                                    unsigned int *err)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= num_tokens)
        return;
    const int64_t pos = positions[i];
    int64_t slot = -1;
    if (pos >= 0) {
        const int64_t seq = seq_ids ? seq_ids[i] : i;
        const int64_t r = ring_blocks > 0 ? pos % (static_cast<int64_t>(ring_blocks) * kBlock) : pos;
        const int64_t entry = r / kBlock;
        const int32_t phys = entry < max_blocks ? block_table[seq * max_blocks + entry] : -1;
        if (phys >= 0 && phys < num_blocks)
            slot = static_cast<int64_t>(phys) * kBlock + r % kBlock;
        else
            record_error(err, PKV_DEV_BAD_BLOCK);
    }
    slots[i] = slot;
}

cudaError_t launch_slot_mapping(const int32_t *block_table, int max_blocks, int ring_blocks,
                                int num_blocks, const int32_t *seq_ids, const int64_t *positions,
                                int num_tokens, int64_t *slots, unsigned int *err, cudaStream_t s)
{
    const int threads = 256;
    slot_mapping_kernel<<<(num_tokens + threads - 1) / threads, threads, 0, s>>>(
        block_table, max_blocks, ring_blocks, num_blocks, seq_ids, positions, num_tokens, slots,
        err);
    note_launch();
    return cudaGetLastError();
}

// The pipelines' bounded waits, run out on purpose: every thread waits on
// an mbarrier phase that nothing completes, with the same wait functions the
// decode kernels use (sleeping and polling), and must give up after
// limit_ns, record PKV_DEV_TIMEOUT and return.  out[threadIdx.x] = 1 if that
// thread's wait returned false.
__global__ void bounded_wait_kernel(uint64_t limit_ns, int spin, int *out, unsigned int *err)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival would complete the phase; none comes
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = spin ? mbar_wait_spin(&bar, 0, err, limit_ns) : mbar_wait(&bar, 0, err, limit_ns);
    out[threadIdx.x] = ok ? 0 : 1;
}

cudaError_t launch_bounded_wait(uint64_t limit_ns, int spin, int *out, int threads,
                                unsigned int *err, cudaStream_t s)
{
    bounded_wait_kernel<<<1, threads, 0, s>>>(limit_ns, spin, out, err);
    note_launch();
    return cudaGetLastError();
}

}  // namespace pkv
