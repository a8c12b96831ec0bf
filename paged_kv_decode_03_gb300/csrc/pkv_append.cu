// pkv_append.cu -- write the step's new K/V rows into their pool slots,
// copying bf16 or quantising to int8, optionally after rotating q and k by
// their positions (RoPE fused with the append).
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
#include "pkv_write.h"

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

// Store one token's row ([H_kv][D] bf16, 16-byte vectors, global or shared
// memory) into its pool slot: a bit copy, or int8 codes under the token's
// scale (per token: max|x| / 127 of this row, written at scale[slot]) or the
// static per-head scales.  Every thread of the block calls it.
template <bool INT8>
__device__ __forceinline__ void store_row(const AppendParams &p, const uint4 *src, int which,
                                          int64_t slot, float *red)
{
    const int nvec = p.row / 8;  // 8 elements per vector
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
    for (int which = 0; which < (p.alias ? 1 : 2); ++which)
        store_row<INT8>(p, reinterpret_cast<const uint4 *>((which ? p.v : p.k) +
                                                           static_cast<int64_t>(t) * p.row),
                        which, slot, red);
}

// ---------------------------------------------------------------- RoPE
// Rotary position embedding (RoFormer, Su et al., section 3.2 and the
// element-wise form of section 3.4.2; p-RoPE, Barbero et al., "Round and
// Round We Go!", keeps only the first rotary_pairs frequencies): pair i of a
// vector at position m turns by m * theta_i,
//     a' = a cos - b sin,  b' = a sin + b cos.
// The table holds fp32(cos), fp32(sin) of the fp64 angle; the rotation is
// t = b * s, a' = fma(a, c, -t), t = b * c, b' = fma(a, s, t) in fp32, each
// rounded once to bf16 (nearest even) -- the precision the API states, so
// that the stored bf16 bits (and int8 codes) are fixed by it.

// table[m * pairs + i] = (cos, sin) of m * theta[i]; grid-stride.
__global__ void rope_table_kernel(const double *theta, int pairs, int64_t total, float2 *table)
{
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = e / pairs;
        const int i = static_cast<int>(e - m * pairs);
        const double ang = static_cast<double>(m) * theta[i];
        double sn, cs;
        sincos(ang, &sn, &cs);
        table[e] = make_float2(__double2float_rn(cs), __double2float_rn(sn));
    }
}

__device__ __forceinline__ void rotate_pair(float a, float b, float2 cs, float &ap, float &bp)
{
    const float t1 = __fmul_rn(b, cs.y);
    ap = __fmaf_rn(a, cs.x, -t1);
    const float t2 = __fmul_rn(b, cs.x);
    bp = __fmaf_rn(a, cs.y, t2);
}

// Two bf16 of a word: the rounded value where the element turned, the input
// bits where it did not (so unrotated dims pass bit for bit, NaNs included).
__device__ __forceinline__ uint32_t repack(uint32_t orig, float lo, float hi, bool rlo, bool rhi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    const uint32_t w = *reinterpret_cast<const uint32_t *>(&h);
    return ((rlo ? w : orig) & 0xffffu) | ((rhi ? w : orig) & 0xffff0000u);
}

// Rotate rows of `heads` vectors of head_dim bf16 from src to dst (global or
// shared; dst may be src), 8-element vectors per thread step.  Halves layout:
// a step takes dims [8v, 8v + 8) and their partners D/2 further; interleaved:
// a step takes dims [8v, 8v + 8), four pairs.
__device__ __forceinline__ void rotate_rows(const uint16_t *src, uint16_t *dst, int heads,
                                            int head_dim, const float2 *cs, int pairs,
                                            int layout)
{
    const int half = head_dim / 2;
    if (layout == PKV_ROPE_HALVES) {
        const int per_head = half / 8;
        for (int w = threadIdx.x; w < heads * per_head; w += blockDim.x) {
            const int h = w / per_head, v = w - h * per_head;
            const int64_t ea = static_cast<int64_t>(h) * head_dim + v * 8;
            const uint4 xa = *reinterpret_cast<const uint4 *>(src + ea);
            const uint4 xb = *reinterpret_cast<const uint4 *>(src + ea + half);
            float a[8], b[8];
            unpack8(xa, a);
            unpack8(xb, b);
            const int i0 = v * 8;  // pair index of element 0
            if (i0 >= pairs) {     // nothing turns in this step
                if (dst != src) {
                    *reinterpret_cast<uint4 *>(dst + ea) = xa;
                    *reinterpret_cast<uint4 *>(dst + ea + half) = xb;
                }
                continue;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (i0 + e < pairs)
                    rotate_pair(a[e], b[e], cs[i0 + e], a[e], b[e]);
            bool r[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                r[e] = i0 + e < pairs;
            *reinterpret_cast<uint4 *>(dst + ea) =
                make_uint4(repack(xa.x, a[0], a[1], r[0], r[1]), repack(xa.y, a[2], a[3], r[2], r[3]),
                           repack(xa.z, a[4], a[5], r[4], r[5]), repack(xa.w, a[6], a[7], r[6], r[7]));
            *reinterpret_cast<uint4 *>(dst + ea + half) =
                make_uint4(repack(xb.x, b[0], b[1], r[0], r[1]), repack(xb.y, b[2], b[3], r[2], r[3]),
                           repack(xb.z, b[4], b[5], r[4], r[5]), repack(xb.w, b[6], b[7], r[6], r[7]));
        }
    } else {
        const int per_head = head_dim / 8;
        for (int w = threadIdx.x; w < heads * per_head; w += blockDim.x) {
            const int h = w / per_head, v = w - h * per_head;
            const int64_t ea = static_cast<int64_t>(h) * head_dim + v * 8;
            const uint4 x = *reinterpret_cast<const uint4 *>(src + ea);
            float f[8];
            unpack8(x, f);
            const int i0 = v * 4;  // pair index of elements 0 and 1
            if (i0 >= pairs) {
                if (dst != src)
                    *reinterpret_cast<uint4 *>(dst + ea) = x;
                continue;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (i0 + e < pairs)
                    rotate_pair(f[2 * e], f[2 * e + 1], cs[i0 + e], f[2 * e], f[2 * e + 1]);
            const bool r0 = i0 < pairs, r1 = i0 + 1 < pairs, r2 = i0 + 2 < pairs,
                       r3 = i0 + 3 < pairs;
            *reinterpret_cast<uint4 *>(dst + ea) =
                make_uint4(repack(x.x, f[0], f[1], r0, r0), repack(x.y, f[2], f[3], r1, r1),
                           repack(x.z, f[4], f[5], r2, r2), repack(x.w, f[6], f[7], r3, r3));
        }
    }
}

// One CTA per token: its v row stored as is (while the table row loads), its
// q rows rotated into q_out, its k row rotated into shared memory and stored
// into the pool from there.
// A negative position is padding (q copied, nothing appended); a position
// past the table is reported (PKV_DEV_BAD_POSITION) and treated the same.
template <bool INT8>
__global__ void __launch_bounds__(APPEND_THREADS) append_rope_kernel(const AppendParams p,
                                                                     const RopeParams r)
{
    extern __shared__ __align__(16) uint8_t rope_sm[];
    __shared__ float red[APPEND_THREADS / 32];
    float2 *cs = reinterpret_cast<float2 *>(rope_sm);                        // [pairs]
    uint16_t *krow = reinterpret_cast<uint16_t *>(rope_sm + ((r.pairs * 8 + 15) & ~15));  // [row]
    const int t = blockIdx.x;
    const int64_t qrow = static_cast<int64_t>(r.num_q_heads) * p.head_dim;
    {
        // the token's q, k and v rows do not depend on its position: start
        // bringing them into L2 while the position and the table row load
        const char *rows[3] = {r.q ? reinterpret_cast<const char *>(r.q + t * qrow) : nullptr,
                               reinterpret_cast<const char *>(p.k + static_cast<int64_t>(t) * p.row),
                               p.alias ? nullptr
                                       : reinterpret_cast<const char *>(p.v + static_cast<int64_t>(t) * p.row)};
        const int64_t bytes[3] = {qrow * 2, static_cast<int64_t>(p.row) * 2,
                                  static_cast<int64_t>(p.row) * 2};
#pragma unroll
        for (int j = 0; j < 3; ++j)
            if (rows[j])
                for (int64_t o = static_cast<int64_t>(threadIdx.x) * 128; o < bytes[j];
                     o += static_cast<int64_t>(blockDim.x) * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(rows[j] + o));
    }
    const int64_t m = r.positions ? r.positions[t] : static_cast<int64_t>(r.seq_lens[t]) - 1;
    const int64_t slot = p.slot_mapping[t];  // loaded beside the position
    const bool valid = m >= 0 && m < r.num_positions;
    if (m >= r.num_positions && threadIdx.x == 0)
        record_error(p.err, PKV_DEV_BAD_POSITION);
    const uint16_t *qs = r.q ? r.q + t * qrow : nullptr;
    uint16_t *qd = r.q ? r.q_out + t * qrow : nullptr;
    if (!valid) {
        if (qs && qd != qs)
            for (int i = threadIdx.x; i < qrow / 8; i += blockDim.x)
                reinterpret_cast<uint4 *>(qd)[i] = reinterpret_cast<const uint4 *>(qs)[i];
        return;
    }
    for (int i = threadIdx.x; i < r.pairs; i += blockDim.x)
        cs[i] = r.table[m * r.pairs + i];
    const bool store = slot >= 0 && slot < p.num_slots;  // uniform over the block
    if (slot >= p.num_slots && threadIdx.x == 0)
        record_error(p.err, PKV_DEV_BAD_SLOT);
    // v needs no rotation: its row goes first, while the table row lands
    if (store && !p.alias)
        store_row<INT8>(p, reinterpret_cast<const uint4 *>(p.v + static_cast<int64_t>(t) * p.row),
                        1, slot, red);
    __syncthreads();
    if (qs)
        rotate_rows(qs, qd, r.num_q_heads, p.head_dim, cs, r.pairs, r.layout);
    if (!store)
        return;
    rotate_rows(p.k + static_cast<int64_t>(t) * p.row, krow, p.row / p.head_dim, p.head_dim, cs,
                r.pairs, r.layout);
    __syncthreads();
    store_row<INT8>(p, reinterpret_cast<const uint4 *>(krow), 0, slot, red);
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

size_t append_rope_smem_bytes(int row, int pairs)
{
    return static_cast<size_t>((pairs * 8 + 15) / 16 * 16) + static_cast<size_t>(row) * 2;
}

cudaError_t launch_append_rope(const AppendParams &p, const RopeParams &r, int int8,
                               cudaStream_t s)
{
    if (p.num_tokens <= 0)
        return cudaSuccess;
    const size_t smem = append_rope_smem_bytes(p.row, r.pairs);
    auto kern = int8 ? append_rope_kernel<true> : append_rope_kernel<false>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess)
            return e;
    }
    kern<<<p.num_tokens, APPEND_THREADS, smem, s>>>(p, r);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_rope_table(const double *theta, int pairs, int64_t num_positions,
                              float *table, cudaStream_t s)
{
    const int64_t total = num_positions * pairs;
    if (total <= 0)
        return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
    rope_table_kernel<<<grid, threads, 0, s>>>(theta, pairs, total,
                                               reinterpret_cast<float2 *>(table));
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
