// pkv_combine.cu -- log-sum-exp combine of split-KV partial states.
//
// What is computed: the pages' online-softmax recurrence ("LLM推理优化底层原理"
// §3.1 step 2; "实验五：Gemma4 端到端推理优化", Flash Attention section) merges
// two partial states (m, l, o) into one; applied to the per-split states of
// a sequence it gives, with lse_s = m_s + ln l_s and o_s normalised,
//   L = max_s lse_s,  w_s = exp(lse_s - L),  out = sum_s w_s o_s / sum_s w_s.
//
// Design: one CTA of 128 threads per (query head, sequence) with more than
// one split.  The split weights are formed in parallel (block max and sum
// over the splits' log-sum-exps), then the threads take 16-byte columns of
// head_dim and, where a row has fewer columns than threads, interleaved
// subsets of the splits, with eight loads in flight per thread; the subsets
// are summed through shared memory.  The work is a few hundred kilobytes
// per sequence, so the kernel is latency-bound: what matters is how many
// dependent memory round trips a CTA makes.  The first batch of partial
// loads is issued before the weights are formed, so rows of up to 8 x
// (threads / columns) splits (16 at head_dim 256) take one.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int CT = 128;         // threads per CTA
constexpr int MAX_SPLITS = 1024;
constexpr int INFLIGHT = 8;     // partial loads in flight per thread

// Splits of a sequence of length len: the block-aligned pieces of its key
// range [lo, pos] (the same rule as the decode kernels').
__device__ __forceinline__ int splits_of(int len, int window, int split_blocks)
{
    if (len <= 0 || split_blocks <= 0)
        return 1;
    const int pos = len - 1;
    const int lo = window > 0 ? max(0, pos - window) : 0;
    const int nblk = pos / kBlock - lo / kBlock + 1;
    return (nblk + split_blocks - 1) / split_blocks;
}

template <bool MAX>
__device__ __forceinline__ float block_reduce(float v, float *red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(FULL_MASK, v, off);
        v = MAX ? fmaxf(v, o) : v + o;
    }
    __syncthreads();  // red may still be read from a previous reduction
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < CT / 32; ++w)
        r = MAX ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

__device__ __forceinline__ void fma4(float4 &a, float w, const float4 &v)
{
    a.x = fmaf(w, v.x, a.x);
    a.y = fmaf(w, v.y, a.y);
    a.z = fmaf(w, v.z, a.z);
    a.w = fmaf(w, v.w, a.w);
}

}  // namespace

__global__ void __launch_bounds__(CT) combine_kernel(const CombineParams p)
{
    __shared__ float w_s[MAX_SPLITS];
    __shared__ float red[CT / 32];
    __shared__ float4 acc_s[CT];
    const int hq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int ns = min(splits_of(p.seq_lens[b], p.window, p.split_blocks), p.num_splits);
    if (ns <= 1)
        return;  // the decode kernel wrote this row's output itself
    const int D = p.head_dim;
    const size_t stride = static_cast<size_t>(p.num_q_heads);  // split-major rows
    const float *lse = p.part_lse + static_cast<size_t>(b) * p.num_splits * stride + hq;
    const float *po = p.part_o + (static_cast<size_t>(b) * p.num_splits * stride + hq) * D;
    const size_t sstride = stride * D;  // floats between splits of one row

    // column layout: 16-byte columns when the row and the pointers allow
    const uintptr_t oa = reinterpret_cast<uintptr_t>(p.out);
    const bool vec = (D & 3) == 0 && (reinterpret_cast<uintptr_t>(p.part_o) & 15) == 0 &&
                     (oa & (p.out_f32 ? 15 : 7)) == 0;
    const int nq = vec ? D / 4 : D;              // columns: float4 or scalar
    const int groups = nq >= CT ? 1 : CT / nq;   // interleaved split subsets
    const int g = tid / (nq >= CT ? CT : nq);
    const size_t row = static_cast<size_t>(b) * p.num_q_heads + hq;
    // INFLIGHT partial values of column c from splits s0, s0 + groups, ...
    auto load_batch = [&](int c, int s0, float4 (&v)[INFLIGHT]) {
#pragma unroll
        for (int k = 0; k < INFLIGHT; ++k) {
            const int s = s0 + k * groups;
            if (s < ns) {
                if (vec)
                    v[k] = *reinterpret_cast<const float4 *>(po + s * sstride + c * 4);
                else
                    v[k] = make_float4(po[s * sstride + c], 0.f, 0.f, 0.f);
            } else {
                v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
    // the first batch is in flight while the weights are formed: one memory
    // round trip fewer for rows of up to INFLIGHT x groups splits
    const bool mine = g < groups;
    float4 first[INFLIGHT];
    if (mine && (nq >= CT ? tid : tid % nq) < nq)
        load_batch(nq >= CT ? tid : tid % nq, g, first);

    // ---- weights: L = max lse, w_s = exp(lse_s - L), Z = sum w_s
    float m = -INFINITY;
    for (int s = tid; s < ns; s += CT) {
        const float l = lse[s * stride];
        w_s[s] = l;
        m = fmaxf(m, l);
    }
    const float M = block_reduce<true>(m, red);
    float z = 0.f;
    for (int s = tid; s < ns; s += CT) {
        const float l = w_s[s];
        const float w = (M == -INFINITY || l == -INFINITY) ? 0.f : expf(l - M);
        w_s[s] = w;
        z += w;
    }
    const float Z = block_reduce<false>(z, red);  // its barriers publish w_s

    // ---- weighted sum of the normalised partials
    for (int c0 = 0; c0 < nq; c0 += CT) {
        const int c = c0 + (nq >= CT ? tid : tid % nq);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (mine && c < nq) {
            for (int s0 = g; s0 < ns; s0 += INFLIGHT * groups) {
                float4 v[INFLIGHT];
                if (c0 == 0 && s0 == g) {
#pragma unroll
                    for (int k = 0; k < INFLIGHT; ++k)
                        v[k] = first[k];
                } else {
                    load_batch(c, s0, v);
                }
#pragma unroll
                for (int k = 0; k < INFLIGHT; ++k) {
                    const int s = s0 + k * groups;
                    const float w = s < ns ? w_s[s] : 0.f;
                    if (w != 0.f)  // a zero weight never multiplies a stale value
                        fma4(acc, w, v[k]);
                }
            }
        }
        if (groups > 1) {
            acc_s[tid] = acc;
            __syncthreads();
            if (g == 0) {
                for (int k = 1; k < groups; ++k) {
                    const float4 o = acc_s[k * nq + c];
                    acc.x += o.x;
                    acc.y += o.y;
                    acc.z += o.z;
                    acc.w += o.w;
                }
            }
        }
        if (g == 0 && c < nq) {
            float y[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                y[k] = Z > 0.f ? y[k] / Z : 0.f;
            if (vec) {
                const size_t o = row * D + c * 4;
                if (p.out_f32) {
                    *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + o) =
                        make_float4(y[0], y[1], y[2], y[3]);
                } else {
                    __nv_bfloat162 lo2 = __floats2bfloat162_rn(y[0], y[1]);
                    __nv_bfloat162 hi2 = __floats2bfloat162_rn(y[2], y[3]);
                    uint2 u;
                    u.x = *reinterpret_cast<uint32_t *>(&lo2);
                    u.y = *reinterpret_cast<uint32_t *>(&hi2);
                    *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + o) = u;
                }
            } else {
                const size_t o = row * D + c;
                if (p.out_f32)
                    reinterpret_cast<float *>(p.out)[o] = y[0];
                else
                    reinterpret_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(y[0]);
            }
        }
    }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s)
{
    dim3 grid(p.num_q_heads, p.batch);
    combine_kernel<<<grid, CT, 0, s>>>(p);
    note_launch();
    return cudaGetLastError();
}

}  // namespace pkv
