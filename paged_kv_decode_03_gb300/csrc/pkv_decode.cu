// pkv_decode.cu -- CUDA-core decode attention over a paged KV pool, and the
// log-sum-exp combine of split-KV partials.
//
// What is computed (sources by page title and section):
//   "CS336 · 第 10 课", KV-cache section: y = softmax(q K^T * scale) V over
//   the cached keys; "实验五：Gemma4 端到端推理优化" (Lab5-Gemma4): keys limited
//   to [pos-w, pos] on sliding layers (滑动窗口注意力), query heads sharing a
//   KV head (分组查询注意力), online softmax with a running max m, sum l and
//   unnormalised output o kept in fp32 and O = o / l at the end, blocks
//   outside the window skipped instead of masked, and a dedicated
//   single-query decode kernel (Flash Attention section); the A100 article
//   "LLM推理优化底层原理" §3.1 step 2 gives the same max/sum recurrence;
//   "推理优化与 AI Infra" section 5: int8 KV dequantised after the gather.
//
// Design (GB300):
//   * One CTA per (split, kv head, query-head chunk, sequence).  The CTA
//     reads each KV byte of its range once and serves every query head of
//     its GQA chunk from it.
//   * Warp specialisation: one producer thread issues TMA tile loads
//     (cp.async.bulk.tensor, 16 rows x head_dim of one kv head per paged
//     block) into an NS-stage shared-memory ring guarded by mbarriers; four
//     consumer warps each own every fourth stage and run an independent
//     online softmax over their blocks; the four states merge at the end.
//   * A consumer warp spreads head_dim over its 32 lanes (16-byte shared
//     loads for bf16 D=256), forms the partial dot products of R keys x GT
//     heads (R*GT = 32 or 16) and finishes them with one butterfly
//     reduce-scatter (31 shuffles per 32 dot products), after which lane
//     (h, r) owns score (key r, head h).
//   * Keys outside [lo, pos] in the first/last block are masked with a
//     select (never arithmetic), so stale or NaN slots contribute nothing.
#include <cuda_bf16.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int NC = 4;                    // consumer warps per CTA
constexpr int THREADS = (NC + 1) * 32;   // + one producer warp
constexpr int BAR_BYTES = 256;           // mbarrier area at the start of smem

struct KeyRange {
    int lo, pos, blk_lo, nblk, nsplit;
};

// Keys a decode at position len-1 may attend to, and the block-aligned
// split of that range.  Shared by the decode and the combine kernels.
__device__ __forceinline__ KeyRange key_range(int len, int window, int split_blocks)
{
    KeyRange r;
    r.pos = len - 1;
    r.lo = window > 0 ? max(0, r.pos - window) : 0;
    if (len <= 0) {
        r.blk_lo = 0;
        r.nblk = 0;
        r.nsplit = 1;
        return r;
    }
    r.blk_lo = r.lo / kBlock;
    r.nblk = r.pos / kBlock - r.blk_lo + 1;
    r.nsplit = split_blocks > 0 ? (r.nblk + split_blocks - 1) / split_blocks : 1;
    return r;
}

template <int D, int GT, bool INT8>
struct Cfg {
    static constexpr int P = kBlock;
    static constexpr int ES = INT8 ? 1 : 2;                // element bytes
    static constexpr int CHE = (D * ES > 256) ? 256 / ES : D;  // elements per TMA box row
    static constexpr int NCH = D / CHE;                     // boxes per tile
    static constexpr int ROWB = CHE * ES;                   // bytes of one box row
    static constexpr int TILE = P * D * ES;                 // one kv head x one block
    static constexpr int DPL = D / 32;                      // elements per lane
    static constexpr int NV = (GT == 1) ? 16 : 32;          // dot products per reduction
    static constexpr int R = NV / GT;                       // keys per reduction group
    static constexpr int GROUPS = P / R;
    static_assert(D % 32 == 0 && DPL >= 2 && DPL <= 8, "head_dim");
    static_assert(P % R == 0, "group");
};

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Bytes of one ring stage: K tile, V tile (unless aliased), per-token scales.
__host__ __device__ inline int stage_bytes(int tile, int alias, int per_token)
{
    int b = tile + (alias ? 0 : tile);
    if (per_token)
        b += 128;  // 16 K scales + 16 V scales
    return round_up(b, 128);
}

// Butterfly reduce-scatter of NV per-lane partial sums: afterwards lane l
// holds the full warp sum of value index l (NV == 32) or l >> 1 (NV == 16).
template <int NV>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane)
{
#pragma unroll
    for (int half = NV / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            float send = upper ? v[i] : v[i + half];
            float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL_MASK, send, off);
        }
    }
    float r = v[0];
    if constexpr (NV == 16)
        r += __shfl_xor_sync(FULL_MASK, r, 1);
    return r;
}

template <int NV, int R>
__device__ __forceinline__ int lane_of(int h, int r)
{
    return NV == 32 ? h * R + r : 2 * r;
}

template <int D, int GT, bool INT8>
__global__ void __launch_bounds__(THREADS) decode_kernel(const DecodeParams p,
                                                         const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv)
{
    using C = Cfg<D, GT, INT8>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + 16;
    uint8_t *ring = smem + BAR_BYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y / p.head_chunks;
    const int chunk = blockIdx.y - g * p.head_chunks;
    const int b = blockIdx.z;
    const int NS = p.num_stages;
    const bool per_token = INT8 && p.scale_mode == PKV_SCALE_PER_TOKEN;
    const bool per_head = INT8 && p.scale_mode == PKV_SCALE_PER_HEAD;
    const int SB = stage_bytes(C::TILE, p.alias, per_token);

    int len = p.seq_lens[b];
    const bool reporter = threadIdx.x == 0 && split == 0 && blockIdx.y == 0;
    if (len > p.max_blocks * C::P) {
        if (reporter)
            record_error(p.err, PKV_DEV_LEN_TABLE);
        len = p.max_blocks * C::P;
    }
    if (len > p.max_seq_len && reporter)
        record_error(p.err, PKV_DEV_LEN_BOUND);
    const KeyRange kr = key_range(len, p.window, p.split_blocks);
    if (split >= kr.nsplit)
        return;
    const int ub0 = kr.blk_lo + split * p.split_blocks;
    const int ub1 = p.split_blocks > 0 ? min(ub0 + p.split_blocks, kr.blk_lo + kr.nblk)
                                       : kr.blk_lo + kr.nblk;
    const int n = max(0, ub1 - ub0);
    const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NC) {
        // ------------------------------------------------------ producer
        if (lane == 0 && n > 0) {
            prefetch_tensormap(&tmk);
            const uint64_t pol = policy_evict_first();
            const uint32_t tx = (p.alias ? 1 : 2) * C::TILE + (per_token ? (p.alias ? 64 : 128) : 0);
            int issued = 0;
            for (int i = 0; i < n; ++i) {
                const int st = i % NS;
                if (i >= NS && !mbar_wait(&empty[st], ((i / NS) - 1) & 1, p.err))
                    break;
                const int phys = bt_row[ub0 + i];
                const bool valid = static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
                if (!valid)
                    record_error(p.err, PKV_DEV_BAD_BLOCK);
                mbar_arrive_expect_tx(&full[st], valid ? tx : 0u);
                ++issued;
                if (!valid)
                    continue;
                uint8_t *kt = ring + st * SB;
                uint8_t *vt = kt + C::TILE;
                const int row0 = phys * C::P;
#pragma unroll
                for (int ch = 0; ch < C::NCH; ++ch)
                    tma_load_3d(kt + ch * C::P * C::ROWB, &tmk, ch * C::CHE, g, row0, &full[st], pol);
                if (!p.alias) {
#pragma unroll
                    for (int ch = 0; ch < C::NCH; ++ch)
                        tma_load_3d(vt + ch * C::P * C::ROWB, &tmv, ch * C::CHE, g, row0, &full[st],
                                    pol);
                }
                if (per_token) {
                    uint8_t *sc = kt + (p.alias ? 1 : 2) * C::TILE;
                    bulk_load(sc, p.k_scale + row0, 64, &full[st]);
                    if (!p.alias)
                        bulk_load(sc + 64, p.v_scale + row0, 64, &full[st]);
                }
            }
            // Drain: do not let the CTA retire with copies in flight.
            for (int i = max(0, issued - NS); i < issued; ++i)
                mbar_wait(&full[i % NS], (i / NS) & 1, p.err, 100000000ull);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    constexpr int DPL = C::DPL, NV = C::NV, R = C::R;
    const int G = p.group;
    const int lane_elem = lane * DPL;
    const int lane_off = (lane_elem / C::CHE) * C::P * C::ROWB + (lane_elem % C::CHE) * C::ES;

    float qf[GT][DPL];
    {
        float qmul = p.qk_scale_log2;
        if (per_head)
            qmul *= p.k_scale[g];
#pragma unroll
        for (int h = 0; h < GT; ++h) {
            const int hl = chunk * GT + h;
            if (hl < G) {
                const uint16_t *qr =
                    p.q + (static_cast<size_t>(b) * p.num_q_heads + g * G + hl) * D + lane_elem;
#pragma unroll
                for (int i = 0; i < DPL; ++i)
                    qf[h][i] = __uint_as_float(static_cast<uint32_t>(qr[i]) << 16) * qmul;
            } else {
#pragma unroll
                for (int i = 0; i < DPL; ++i)
                    qf[h][i] = 0.f;
            }
        }
    }

    float o[GT][DPL];
    float m[GT];
#pragma unroll
    for (int h = 0; h < GT; ++h) {
        m[h] = -INFINITY;
#pragma unroll
        for (int i = 0; i < DPL; ++i)
            o[h][i] = 0.f;
    }
    float l_lane = 0.f;
    const int my_idx = (NV == 32) ? lane : (lane >> 1);
    const int my_h = my_idx / R, my_r = my_idx % R;

    for (int i = warp; i < n; i += NC) {
        const int st = i % NS;
        if (!mbar_wait(&full[st], (i / NS) & 1, p.err))
            break;
        const int phys = bt_row[ub0 + i];
        if (static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks)) {
            const uint8_t *kt = ring + st * SB;
            const uint8_t *vt = p.alias ? kt : kt + C::TILE;
            const float *ksc = reinterpret_cast<const float *>(kt + (p.alias ? 1 : 2) * C::TILE);
            const float *vsc = p.alias ? ksc : ksc + 16;
            const int j0 = (ub0 + i) * C::P;
            const bool all_in = j0 >= kr.lo && j0 + C::P - 1 <= kr.pos;
#pragma unroll
            for (int grp = 0; grp < C::GROUPS; ++grp) {
                const int r0 = grp * R;
                float acc[NV];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    float kf[DPL];
                    load_row_chunk<DPL, INT8>(kt + lane_off + (r0 + r) * C::ROWB, kf);
#pragma unroll
                    for (int h = 0; h < GT; ++h) {
                        float a = 0.f;
#pragma unroll
                        for (int e = 0; e < DPL; ++e)
                            a = fmaf(qf[h][e], kf[e], a);
                        acc[h * R + r] = a;
                    }
                }
                float sc = reduce_scatter<NV>(acc, lane);
                const int jm = j0 + r0 + my_r;
                const bool ok = all_in || (jm >= kr.lo && jm <= kr.pos);
                if (per_token)
                    sc *= ksc[r0 + my_r];
                sc = ok ? sc : -INFINITY;
                // max over the R keys of this lane's head
                float mx = sc;
                if constexpr (NV == 32) {
#pragma unroll
                    for (int off = 1; off < R; off <<= 1)
                        mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, off));
                } else {
#pragma unroll
                    for (int off = 2; off < 32; off <<= 1)
                        mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, off));
                }
                float alpha[GT];
                float m_mine = 0.f, a_mine = 1.f;
#pragma unroll
                for (int h = 0; h < GT; ++h) {
                    const float tm = __shfl_sync(FULL_MASK, mx, lane_of<NV, R>(h, 0));
                    const float mn = fmaxf(m[h], tm);
                    alpha[h] = (mn == -INFINITY) ? 1.f : fast_exp2(m[h] - mn);
                    m[h] = mn;
                    if (h == my_h) {
                        m_mine = mn;
                        a_mine = alpha[h];
                    }
                }
                const float pr = ok ? fast_exp2(sc - m_mine) : 0.f;
                l_lane = l_lane * a_mine + ((NV == 16 && (lane & 1)) ? 0.f : pr);
#pragma unroll
                for (int h = 0; h < GT; ++h)
#pragma unroll
                    for (int e = 0; e < DPL; ++e)
                        o[h][e] *= alpha[h];
                float pv = pr;
                if (per_token)
                    pv = ok ? pr * vsc[r0 + my_r] : 0.f;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int j = j0 + r0 + r;
                    if (!all_in && (j < kr.lo || j > kr.pos))
                        continue;  // warp-uniform: masked key, data may be stale
                    float vf[DPL];
                    load_row_chunk<DPL, INT8>(vt + lane_off + (r0 + r) * C::ROWB, vf);
#pragma unroll
                    for (int h = 0; h < GT; ++h) {
                        const float w = __shfl_sync(FULL_MASK, pv, lane_of<NV, R>(h, r));
#pragma unroll
                        for (int e = 0; e < DPL; ++e)
                            o[h][e] = fmaf(w, vf[e], o[h][e]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }

    // per-head l: sum the lanes of each head
    {
        float ls = l_lane;
        if constexpr (NV == 32) {
#pragma unroll
            for (int off = 1; off < R; off <<= 1)
                ls += __shfl_xor_sync(FULL_MASK, ls, off);
        } else {
#pragma unroll
            for (int off = 1; off < 32; off <<= 1)
                ls += __shfl_xor_sync(FULL_MASK, ls, off);
        }
        l_lane = ls;
    }
    float lh[GT];
#pragma unroll
    for (int h = 0; h < GT; ++h)
        lh[h] = __shfl_sync(FULL_MASK, l_lane, lane_of<NV, R>(h, 0));

    // ------------------------------------------- merge the warps' states
    asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");  // ring no longer read
    float *mrg_m = reinterpret_cast<float *>(ring);             // [NC][GT]
    float *mrg_l = mrg_m + NC * GT;                             // [NC][GT]
    float *mrg_o = mrg_l + NC * GT;                             // [NC][GT][D]
    if (lane < GT) {
        float mm = m[0], ll = lh[0];
#pragma unroll
        for (int h = 1; h < GT; ++h)
            if (lane == h) {
                mm = m[h];
                ll = lh[h];
            }
        mrg_m[warp * GT + lane] = mm;
        mrg_l[warp * GT + lane] = ll;
    }
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e)
            mrg_o[(warp * GT + h) * D + lane_elem + e] = o[h][e];
    asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");

    const bool single = kr.nsplit == 1;
    const float vmul = per_head ? p.v_scale[g] : 1.f;
    for (int idx = threadIdx.x; idx < GT * D; idx += NC * 32) {
        const int h = idx / D, d = idx - h * D;
        const int hl = chunk * GT + h;
        if (hl >= G)
            continue;
        const int hq = g * G + hl;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NC; ++w)
            M = fmaxf(M, mrg_m[w * GT + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NC; ++w) {
                const float mw = mrg_m[w * GT + h];
                if (mw == -INFINITY)
                    continue;
                const float f = fast_exp2(mw - M);
                L = fmaf(mrg_l[w * GT + h], f, L);
                O = fmaf(mrg_o[(w * GT + h) * D + d], f, O);
            }
        }
        const float y = L > 0.f ? (O / L) * vmul : 0.f;
        const size_t row = static_cast<size_t>(b) * p.num_q_heads + hq;
        if (single) {
            if (p.out_f32)
                reinterpret_cast<float *>(p.out)[row * D + d] = y;
            else
                reinterpret_cast<__nv_bfloat16 *>(p.out)[row * D + d] = __float2bfloat16_rn(y);
        } else {
            p.part_o[(row * p.num_splits + split) * D + d] = y;
            if (d == 0)
                p.part_lse[row * p.num_splits + split] =
                    L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
        }
    }
}

// One CTA per (query head, sequence) with more than one split.
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p)
{
    __shared__ float w_s[1024];
    __shared__ float red[2];
    const int hq = blockIdx.x, b = blockIdx.y;
    const KeyRange kr = key_range(p.seq_lens[b], p.window, p.split_blocks);
    const int ns = min(kr.nsplit, p.num_splits);
    if (ns <= 1)
        return;
    const size_t row = static_cast<size_t>(b) * p.num_q_heads + hq;
    const float *lse = p.part_lse + row * p.num_splits;
    if (threadIdx.x == 0) {
        float M = -INFINITY;
        for (int s = 0; s < ns; ++s)
            M = fmaxf(M, lse[s]);
        float Z = 0.f;
        for (int s = 0; s < ns && s < 1024; ++s) {
            const float w = (M == -INFINITY || lse[s] == -INFINITY) ? 0.f : expf(lse[s] - M);
            w_s[s] = w;
            Z += w;
        }
        red[0] = Z;
    }
    __syncthreads();
    const float Z = red[0];
    const float *po = p.part_o + row * p.num_splits * p.head_dim;
    for (int d = threadIdx.x; d < p.head_dim; d += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < ns && s < 1024; ++s)
            acc = fmaf(w_s[s], po[static_cast<size_t>(s) * p.head_dim + d], acc);
        const float y = Z > 0.f ? acc / Z : 0.f;
        if (p.out_f32)
            reinterpret_cast<float *>(p.out)[row * p.head_dim + d] = y;
        else
            reinterpret_cast<__nv_bfloat16 *>(p.out)[row * p.head_dim + d] = __float2bfloat16_rn(y);
    }
}

// ------------------------------------------------------------ host side
int decode_group_tile(int group)
{
    return group >= 4 ? 4 : (group >= 2 ? (group == 2 ? 2 : 4) : 1);
}

size_t decode_smem_bytes(int head_dim, int int8, int alias, int per_token, int group_tile,
                         int num_stages)
{
    const int tile = kBlock * head_dim * (int8 ? 1 : 2);
    const size_t ring = static_cast<size_t>(num_stages) * stage_bytes(tile, alias, per_token);
    const size_t merge = (2 * NC * group_tile + static_cast<size_t>(NC) * group_tile * head_dim) *
                         sizeof(float);
    return BAR_BYTES + (ring > merge ? ring : merge);
}

template <int D, int GT, bool INT8>
static cudaError_t launch_one(const DecodeParams &p, const CUtensorMap &tmk,
                              const CUtensorMap &tmv, cudaStream_t s)
{
    const size_t smem =
        decode_smem_bytes(D, INT8, p.alias, INT8 && p.scale_mode == PKV_SCALE_PER_TOKEN, GT,
                          p.num_stages);
    auto kern = decode_kernel<D, GT, INT8>;
    static int configured = 0;  // largest dynamic smem set so far (per process)
    if (static_cast<int>(smem) > configured) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured = static_cast<int>(smem);
    }
    dim3 grid(p.num_splits, p.num_kv_heads * p.head_chunks, p.batch);
    kern<<<grid, THREADS, smem, s>>>(p, tmk, tmv);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_d(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                            int int8, int gt, cudaStream_t s)
{
    if (int8) {
        if (gt == 1) return launch_one<D, 1, true>(p, tmk, tmv, s);
        if (gt == 2) return launch_one<D, 2, true>(p, tmk, tmv, s);
        return launch_one<D, 4, true>(p, tmk, tmv, s);
    }
    if (gt == 1) return launch_one<D, 1, false>(p, tmk, tmv, s);
    if (gt == 2) return launch_one<D, 2, false>(p, tmk, tmv, s);
    return launch_one<D, 4, false>(p, tmk, tmv, s);
}

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                          int head_dim, int int8, int group_tile, cudaStream_t s)
{
    switch (head_dim) {
    case 64: return launch_d<64>(p, tmk, tmv, int8, group_tile, s);
    case 128: return launch_d<128>(p, tmk, tmv, int8, group_tile, s);
    case 256: return launch_d<256>(p, tmk, tmv, int8, group_tile, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s)
{
    dim3 grid(p.num_q_heads, p.batch);
    combine_kernel<<<grid, 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
