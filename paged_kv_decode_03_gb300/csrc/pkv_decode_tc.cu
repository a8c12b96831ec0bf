// pkv_decode_tc.cu -- decode attention over a bf16 paged KV pool on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// Same problem and sources as pkv_decode.cu: y = softmax(scale * q K^T) V
// over the keys [lo, pos] of each sequence ("CS336 · 第 10 课", KV-cache
// section; "实验五：Gemma4 端到端推理优化", sliding-window, GQA and Flash
// Attention sections: online softmax with running max/sum in fp32, blocks
// outside the window never read).
//
// Why tensor cores here: at head_dim 256 the bf16 inner products cost the
// CUDA cores more issue slots than HBM needs time to deliver the bytes (a
// variant of the CUDA-core kernel that skips every memory wait runs longer
// than the memory-bound time), so both contractions move to tcgen05 and the
// CUDA cores only do the softmax.
//
// One CTA per (split, kv head, sequence), 12 warps:
//   warps 4-9 (producers): TMA loads of 128-key tiles into a ring of six
//     32 KB units.  With K and V separate the ring is split into a K ring
//     (read only by the score warp) and a V ring (read only by the P.V
//     warp); with K == V one ring is read by both in the same order.  Each
//     consumer thus waits on every phase of the slots it reads, which is
//     what makes parity waits sound.  Producer warp w owns slot w and
//     issues its uses in order; several issuing warps are needed because
//     the rate of 2 KB TMA boxes scales with the number of issuing warps.
//   warp 10 (one thread): S^T[128 keys x 16] = K Q^T (M=128, N=16 query
//     heads padded, K=16 per instruction) into TMEM;
//   warp 11 (one thread): O^T[128 dims x 16] = V^T P^T per 128-dim half.
//     A thread issues small tcgen05.mma one after another at a fixed cost
//     each (about 40 ns here); two issuing threads run side by side, so
//     each contraction has its own.  tcgen05.commit signals the mbarriers
//     that free ring units and hand results on.
//   warps 0-3 (softmax): thread t owns key t of the tile (TMEM lane t):
//     loads its 16 scores, masks keys outside [lo, pos], forms the tile max
//     per head (warp shuffles + one exchange through shared memory), keeps
//     running max / sums in fp32, writes P^T in bf16 (K-major, swizzled)
//     for the P.V MMA -- for fp32 output also the bf16 residual p - bf16(p),
//     multiplied in a second pass, which keeps the error near 2^-17 -- and
//     accumulates the per-tile O^T (thread t owns
//     output dims t and 128+t) with the rescale alpha = 2^(m_old - m_new).
//     The P.V warp zeroes the V rows of masked keys inside loaded blocks
//     (stale slots past pos, keys before the window start) before its MMAs
//     read them, so no stale value (not even a NaN) reaches the output.
#include <cuda_bf16.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int PRODUCER_WARPS = 6;  // one per ring unit; TMA issue rate scales with issuing warps
constexpr int PRODUCER_WARP = 4;   // first producer warp
constexpr int MMA_WARP = PRODUCER_WARP + PRODUCER_WARPS;  // issues the score MMAs, owns TMEM
constexpr int PV_WARP = MMA_WARP + 1;                     // issues the P.V MMAs
constexpr int TC_WARPS = PV_WARP + 1;
constexpr int TC_THREADS = TC_WARPS * 32;
constexpr int NPAD = 16;          // N of every MMA: query heads padded to 16
constexpr int UNIT = 32768;       // 128 keys x 128 dims bf16
constexpr int CHUNK = 16384;      // 128 keys x 64 dims bf16 (one swizzled column)
constexpr int CTRL = 1024;        // barriers, TMEM address, flags, exchange
constexpr int QBYTES = 8192;      // Q^T: up to 4 columns x 16 heads x 128 B
constexpr int PBYTES = 16384;     // P^T: 2 buffers x (hi, lo) x 2 columns x 16 heads x 128 B
constexpr int RING_OFF = CTRL + QBYTES + PBYTES;
constexpr uint32_t TMEM_COLS = 128;

__device__ __forceinline__ uint32_t s_col(int sb) { return sb * 16; }
__device__ __forceinline__ uint32_t o_col(int sb, int half) { return 32 + sb * 32 + half * 16; }

// Byte offset of element (row, col) of a [rows][64] bf16 column stored with
// the 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ int swz(int row, int col)
{
    return row * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2;
}

struct Flags {
    volatile int *abort;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, const Flags &f,
                                              unsigned int *err)
{
    if (*f.abort)
        return false;
    if (!mbar_wait(bar, parity, err)) {
        *f.abort = 1;
        return false;
    }
    return true;
}

// TMEM columns of this thread's lane: N = 2, 4, 8 or 16.
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&v)[N])
{
    if constexpr (N == 16)
        tmem_ld16(taddr, v);
    else
        tmem_ld<N>(taddr, v);
}

// OR of a predicate over the 128 softmax threads (named barrier 1).
__device__ __forceinline__ bool softmax_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u)
        : "memory");
    return r != 0;
}

}  // namespace

template <int D, int GP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv)
{
    constexpr int HALVES = D / 128;
    static_assert(D == 128 || D == 256, "head_dim");
    static_assert(GP == 2 || GP == 4 || GP == 8 || GP == 16, "padded group");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *unit_full = reinterpret_cast<uint64_t *>(sm);  // [8]
    uint64_t *unit_empty = unit_full + 8;                    // [8]
    uint64_t *s_full = unit_full + 16;                       // [2]
    uint64_t *s_empty = s_full + 2;                          // [2]
    uint64_t *p_full = s_full + 4;                           // [2]
    uint64_t *o_full = s_full + 6;                           // [2]
    uint64_t *o_empty = s_full + 8;                          // [2]
    uint64_t *q_full = s_full + 10;                          // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 256);
    Flags flags{reinterpret_cast<volatile int *>(sm + 260)};
    float *red = reinterpret_cast<float *>(sm + 512);        // [4][16]
    uint8_t *qs = sm + CTRL;
    uint8_t *ps = sm + CTRL + QBYTES;
    uint8_t *units = sm + RING_OFF;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int G = p.group;
    const bool alias = p.alias != 0;
    const int NU = p.num_stages;
    const bool precise = p.out_f32 != 0;  // P as bf16 hi + lo: two P.V passes

    int len = p.seq_lens[b];
    const bool reporter = threadIdx.x == 0 && split == 0 && g == 0;
    if (len > p.max_blocks * kBlock) {
        if (reporter)
            record_error(p.err, PKV_DEV_LEN_TABLE);
        len = p.max_blocks * kBlock;
    }
    if (len > p.max_seq_len && reporter)
        record_error(p.err, PKV_DEV_LEN_BOUND);
    // key range and block-aligned split (as in the CUDA-core kernel)
    const int pos = len - 1;
    const int lo = p.window > 0 ? max(0, pos - p.window) : 0;
    const int blk_lo = len > 0 ? lo / kBlock : 0;
    const int nblk = len > 0 ? pos / kBlock - blk_lo + 1 : 0;
    const int nsplit = (p.split_blocks > 0 && nblk > 0) ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    if (split >= nsplit)
        return;
    const int ub0 = blk_lo + split * p.split_blocks;
    const int ub1 = p.split_blocks > 0 ? min(ub0 + p.split_blocks, blk_lo + nblk) : blk_lo + nblk;
    const int n = max(0, ub1 - ub0);
    const int T = (n + 7) / 8;  // 128-key tiles
    const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks + ub0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; ++i) {
            mbar_init(&unit_full[i], 1);
            mbar_init(&unit_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], 4);
        }
        mbar_init(q_full, 4);
        *flags.abort = 0;
        fence_barrier_init();
    }
    if (warp == MMA_WARP)
        tmem_alloc(tmem_slot, TMEM_COLS);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp < 4) {
        // Q^T (B operand of the score MMA): K-major, [D/64 columns][16 heads][64 dims].
        // Staged while the first tiles are already in flight; the MMA thread
        // waits on q_full.
        for (int idx = threadIdx.x; idx < NPAD * (D / 8); idx += 128) {
            const int h = idx / (D / 8), c8 = idx % (D / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (h < G)
                v = *reinterpret_cast<const uint4 *>(
                    p.q + (static_cast<size_t>(b) * p.num_q_heads + g * G + h) * D + c8 * 8);
            const int d0 = c8 * 8;
            *reinterpret_cast<uint4 *>(qs + (d0 / 64) * 2048 + swz(h, d0 % 64)) = v;
        }
        // P^T buffers start at zero: padded heads stay zero for the whole kernel
        for (int idx = threadIdx.x; idx < PBYTES / 16; idx += 128)
            reinterpret_cast<uint4 *>(ps)[idx] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(q_full);
    }

    constexpr int GL = GP < 16 ? GP : 16;  // TMEM columns read per result
    // Unit j = tile * HALVES + half of the K stream lives in slot j % NKU,
    // use j / NKU; of the V stream in slot VBASE + j % NVU, use j / NVU.
    const int NKU = alias ? NU : NU / 2;
    const int NVU = alias ? NU : NU - NKU;
    const int VBASE = alias ? 0 : NKU;

    if (warp >= PRODUCER_WARP && warp < MMA_WARP) {
        // ------------------------------------------------------ producers
        const int slot = warp - PRODUCER_WARP;  // the ring slot this warp owns
        const bool vwarp = !alias && slot >= NKU;
        const int ring = vwarp ? NVU : NKU, rbase = vwarp ? VBASE : 0;
        if (T > 0 && slot < NU) {
            const CUtensorMap *map = vwarp ? &tmv : &tmk;
            if (lane == 0)
                prefetch_tensormap(map);
            const uint64_t pol = policy_evict_first();
            TableCursor tc;
            tc.init(bt_row, n, lane);
            int last_use = -1;
            bool stop = false;
            for (int i = 0; i < T && !stop; ++i) {
                int row[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int blk = i * 8 + t;
                    const int phys = blk < n ? tc.get(blk, lane) : -1;
                    const bool valid =
                        static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
                    if (blk < n && !valid && lane == 0 && slot == 0)
                        record_error(p.err, PKV_DEV_BAD_BLOCK);
                    // an out-of-range row: the TMA fills the box with zeros
                    row[t] = valid ? phys * kBlock : p.num_blocks * kBlock;
                }
                for (int h = 0; h < HALVES; ++h) {
                    const int j = i * HALVES + h;
                    if (rbase + j % ring != slot)
                        continue;
                    const int use = j / ring;
                    const bool room =
                        use == 0 || wait_or_abort(&unit_empty[slot], (use - 1) & 1, flags, p.err);
                    if (!__all_sync(FULL_MASK, room)) {
                        stop = true;
                        break;
                    }
                    // lane 0 posts the unit's byte count, then 16 lanes issue
                    // one 2 KB box each (block t = lane / 2, column c = lane % 2)
                    if (lane == 0)
                        mbar_arrive_expect_tx(&unit_full[slot], UNIT);
                    __syncwarp();
                    if (lane < 16) {
                        const int t = lane >> 1, c = lane & 1;
                        int rt = row[0];
#pragma unroll
                        for (int k = 1; k < 8; ++k)
                            rt = (t == k) ? row[k] : rt;
                        tma_load_3d(units + slot * UNIT + c * CHUNK + t * 2048, map,
                                    h * 128 + c * 64, g, rt, &unit_full[slot], pol);
                    }
                    last_use = use;
                }
                __syncwarp();
            }
            // Drain: do not retire with this warp's copies in flight.
            if (lane == 0 && last_use >= 0)
                mbar_wait(&unit_full[slot], last_use & 1, p.err, 100000000ull);
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------ score MMAs
        // tile i needs its K units and a free S buffer
        if (lane == 0 && T > 0) {
            constexpr uint32_t IDESC_QK = umma_idesc_bf16(128, NPAD, false, false);
            const uint32_t q_base = smem_u32(qs), u_base = smem_u32(units);
            if (wait_or_abort(q_full, 0, flags, p.err)) {
                for (int i = 0; i < T; ++i) {
                    const int sb = i & 1;
                    if (i >= 2 && !wait_or_abort(&s_empty[sb], ((i / 2) - 1) & 1, flags, p.err))
                        break;
                    bool ok = true;
                    for (int h = 0; h < HALVES; ++h) {
                        const int j = i * HALVES + h, slot = j % NKU;
                        ok = wait_or_abort(&unit_full[slot], (j / NKU) & 1, flags, p.err);
                        if (!ok)
                            break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = umma_smem_desc(
                                u_base + slot * UNIT + (kk >> 2) * CHUNK + (kk & 3) * 32, 16, 1024);
                            const int kq = h * 8 + kk;
                            const uint64_t bd =
                                umma_smem_desc(q_base + (kq >> 2) * 2048 + (kq & 3) * 32, 16, 1024);
                            umma_bf16(tmem + s_col(sb), a, bd, IDESC_QK, (h | kk) != 0);
                        }
                        if (!alias)
                            umma_commit(&unit_empty[slot]);  // K unit free once read
                    }
                    if (!ok)
                        break;
                    umma_commit(&s_full[sb]);
                }
            }
        }
        __syncwarp();
    } else if (warp == PV_WARP) {
        // ------------------------------------------------------ P.V MMAs
        // tile i needs P^T, a free O buffer and its V units; the whole warp
        // first zeroes V rows of masked keys inside loaded blocks (only the
        // block holding the window start and the block holding pos can have
        // them), lane 0 then issues the MMAs.
        if (T > 0) {
            constexpr uint32_t IDESC_PV = umma_idesc_bf16(128, NPAD, true, false);
            const uint32_t p_base = smem_u32(ps), u_base = smem_u32(units);
            const int lo_blk = lo / kBlock, pos_blk = pos / kBlock;
            for (int i = 0; i < T; ++i) {
                const int sb = i & 1;
                bool go = wait_or_abort(&p_full[sb], (i / 2) & 1, flags, p.err);
                go = go && (i < 2 || wait_or_abort(&o_empty[sb], ((i / 2) - 1) & 1, flags, p.err));
                if (!__all_sync(FULL_MASK, go))
                    break;
                const int tb0 = ub0 + i * 8;  // first block of the tile
                const int key0 = tb0 * kBlock;
                // rows [z0a, z0b) before lo and [z1a, z1b) after pos, in this tile
                int z0a = 0, z0b = 0, z1a = 0, z1b = 0;
                if (lo_blk >= tb0 && lo_blk < tb0 + 8 && lo_blk < ub1 && lo > lo_blk * kBlock) {
                    z0a = lo_blk * kBlock - key0;
                    z0b = lo - key0;
                }
                if (pos_blk >= tb0 && pos_blk < tb0 + 8 && pos_blk < ub1 &&
                    pos < pos_blk * kBlock + kBlock - 1) {
                    z1a = pos + 1 - key0;
                    z1b = (pos_blk + 1) * kBlock - key0;
                }
                bool ok = true;
                for (int h = 0; h < HALVES; ++h) {
                    const int j = i * HALVES + h, slot = VBASE + j % NVU;
                    ok = wait_or_abort(&unit_full[slot], (j / NVU) & 1, flags, p.err);
                    if (!__all_sync(FULL_MASK, ok)) {
                        ok = false;
                        break;
                    }
                    if (z0b > z0a || z1b > z1a) {
                        uint8_t *ub = units + slot * UNIT;
                        for (int idx = lane; idx < 128 * 16; idx += 32) {
                            const int r = idx >> 4, ch = idx & 15;
                            if ((r >= z0a && r < z0b) || (r >= z1a && r < z1b))
                                *reinterpret_cast<uint4 *>(ub + (ch >> 3) * CHUNK + r * 128 +
                                                           (ch & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) {
                        tc_fence_after();
                        for (int pass = 0; pass < (precise ? 2 : 1); ++pass) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                // V^T half h: MN-major, 64-dim columns CHUNK apart,
                                // 8-key groups 1 KB apart
                                const uint64_t a =
                                    umma_smem_desc(u_base + slot * UNIT + kk * 2048, CHUNK, 1024);
                                const uint64_t bd = umma_smem_desc(
                                    p_base + sb * 8192 + pass * 4096 + (kk >> 2) * 2048 + (kk & 3) * 32,
                                    16, 1024);
                                umma_bf16(tmem + o_col(sb, h), a, bd, IDESC_PV, (pass | kk) != 0);
                            }
                        }
                        umma_commit(&unit_empty[slot]);  // V (or K = V) unit free once read
                    }
                    __syncwarp();
                }
                if (!ok)
                    break;
                if (lane == 0)
                    umma_commit(&o_full[sb]);
                __syncwarp();
            }
        }
    } else {
        // ------------------------------------------------------ softmax
        const int t = threadIdx.x;  // key row of the tile == TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float qk = p.qk_scale_log2;
        // oacc holds the running O^T relative to the current running max:
        // after tile i-1's O^T is added it is rescaled by tile i's alpha.
        float m_run[GP], lpart[GP];
        float oacc[HALVES][GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            m_run[h] = -INFINITY;
            lpart[h] = 0.f;
#pragma unroll
            for (int hv = 0; hv < HALVES; ++hv)
                oacc[hv][h] = 0.f;
        }
        auto accumulate_o = [&](int k) {
            const int sb = k & 1;
            const bool live = wait_or_abort(&o_full[sb], (k / 2) & 1, flags, p.err);
            tc_fence_after();
#pragma unroll
            for (int hv = 0; hv < HALVES; ++hv) {
                float ot[GL];
                if (live)
                    ld_cols<GL>(lane_base + o_col(sb, hv), ot);
#pragma unroll
                for (int h = 0; h < GP; ++h)
                    oacc[hv][h] += live ? ot[h] : 0.f;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&o_empty[sb]);
        };
        int phys_next = (t >> 4) < n ? __ldg(bt_row + (t >> 4)) : -1;
        for (int i = 0; i < T; ++i) {
            const int sb = i & 1;
            const int blk = i * 8 + (t >> 4);
            const int phys = phys_next;
            {
                const int nb = (i + 1) * 8 + (t >> 4);
                phys_next = nb < n ? __ldg(bt_row + nb) : -1;
            }
            const bool loaded = blk < n && static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
            const int j = (ub0 + i * 8) * kBlock + t;
            const bool ok = loaded && j >= lo && j <= pos;
            // ---- scores
            const bool live = wait_or_abort(&s_full[sb], (i / 2) & 1, flags, p.err);
            tc_fence_after();
            float s[GL];
            if (live)
                ld_cols<GL>(lane_base + s_col(sb), s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s_empty[sb]);
            float sc[GP];
            bool big = false;
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                sc[h] = (live && ok && h < G) ? s[h] * qk : -INFINITY;
                big |= sc[h] > m_run[h] + 8.f;
            }
            // ---- running max: reduce only when some score exceeds it by more
            // than 2^8 (any reference max >= the true one gives the same
            // result; this one keeps every p <= 256)
            float alpha[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h)
                alpha[h] = 1.f;
            const bool rescale = softmax_any(big);
            if (rescale) {
                float mx[GP];
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    float v = sc[h];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, off));
                    mx[h] = v;
                }
                if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < GP; ++h)
                        red[warp * 16 + h] = mx[h];
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    const float tm =
                        fmaxf(fmaxf(red[h], red[16 + h]), fmaxf(red[32 + h], red[48 + h]));
                    const float mn = fmaxf(m_run[h], tm);
                    alpha[h] = mn == -INFINITY ? 1.f : fast_exp2(m_run[h] - mn);
                    m_run[h] = mn;
                }
                asm volatile("bar.sync 1, 128;" ::: "memory");  // red is reused
            }
            // ---- probabilities, running sums, P^T (bf16, K-major, swizzled)
            uint8_t *pb = ps + sb * 8192 + (t >> 6) * 2048;
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float pr = sc[h] == -INFINITY ? 0.f : fast_exp2(sc[h] - m_run[h]);
                lpart[h] = fmaf(lpart[h], alpha[h], pr);
                const __nv_bfloat16 hi = __float2bfloat16_rn(pr);
                *reinterpret_cast<__nv_bfloat16 *>(pb + swz(h, t & 63)) = hi;
                if (precise)
                    *reinterpret_cast<__nv_bfloat16 *>(pb + 4096 + swz(h, t & 63)) =
                        __float2bfloat16_rn(pr - __bfloat162float(hi));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[sb]);
            // ---- O^T of the previous tile, then rescale to this tile's max
            if (i >= 1)
                accumulate_o(i - 1);
            if (rescale) {
#pragma unroll
                for (int h = 0; h < GP; ++h)
#pragma unroll
                    for (int hv = 0; hv < HALVES; ++hv)
                        oacc[hv][h] *= alpha[h];
            }
        }
        if (T > 0)
            accumulate_o(T - 1);

        // ---- final sums over the 128 keys of each head, then the output
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            float v = lpart[h];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                v += __shfl_xor_sync(FULL_MASK, v, off);
            lpart[h] = v;
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GP; ++h)
                red[warp * 16 + h] = lpart[h];
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const bool single = nsplit == 1;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            if (h >= G)
                continue;
            const float L = (red[h] + red[16 + h]) + (red[32 + h] + red[48 + h]);
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const size_t orow = static_cast<size_t>(b) * p.num_q_heads + g * G + h;
#pragma unroll
            for (int hv = 0; hv < HALVES; ++hv) {
                const int d = hv * 128 + t;
                const float y = oacc[hv][h] * inv;
                if (single) {
                    if (p.out_f32)
                        reinterpret_cast<float *>(p.out)[orow * D + d] = y;
                    else
                        reinterpret_cast<__nv_bfloat16 *>(p.out)[orow * D + d] = __float2bfloat16_rn(y);
                } else {
                    p.part_o[(orow * p.num_splits + split) * D + d] = y;
                }
            }
            if (!single && t == 0)
                p.part_lse[orow * p.num_splits + split] =
                    L > 0.f ? (m_run[h] + log2f(L)) * LN2 : -INFINITY;
        }
    }

    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------ host side
size_t decode_tc_smem_bytes(int num_units) { return 1024 + RING_OFF + static_cast<size_t>(num_units) * UNIT; }

int decode_tc_group_pad(int group)
{
    return group <= 2 ? 2 : group <= 4 ? 4 : group <= 8 ? 8 : group <= 16 ? 16 : 0;
}

template <int D, int GP>
static cudaError_t launch_tc_one(const DecodeParams &p, const CUtensorMap &tmk,
                                 const CUtensorMap &tmv, cudaStream_t s)
{
    const size_t smem = decode_tc_smem_bytes(p.num_stages);
    auto kern = decode_tc_kernel<D, GP>;
    static int configured = 0;
    if (static_cast<int>(smem) > configured) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured = static_cast<int>(smem);
    }
    dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    kern<<<grid, TC_THREADS, smem, s>>>(p, tmk, tmv);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_tc_d(const DecodeParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, int gp, cudaStream_t s)
{
    switch (gp) {
    case 2: return launch_tc_one<D, 2>(p, tmk, tmv, s);
    case 4: return launch_tc_one<D, 4>(p, tmk, tmv, s);
    case 8: return launch_tc_one<D, 8>(p, tmk, tmv, s);
    case 16: return launch_tc_one<D, 16>(p, tmk, tmv, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_tc(const DecodeParams &p, const CUtensorMap &tmk,
                             const CUtensorMap &tmv, int head_dim, cudaStream_t s)
{
    const int gp = decode_tc_group_pad(p.group);
    if (head_dim == 128)
        return launch_tc_d<128>(p, tmk, tmv, gp, s);
    if (head_dim == 256)
        return launch_tc_d<256>(p, tmk, tmv, gp, s);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
