// pkv_prefill.cu -- attention of a chunk of new tokens per sequence over a
// bf16 paged KV pool (q_len > 1: chunked prefill, or the gamma + 1 tokens a
// speculative step verifies) on the 5th-generation tensor cores.
//
// Sources: "实验五：Gemma4 端到端推理优化", Flash Attention section (blocks of
// Q, K and V through on-chip memory, online softmax with running max m, sum
// l and unnormalised o, O = o / l; causal and sliding-window masks; GQA
// without repeating K/V; q_len > 1 as well as 1; the cache's history and the
// partial last tile), and "推理优化与 AI Infra" section 7 (the verify step
// feeds gamma + 1 tokens at once).  Sequence b's chunk is its last n_b
// tokens (appended to the cache before this call): token i sits at position
// len_b - n_b + i and attends keys [lo, pos] of its own position, so the
// chunk is causal among itself.
//
// Decomposition: one CTA per (query tile, kv head, sequence).  A query tile
// is 128 rows, row r = (token r / G, query head kvh * G + r % G) of the
// chunk: the rows of one kv head's group share every K/V byte the CTA
// reads.  The CTA walks the 64-key tiles of [lo(first token), last token]:
//   warps 0-3 first copy their rows of Q into TMEM (thread r = row r = TMEM
//     lane r; zeros for rows past the chunk): the score MMAs take their A
//     operand from there, which leaves shared memory to the K/V slots;
//   warp 5: TMA loads of each key tile's K and V blocks (boxes of 16 rows x
//     64 dims, 128-byte swizzle) into separate K and V slots, a K slot being
//     free once the scores have read it and a V slot once the P.V has;
//   warp 4 (one thread): S = Q K^T (M = 128 rows, N = 64 keys, K = 16) into
//     one of two TMEM score buffers, then O += P V (M = 128, N = head_dim,
//     K = 16 keys) into TMEM, accumulating over the key tiles; the previous
//     tile's P.V goes first when this tile's K has not landed yet; the whole
//     warp first zeroes V rows of keys no row may see inside loaded blocks,
//     so that no stale value (not even a NaN) meets a zero probability;
//   warps 0-3 (thread r = row r = TMEM lane r): load the row's 64 scores,
//     mask them by the row's own key range, keep the row's running max and
//     sum in fp32 (the max changes only when a score exceeds it by more
//     than 2^8; O's row is then scaled in TMEM by the thread that owns it,
//     after the previous tile's P.V), write the row's probabilities as bf16
//     (K-major, swizzled; two P buffers for bf16 outputs) for the P.V MMA,
//     and finally read O's row, divide by the sum and store it.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int PF_ROWS = 128;       // query rows per CTA (M of every MMA)
constexpr int PF_KEYS = 64;        // keys per tile (N of S, K of P.V)
constexpr int PF_THREADS = 192;    // warps 0-3 softmax, 4 MMA, 5 TMA
constexpr int PF_MMA_WARP = 4;
constexpr int PF_TMA_WARP = 5;
constexpr int PF_CTRL = 1024;
constexpr int PF_KCHUNK = PF_KEYS * 128;   // 64 keys x 64 dims bf16
constexpr int PF_PROW = PF_ROWS * 128;     // 128 rows x 64 keys bf16
// P: two bf16 buffers (bf16 output), or one P and its bf16 residual (fp32 output)
constexpr int PF_PBYTES = 2 * PF_PROW;
constexpr int PF_MAX_BUF = 4;

__device__ __forceinline__ int pf_swz(int row, int chunk16)
{
    return row * 128 + (((chunk16 ^ row) & 7) << 4);
}

// The chunk of sequence b and the key range of query tile `tile` of it.
struct ChunkTile {
    int n, len, q0;       // tokens in the chunk, sequence length, first query row
    int t0, nt;           // first token of this tile and tokens in it
    int lo, last;         // keys [lo, last] some row of the tile may see
    int blk0, nblk, T;    // first paged block, blocks, 64-key tiles
};

__device__ __forceinline__ bool chunk_tile(const PrefillParams &p, int b, int tile, int tpt,
                                           ChunkTile &c)
{
    c.q0 = p.q_start[b];
    c.n = p.q_start[b + 1] - c.q0;
    c.len = p.seq_lens[b];
    if (p.ring_blocks == 0 && c.len > p.max_blocks * kBlock)
        c.len = p.max_blocks * kBlock;  // reported by the reporter thread
    c.t0 = tile * tpt;
    if (c.n <= 0 || c.t0 >= c.n || c.n > c.len)
        return false;
    c.nt = min(tpt, c.n - c.t0);
    const int first = c.len - c.n + c.t0;
    c.last = first + c.nt - 1;
    c.lo = p.window > 0 ? max(0, first - p.window) : 0;
    c.blk0 = c.lo / kBlock;
    c.nblk = c.last / kBlock - c.blk0 + 1;
    c.T = (c.nblk + 3) / 4;
    return true;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tmq)
{
    static_assert(D == 64 || D == 128 || D == 256, "head_dim");
    constexpr int NCH = D / 64;                 // 64-dim chunks
    constexpr int KV_TILE = NCH * PF_KCHUNK;    // one K (or V) tile
    // TMEM: S buffers at 0 and 64, O (D fp32 columns), then Q (D / 2 columns
    // of bf16 pairs: the A operand of the score MMAs, read from TMEM so that
    // shared memory holds a third K/V tile instead of Q)
    constexpr uint32_t TMEM_COLS = 2 * PF_KEYS + D + D / 2 <= 256 ? 256 : 512;
    constexpr uint32_t O_COL = 2 * PF_KEYS;
    constexpr uint32_t Q_COL = O_COL + D;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *kv_full = reinterpret_cast<uint64_t *>(sm);   // [PF_MAX_BUF]
    uint64_t *kv_empty = kv_full + PF_MAX_BUF;               // [PF_MAX_BUF]
    uint64_t *s_full = kv_full + 2 * PF_MAX_BUF;             // [2]
    uint64_t *s_empty = s_full + 2;                          // [2]
    uint64_t *p_full = s_full + 4;   // [2] P of a tile written
    uint64_t *pv_done = s_full + 6;  // [2] a tile's P.V complete
    uint64_t *q_full = s_full + 8;
    // separate K and V: K slot i is free once the scores have read it, V
    // slot i once the P.V has (kv_full / kv_empty then serve the K slots)
    uint64_t *v_full = s_full + 9;                           // [PF_MAX_BUF]
    uint64_t *v_empty = v_full + PF_MAX_BUF;                 // [PF_MAX_BUF]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 256);
    volatile int *abort_f = reinterpret_cast<volatile int *>(sm + 260);
    uint8_t *ps = sm + PF_CTRL;
    uint8_t *kvs = ps + PF_PBYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group, tpt = PF_ROWS / G;
    const int tile = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const bool alias = p.alias != 0;
    const int NB = p.num_buffers;
    // P buffers: tile i's P in buffer i % NPB; with fp32 output the second
    // half holds the residual of the one buffer
    const int NPB = p.out_f32 ? 1 : 2;
    const int KVB = alias ? KV_TILE : 2 * KV_TILE;  // one buffer: K [+ V]

    if (threadIdx.x == 0 && tile == 0 && kvh == 0) {
        if (p.seq_lens[b] > p.max_seq_len)
            record_error(p.err, PKV_DEV_LEN_BOUND);
        const int n = p.q_start[b + 1] - p.q_start[b];
        if (n > p.max_q_len || n > p.seq_lens[b] || n < 0)
            record_error(p.err, PKV_DEV_LEN_BOUND);
        if (p.ring_blocks == 0 && p.seq_lens[b] > p.max_blocks * kBlock)
            record_error(p.err, PKV_DEV_LEN_TABLE);
    }
    ChunkTile ct;
    if (!chunk_tile(p, b, tile, tpt, ct))
        return;  // uniform over the CTA: nothing to compute

    if (threadIdx.x == 0) {
        for (int i = 0; i < PF_MAX_BUF; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&p_full[i], 4);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(q_full, 4);  // the softmax warps, once Q is in TMEM
        *abort_f = 0;
        fence_barrier_init();
    }
    if (warp == PF_MMA_WARP)
        tmem_alloc(tmem_slot, TMEM_COLS);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto waitb = [&](uint64_t *bar, uint32_t parity) {
        if (*abort_f)
            return false;
        if (!mbar_wait_spin(bar, parity, p.err)) {
            *abort_f = 1;
            return false;
        }
        return true;
    };

    if (warp == PF_TMA_WARP) {
        // ---------------------------------------------------------- loads
        const uint64_t pol = policy_evict_first();
        int last_use = -1;
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            if (!alias)
                prefetch_tensormap(&tmv);
        }
        TableCursor tcur;
        tcur.init(p.block_table + static_cast<size_t>(b) * p.max_blocks, ct.blk0, ct.nblk,
                  p.ring_blocks, lane);
        for (int i = 0; i < ct.T; ++i) {
            const int buf = i % NB;
            const bool room = i < NB || waitb(&kv_empty[buf], ((i / NB) - 1) & 1);
            if (!__all_sync(FULL_MASK, room))
                break;
            int row[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int blk = i * 4 + t;
                const int phys = blk < ct.nblk ? tcur.get(blk, lane) : -1;
                const bool valid = static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
                if (blk < ct.nblk && !valid && lane == 0)
                    record_error(p.err, PKV_DEV_BAD_BLOCK);
                row[t] = valid ? phys * kBlock : p.num_blocks * kBlock;  // zero fill
            }
            // lanes (t, c): block t, 64-dim chunk c of the K (or K == V) tile,
            // then of the V tile once its slot is free
            const int nbox = 4 * NCH;
            for (int which = 0; which < (alias ? 1 : 2); ++which) {
                if (which == 1) {
                    const bool vroom = i < NB || waitb(&v_empty[buf], ((i / NB) - 1) & 1);
                    if (!__all_sync(FULL_MASK, vroom))
                        break;
                }
                uint64_t *fullb = which ? &v_full[buf] : &kv_full[buf];
                if (lane == 0)
                    mbar_arrive_expect_tx(fullb, KV_TILE);
                __syncwarp();
                for (int k = lane; k < nbox; k += 32) {
                    const int t = k / NCH, c = k % NCH;
                    const int rt = t == 0 ? row[0] : t == 1 ? row[1] : t == 2 ? row[2] : row[3];
                    uint8_t *dst = kvs + buf * KVB + which * KV_TILE + c * PF_KCHUNK + t * 2048;
                    tma_load_3d(dst, which ? &tmv : &tmk, c * 64, kvh, rt, fullb, pol);
                }
                __syncwarp();
            }
            last_use = i;
        }
        if (lane == 0) {
            if (last_use >= 0) {
                mbar_wait(&kv_full[last_use % NB], (last_use / NB) & 1, p.err, 100000000ull);
                if (!alias)
                    mbar_wait(&v_full[last_use % NB], (last_use / NB) & 1, p.err, 100000000ull);
            }
        }
    } else if (warp == PF_MMA_WARP) {
        // ---------------------------------------------------------- MMAs
        constexpr uint32_t IDESC_QK = umma_idesc_bf16(PF_ROWS, PF_KEYS, false, false);
        constexpr uint32_t IDESC_PV = umma_idesc_bf16(PF_ROWS, D, false, true);
        const uint32_t p_base = smem_u32(ps), kv_base = smem_u32(kvs);
        bool ok = waitb(q_full, 0);
        tc_fence_after();
        auto pv = [&](int j) {
            // V rows of keys no row may see (before lo, after the last token)
            // inside this tile's loaded blocks: zero them, so 0 * stale = 0
            const int key0 = (ct.blk0 + j * 4) * kBlock;
            const int za = max(0, min(PF_KEYS, ct.lo - key0));
            const int zb = max(0, min(PF_KEYS, ct.last + 1 - key0));
            const int pbuf = j % NPB;
            bool go = waitb(&p_full[pbuf], (j / NPB) & 1);
            if (!alias)
                go = go && waitb(&v_full[j % NB], (j / NB) & 1);
            if (!__all_sync(FULL_MASK, go))
                return false;
            uint8_t *vt = kvs + (j % NB) * KVB + (alias ? 0 : KV_TILE);
            if (za > 0 || zb < PF_KEYS) {
                for (int idx = lane; idx < PF_KEYS * NCH * 8; idx += 32) {
                    const int r = idx / (NCH * 8), c = (idx / 8) % NCH, q16 = idx & 7;
                    if (r < za || r >= zb)
                        *reinterpret_cast<uint4 *>(vt + c * PF_KCHUNK + r * 128 + q16 * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
                tc_fence_after();
                const uint32_t v_base = smem_u32(vt);
                for (int pass = 0; pass < (p.out_f32 ? 2 : 1); ++pass) {
#pragma unroll
                    for (int kk = 0; kk < PF_KEYS / 16; ++kk) {
                        const uint64_t a = umma_smem_desc(
                            p_base + (pbuf + pass) * PF_PROW + kk * 32, 16, 1024);
                        const uint64_t bv = umma_smem_desc(v_base + kk * 2048, PF_KCHUNK, 1024);
                        umma_bf16(tmem + O_COL, a, bv, IDESC_PV, j > 0 || pass > 0 || kk > 0);
                    }
                }
                umma_commit(&pv_done[pbuf]);
                umma_commit(alias ? &kv_empty[j % NB] : &v_empty[j % NB]);
            }
            __syncwarp();
            return true;
        };
        for (int i = 0; i < ct.T && ok; ++i) {
            const int buf = i % NB, sb = i & 1;
            // The previous tile's P.V goes first when this tile's data has not
            // landed yet: the softmax waits for that P.V, not for these loads.
            bool prev_done = i == 0;
            if (!prev_done) {
                const bool landed = __shfl_sync(
                    FULL_MASK, lane == 0 ? mbar_test(&kv_full[buf], (i / NB) & 1) : false, 0);
                if (!landed) {
                    ok = pv(i - 1);
                    prev_done = true;
                    if (!ok)
                        break;
                }
            }
            ok = waitb(&kv_full[buf], (i / NB) & 1);
            ok = ok && (i < 2 || waitb(&s_empty[sb], ((i >> 1) - 1) & 1));
            ok = __all_sync(FULL_MASK, ok);
            if (!ok)
                break;
            if (lane == 0) {
                tc_fence_after();
                const uint32_t k_base = kv_base + buf * KVB;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t bk = umma_smem_desc(
                        k_base + (kk >> 2) * PF_KCHUNK + (kk & 3) * 32, 16, 1024);
                    umma_bf16_ts(tmem + sb * PF_KEYS, tmem + Q_COL + kk * 8, bk, IDESC_QK, kk > 0);
                }
                umma_commit(&s_full[sb]);
                if (!alias)
                    umma_commit(&kv_empty[buf]);  // the K slot is free once read
            }
            __syncwarp();
            if (!prev_done)
                ok = pv(i - 1);
        }
        if (ok && ct.T > 0)
            pv(ct.T - 1);
    } else {
        // ---------------------------------------------------------- softmax
        const int r = threadIdx.x;  // query row == TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const int t = r / G;
        const bool valid = t < ct.nt;
        const int pos = ct.len - ct.n + ct.t0 + t;
        const int lo_r = p.window > 0 ? max(0, pos - p.window) : 0;
        const float qk = p.qk_scale_log2;
        // ---- this row of Q into TMEM (zeros for rows past the chunk): the
        // score MMAs read their A operand there
        {
            const uint4 *qrow = reinterpret_cast<const uint4 *>(
                p.q + (static_cast<size_t>(ct.q0 + ct.t0 + t) * p.num_q_heads + kvh * G + r % G) * D);
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 16) {  // 16 columns = 32 dims = four 16-byte loads
                float v[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 u = valid ? __ldg(qrow + c0 / 4 + k) : make_uint4(0u, 0u, 0u, 0u);
                    v[4 * k] = __uint_as_float(u.x);
                    v[4 * k + 1] = __uint_as_float(u.y);
                    v[4 * k + 2] = __uint_as_float(u.z);
                    v[4 * k + 3] = __uint_as_float(u.w);
                }
                tmem_st<16>(lane_base + Q_COL + c0, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(q_full);
        }
        float m = -INFINITY, l = 0.f;
        bool live = true;
        for (int i = 0; i < ct.T; ++i) {
            const int sb = i & 1;
            live = live && waitb(&s_full[sb], (i >> 1) & 1);
            live = __all_sync(FULL_MASK, live);  // TMEM loads below are warp-collective
            tc_fence_after();
            float s[PF_KEYS];
            if (live) {
#pragma unroll
                for (int c0 = 0; c0 < PF_KEYS; c0 += 16) {
                    float v[16];
                    tmem_ld16(lane_base + sb * PF_KEYS + c0, v);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        s[c0 + k] = v[k];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&s_empty[sb]);
            const int key0 = (ct.blk0 + i * 4) * kBlock;
            float mt = -INFINITY;
            // every key of the tile visible to this row: no per-key tests
            const bool all_in = live && valid && key0 >= lo_r && key0 + PF_KEYS - 1 <= pos &&
                                (i + 1) * 4 <= ct.nblk;
            if (all_in) {
#pragma unroll
                for (int k = 0; k < PF_KEYS; ++k) {
                    s[k] *= qk;
                    mt = fmaxf(mt, s[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < PF_KEYS; ++k) {
                    const int j = key0 + k;
                    const bool ok = live && valid && j >= lo_r && j <= pos &&
                                    (j - ct.blk0 * kBlock) < ct.nblk * kBlock;
                    s[k] = ok ? s[k] * qk : -INFINITY;
                    mt = fmaxf(mt, s[k]);
                }
            }
            // this tile's P buffer was last read by the P.V of tile i - NPB
            if (i >= NPB)
                live = live && waitb(&pv_done[(i - NPB) % NPB], ((i - NPB) / NPB) & 1);
            live = __all_sync(FULL_MASK, live);
            // a new reference max for this row when a score exceeds the old by
            // more than 2^8; O's row (through the previous tile) is scaled in
            // place by the thread that owns it -- the TMEM accesses are
            // warp-collective, so the warp does them if any row needs them
            // and the other rows scale by 1
            const bool grow = mt > m + 8.f;
            const float alpha = !grow ? 1.f : (m == -INFINITY ? 0.f : fast_exp2(m - mt));
            if (__any_sync(FULL_MASK, grow && m != -INFINITY) && i >= 1 && live) {
                // O through the previous tile must be complete before scaling
                live = waitb(&pv_done[(i - 1) % NPB], ((i - 1) / NPB) & 1);
                live = __all_sync(FULL_MASK, live);
            }
            if (__any_sync(FULL_MASK, grow && m != -INFINITY) && i >= 1 && live) {
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 16) {
                    float o[16];
                    tmem_ld16(lane_base + O_COL + c0, o);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        o[k] *= alpha;
                    tmem_st<16>(lane_base + O_COL + c0, o);
                }
                tc_fence_before();
            }
            if (grow) {
                l *= alpha;
                m = mt;
            }
            // probabilities of the row, written as one 128-byte swizzled row;
            // for fp32 output also the bf16 residual p - bf16(p), multiplied
            // in a second P.V pass (error near 2^-17 instead of 2^-9)
            uint8_t *pbuf = ps + (i % NPB) * PF_PROW;
            auto put_p = [&](auto residual) {
#pragma unroll
                for (int c16 = 0; c16 < PF_KEYS / 8; ++c16) {
                    uint32_t w[4], wl[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x0 = s[c16 * 8 + 2 * e], x1 = s[c16 * 8 + 2 * e + 1];
                        const float p0 = x0 == -INFINITY ? 0.f : fast_exp2(x0 - m);
                        const float p1 = x1 == -INFINITY ? 0.f : fast_exp2(x1 - m);
                        l += p0 + p1;
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                        w[e] = *reinterpret_cast<uint32_t *>(&h2);
                        if constexpr (decltype(residual)::value) {
                            const float2 back = __bfloat1622float2(h2);
                            __nv_bfloat162 l2 = __floats2bfloat162_rn(p0 - back.x, p1 - back.y);
                            wl[e] = *reinterpret_cast<uint32_t *>(&l2);
                        }
                    }
                    *reinterpret_cast<uint4 *>(pbuf + pf_swz(r, c16)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                    if constexpr (decltype(residual)::value)
                        *reinterpret_cast<uint4 *>(ps + PF_PROW + pf_swz(r, c16)) =
                            make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
            };
            if (p.out_f32)
                put_p(std::true_type{});
            else
                put_p(std::false_type{});
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&p_full[i % NPB]);
        }
        // ---- the row's output: O / l after the last P.V
        if (ct.T > 0)
            live = live && waitb(&pv_done[(ct.T - 1) % NPB], ((ct.T - 1) / NPB) & 1);
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t orow = (static_cast<size_t>(ct.q0 + ct.t0 + t) * p.num_q_heads +
                             kvh * G + r % G) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
            float o[16];
            tmem_ld16(lane_base + O_COL + c0, o);
            if (valid && live) {
                if (p.out_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + orow + c0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_float4(o[4 * k] * inv, o[4 * k + 1] * inv, o[4 * k + 2] * inv,
                                             o[4 * k + 3] * inv);
                } else {
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * k] * inv, o[2 * k + 1] * inv);
                        w[k] = *reinterpret_cast<uint32_t *>(&h2);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + orow + c0);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == PF_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------ host side
static size_t prefill_fixed_bytes(int head_dim)
{
    return 1024 + PF_CTRL + PF_PBYTES;  // Q lives in TMEM
}

int prefill_num_buffers(int head_dim, int alias)
{
    const size_t tile = static_cast<size_t>(head_dim / 64) * PF_KCHUNK * (alias ? 1 : 2);
    const size_t room = 227u * 1024u - prefill_fixed_bytes(head_dim);
    const int nb = static_cast<int>(room / tile);
    return nb < PF_MAX_BUF ? nb : PF_MAX_BUF;
}

size_t prefill_smem_bytes(int head_dim, int alias, int num_buffers)
{
    return prefill_fixed_bytes(head_dim) +
           static_cast<size_t>(num_buffers) * (head_dim / 64) * PF_KCHUNK * (alias ? 1 : 2);
}

template <int D>
static cudaError_t launch_prefill_d(const PrefillParams &p, const CUtensorMap &tmk,
                                    const CUtensorMap &tmv, const CUtensorMap &tmq, dim3 grid,
                                    cudaStream_t s)
{
    const size_t smem = prefill_smem_bytes(D, p.alias, p.num_buffers);
    auto kern = prefill_tc_kernel<D>;
    static std::atomic<int> configured{0};
    if (static_cast<int>(smem) > configured.load(std::memory_order_relaxed)) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured.store(static_cast<int>(smem), std::memory_order_relaxed);
    }
    kern<<<grid, PF_THREADS, smem, s>>>(p, tmk, tmv, tmq);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           const CUtensorMap &tmq, int head_dim, cudaStream_t s)
{
    const int tiles = (p.max_q_len * p.group + PF_ROWS - 1) / PF_ROWS;
    const dim3 grid(tiles, p.num_kv_heads, p.batch);
    switch (head_dim) {
    case 64: return launch_prefill_d<64>(p, tmk, tmv, tmq, grid, s);
    case 128: return launch_prefill_d<128>(p, tmk, tmv, tmq, grid, s);
    case 256: return launch_prefill_d<256>(p, tmk, tmv, tmq, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
