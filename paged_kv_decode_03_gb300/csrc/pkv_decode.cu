// pkv_decode.cu -- CUDA-core decode attention over a paged KV pool.
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
//     block) into an NS-stage shared-memory ring guarded by mbarriers, with
//     separate K and V slots; all four consumer warps work on every stage
//     (a quarter of its keys each) and keep independent online-softmax
//     states that merge at the end.
//   * A lane owns one 16-byte chunk of a key row (8 bf16 or 16 int8
//     values; 8-byte chunks where four heads per CTA would otherwise hold
//     too many q and o values per lane), so head_dim spans LPK = row bytes /
//     chunk bytes lanes and a warp reads 32/LPK keys at once with vector
//     shared loads.  The partial dot products of a lane's keys x GT heads
//     finish with one butterfly reduce-scatter inside its LPK-lane group;
//     P.V accumulates per lane and the key groups are summed once at the end.
//   * int8 with two or more heads per CTA, where unpacking makes each key's
//     work long and registers scarce: each partial score goes to shared
//     memory as it is formed and lane i sums row i of that transpose, and
//     the P.V weights are read back from shared memory as (p, p) pairs
//     (measured 68% -> 77% of the HBM copy bandwidth on the Gemma4 sliding
//     layer with int8 KV).
//   * The running max is warp-uniform, so o and l are rescaled only in
//     stages where a max grows.
//   * Keys outside [lo, pos] in the first/last block are masked with a
//     select (never arithmetic), so stale or NaN slots contribute nothing.
#include <cuda_bf16.h>
#include <limits.h>
#include <math.h>

#include <atomic>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int NC = 4;                    // consumer warps per CTA
constexpr int THREADS = (NC + 1) * 32;   // + one producer warp
// Start of smem: mbarriers (512 B) and stage masks (64 B); at PW_OFF the
// consumer warps' P.V weights of a stage (NC x at most 32 x 8 B); at RED_OFF
// the int8 score transposes (Cfg::RED_BYTES, instances with a GQA tile); the
// ring after them.
constexpr int PW_OFF = 640;
constexpr int RED_OFF = PW_OFF + NC * 32 * 8;
constexpr int BAR_BYTES = RED_OFF;

// Paged blocks per ring stage: about 8 KB of K per stage (int8: at least four
// blocks, i.e. 16 keys per consumer warp, since unpacking makes its per-key
// work larger and the per-stage costs must be spread over more keys), and at
// most 8 / GT so that one reduce-scatter covers a warp's dot products.
__host__ __device__ constexpr int blocks_per_stage(int tile, int gt, bool int8)
{
    const int by_bytes = 8192 / tile;
    const int least = int8 ? 4 : 1;
    const int want = by_bytes > least ? by_bytes : least;
    return want < 8 / gt ? want : 8 / gt;
}

#ifndef PKV_CHUNK_RULE
#define PKV_CHUNK_RULE ((INT8 ? GT >= 4 : (GT >= 4 && D <= 128)) ? 8 : 16)
#endif

struct KeyRange {
    int lo, pos, blk_lo, nblk, nsplit;
};

// Keys a decode at position len-1 may attend to, and the block-aligned
// split of that range.
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
    static constexpr int ES = INT8 ? 1 : 2;                    // element bytes
    static constexpr int CHE = (D * ES > 256) ? 256 / ES : D;  // elements per TMA box row
    static constexpr int NCH = D / CHE;                         // boxes per tile
    static constexpr int ROWB = CHE * ES;                       // bytes of one box row
    static constexpr int TILE = P * D * ES;                     // one kv head x one block
    // A lane owns one CB-byte chunk of a key row: EPL elements, NPR pairs.
    // 8-byte chunks where 16 would hold 32 or more q (and o) values per lane
    // over the GT heads (registers, hence CTAs per SM); 16 bytes elsewhere.
    static constexpr int CB = PKV_CHUNK_RULE;
    static constexpr int EPL = CB / ES;
    static constexpr int NPR = EPL / 2;
    static constexpr int LPK = D / EPL;                         // lanes per key row
    static constexpr int KG = 32 / LPK;                         // keys a warp reads at once
    static constexpr int BPS = blocks_per_stage(TILE, GT, INT8);
    static constexpr int KEYS = P * BPS;                        // keys per stage
    static constexpr int KPW = KEYS / NC;                       // keys per warp per stage
    static constexpr int KPL = KPW / KG;                        // keys per lane per stage
    static constexpr int NV = KPL * GT;                         // dot products per lane
    static constexpr int DUP = LPK / NV;                        // lanes holding each sum
    static_assert(D % EPL == 0 && LPK >= 4 && LPK <= 32, "head_dim");
    static_assert(KPL >= 1 && KPW % KG == 0, "keys per lane");
    static_assert(NV >= 1 && NV <= LPK && LPK % NV == 0, "reduction width");
    static_assert(KPW <= P || KPW % P == 0, "warp keys within or across whole blocks");
    static_assert(KPW * GT <= 32, "weights of a warp's stage fit its PW_OFF slice");
    // int8 with a GQA tile: the scores' cross-lane sums go through shared
    // memory (a transpose) instead of a shuffle reduce-scatter
    static constexpr bool RED = INT8 && GT >= 2 && NV == LPK && (LPK == 8 || LPK == 16);
    static constexpr int RED_KG = NV * LPK + LPK;               // floats per key group
    static constexpr int RED_BYTES = RED ? NC * KG * RED_KG * 4 : 0;
};

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Bytes of one ring slot: bps K (or V) tiles plus their per-token scales.
__host__ __device__ inline int slot_bytes(int tile, int bps, int per_token)
{
    return round_up(bps * tile + (per_token ? bps * 64 : 0), 128);
}


// Butterfly reduce-scatter of NV per-lane partial sums within aligned groups
// of W lanes (NV <= W, both powers of two): after log2(NV) halving steps lane
// l holds value index (l % W) / (W / NV) summed over the lanes of its group
// that share those bits; the remaining xor steps complete the sum, so the
// W / NV lanes of each value hold its full sum.  NV - 1 + log2(W / NV)
// shuffles for NV dot products.
template <int NV, int W>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane)
{
#pragma unroll
    for (int half = NV / 2, off = W / 2; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            float send = upper ? v[i] : v[i + half];
            float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL_MASK, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = W / NV / 2; off >= 1; off >>= 1)
        r += __shfl_xor_sync(FULL_MASK, r, off);
    return r;
}

// CB (8 or 16) bytes of a tile row as float2 pairs (exact).  bf16: the two
// halves of each 32-bit word.  int8: each byte b is placed in the low
// mantissa bits of 2^23 (after flipping its sign bit, giving b+128) and
// 2^23+128 is subtracted, which yields b exactly.
template <bool INT8, int CB>
__device__ __forceinline__ void load_chunk(const uint8_t *p, float2 (&f)[INT8 ? CB / 2 : CB / 4])
{
    constexpr int NW = CB / 4;
    uint32_t w[NW];
    if constexpr (CB == 16) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else {
        static_assert(CB == 8, "chunk bytes");
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        w[0] = u.x; w[1] = u.y;
    }
    if constexpr (!INT8) {
#pragma unroll
        for (int i = 0; i < NW; ++i)
            f[i] = make_float2(bf16lo(w[i]), bf16hi(w[i]));
    } else {
        const float2 bias = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
        for (int i = 0; i < 2 * NW; ++i) {
            const uint32_t x = w[i / 2] ^ 0x80808080u;
            const int b0 = (i % 2) * 2;
            const float lo = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540 + b0));
            const float hi = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540 + b0 + 1));
            f[i] = __fadd2_rn(make_float2(lo, hi), bias);
        }
    }
}

template <int D, int GT, bool INT8>
__device__ __forceinline__ void decode_body(const DecodeParams &p, const CUtensorMap *tmk,
                                            const CUtensorMap *tmv)
{
    using C = Cfg<D, GT, INT8>;
    constexpr int BPS = C::BPS;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *kfull = reinterpret_cast<uint64_t *>(smem);
    uint64_t *kempty = kfull + 16;
    uint64_t *vfull = kfull + 32;
    uint64_t *vempty = kfull + 48;
    uint32_t *smask = reinterpret_cast<uint32_t *>(kfull + 64);  // valid blocks per stage
    uint8_t *ring = smem + BAR_BYTES + C::RED_BYTES;
    float *red = reinterpret_cast<float *>(smem + RED_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y / p.head_chunks;
    const int chunk = blockIdx.y - g * p.head_chunks;
    // in order, or the order kernel's (sequence, length) pair: one load either way
    int b, len;
    if (p.seq_order) {
        pdl_wait();  // the order kernel has completed
        const int2 e = reinterpret_cast<const int2 *>(p.seq_order)[blockIdx.z];
        b = e.x;
        len = e.y;
    } else {
        b = blockIdx.z;
        len = p.seq_lens[b];
    }
    const int NS = p.num_stages;
    const bool alias = p.alias != 0;
    const bool per_token = INT8 && p.scale_mode == PKV_SCALE_PER_TOKEN;
    const bool per_head = INT8 && p.scale_mode == PKV_SCALE_PER_HEAD;
    const int KS = slot_bytes(C::TILE, BPS, per_token);
    const int SB = alias ? KS : 2 * KS;  // one stage: K slot [+ V slot]

    const bool reporter = threadIdx.x == 0 && split == 0 && blockIdx.y == 0;
    if (p.ring_blocks == 0 && len > p.max_blocks * C::P) {  // a ring does not bound the length
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
    const int n = max(0, ub1 - ub0);          // paged blocks of this unit
    const int nst = (n + BPS - 1) / BPS;      // ring stages of this unit
    const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], NC);
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], NC);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NC) {
        // ------------------------------------------------------ producer
        // The producer warp walks the stages in order.  Lane 0 fills the K
        // slot of stage s % NS as soon as the consumers have formed the
        // scores of its previous contents, then the V slot as soon as the
        // previous P.V on it is done, and publishes which blocks of the
        // stage hold data; the other lanes only help read the block table.
        if (nst > 0) {
            if (lane == 0) {
                prefetch_tensormap(tmk);
                if (!alias)
                    prefetch_tensormap(tmv);
            }
            const uint64_t pol = policy_evict_first();
            TableCursor tc;
            tc.init(bt_row, ub0, n, p.ring_blocks, lane);
            int issued[2] = {0, 0};
            bool ok = true;
            int st = 0;             // ring slot of stage sidx
            uint32_t rpar = 0;      // parity of the ring round of stage sidx
            for (int sidx = 0; sidx < nst && ok; ++sidx) {
                int phys[BPS];
                uint32_t tx = 0, vm = 0;
#pragma unroll
                for (int t = 0; t < BPS; ++t) {
                    const int i = sidx * BPS + t;
                    phys[t] = i < n ? tc.get(i, lane) : -1;
                    const bool valid = static_cast<unsigned>(phys[t]) <
                                       static_cast<unsigned>(p.num_blocks);
                    if (!valid && i < n && lane == 0)
                        record_error(p.err, PKV_DEV_BAD_BLOCK);
                    if (!valid) {
                        phys[t] = -1;
                    } else {
                        tx += C::TILE + (per_token ? 64u : 0u);
                        vm |= 1u << t;
                    }
                }
                for (int which = 0; which < (alias ? 1 : 2); ++which) {
                    uint64_t *fullb = which == 0 ? kfull : vfull;
                    uint64_t *emptyb = which == 0 ? kempty : vempty;
                    if (sidx >= NS && !mbar_wait(&emptyb[st], rpar ^ 1u, p.err)) {
                        ok = false;
                        break;
                    }
                    issued[which] = sidx + 1;
                    if (lane != 0)
                        continue;
                    if (which == 0)
                        smask[st] = vm;  // released by the arrive below
                    mbar_arrive_expect_tx(&fullb[st], tx);
                    uint8_t *dst = ring + st * SB + which * KS;
                    const CUtensorMap *map = which == 0 ? tmk : tmv;
                    const float *scales = which == 0 ? p.k_scale : p.v_scale;
#pragma unroll
                    for (int t = 0; t < BPS; ++t) {
                        if (phys[t] < 0)
                            continue;
                        const int row0 = phys[t] * C::P;
#pragma unroll
                        for (int ch = 0; ch < C::NCH; ++ch)
                            tma_load_3d(dst + t * C::TILE + ch * C::P * C::ROWB, map, ch * C::CHE,
                                        g, row0, &fullb[st], pol);
                        if (per_token)
                            bulk_load(dst + BPS * C::TILE + t * 64, scales + row0, 64, &fullb[st]);
                    }
                }
                ok = __all_sync(FULL_MASK, ok);
                if (++st == NS) {
                    st = 0;
                    rpar ^= 1u;
                }
            }
            // Drain: do not let the CTA retire with copies in flight.
            if (lane == 0)
                for (int which = 0; which < 2; ++which)
                    for (int i = max(0, issued[which] - NS); i < issued[which]; ++i)
                        mbar_wait(&(which == 0 ? kfull : vfull)[i % NS], (i / NS) & 1, p.err,
                                  100000000ull);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // Every consumer warp works on every stage: warp w takes the stage's
    // keys [w*KPW, (w+1)*KPW), so a stage is released after a quarter of
    // its work and the rest of the ring stays in flight.  Within a warp,
    // lane (kg, dl) owns the CB-byte chunk dl of a key row and reads keys
    // kg, kg+KG, kg+2KG, ... of the warp's share: consecutive lanes read
    // consecutive bytes, and the score reductions stay within the LPK lanes
    // of one key.
    constexpr int NPR = C::NPR, NV = C::NV, KPW = C::KPW, KPL = C::KPL, KG = C::KG;
    constexpr int LPK = C::LPK, DUP = C::DUP;
    const int G = p.group;
    const int kg = lane / LPK, dl = lane % LPK;
    const int lane_elem = dl * C::EPL;
    const int lane_off = (lane_elem / C::CHE) * C::P * C::ROWB + (lane_elem % C::CHE) * C::ES;
    const int k0w = warp * KPW;   // this warp's first key within a stage
    const int kb = k0w + kg;      // this lane's first key within a stage
    // Slot offset of this lane's key r = its first key's offset + koff(r): KG
    // divides P and KPW is a divisor or a multiple of P, so the keys
    // kb + KG*r never straddle a block differently from KG*r.
    const int lane_base = (k0w / C::P) * C::TILE + (k0w % C::P + kg) * C::ROWB + lane_off;
    auto koff = [](int r) { return ((KG * r) / C::P) * C::TILE + ((KG * r) % C::P) * C::ROWB; };

    float2 qf[GT][NPR];
    {
        float qmul = p.qk_scale_log2;
        if (per_head)
            qmul *= p.k_scale[g];
#pragma unroll
        for (int h = 0; h < GT; ++h) {
            const int hl = chunk * GT + h;
            if (hl < G) {
                const uint8_t *qr = reinterpret_cast<const uint8_t *>(
                    p.q + (static_cast<size_t>(b) * p.num_q_heads + g * G + hl) * D + lane_elem);
#pragma unroll
                for (int c = 0; c < NPR / 2; ++c) {
                    float2 t[2];
                    load_chunk<false, 8>(qr + 8 * c, t);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        qf[h][2 * c + i] = make_float2(t[i].x * qmul, t[i].y * qmul);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NPR; ++i)
                    qf[h][i] = make_float2(0.f, 0.f);
            }
        }
    }

    float2 o[GT][NPR];
    float m[GT];
#pragma unroll
    for (int h = 0; h < GT; ++h) {
        m[h] = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPR; ++i)
            o[h][i] = make_float2(0.f, 0.f);
    }
    float l_lane = 0.f;
    const int my_idx = dl / DUP;            // value index this lane holds
    const int my_h = my_idx / KPL, my_r = my_idx % KPL;
    const int km = kb + KG * my_r;          // its key within a stage
    const bool l_owner = (dl % DUP) == 0;   // one lane per value adds to l
    const uint32_t km_bit = 1u << (km / C::P);  // its block within a stage
    // the blocks of a stage that hold this warp's keys
    uint32_t wmask = 0;
#pragma unroll
    for (int t = 0; t < BPS; ++t)
        if (t * C::P < k0w + KPW && (t + 1) * C::P > k0w)
            wmask |= 1u << t;
    // This key group's P.V weights of a stage, [key][head], each stored as a
    // (p, p) pair so that the packed FMAs take it as it is loaded.
    float2 *pw = reinterpret_cast<float2 *>(smem + PW_OFF) + (warp * KG + kg) * (KPL * GT);

    int st = 0;          // ring slot of stage sidx
    uint32_t par = 0;    // parity of its fill
    for (int sidx = 0; sidx < nst; ++sidx, st = (st + 1 == NS) ? 0 : st + 1, par ^= (st == 0)) {
        if (!__all_sync(FULL_MASK, mbar_wait(&kfull[st], par, p.err)))
            break;
        const uint32_t vmask = smask[st];  // blocks of the stage that hold data
        const uint8_t *kt = ring + st * SB;
        const uint8_t *vt = alias ? kt : kt + KS;
        const float *ksc = reinterpret_cast<const float *>(kt + BPS * C::TILE);
        const float *vsc = reinterpret_cast<const float *>(vt + BPS * C::TILE);
        const int jst = (ub0 + sidx * BPS) * C::P;  // key index of the stage's first row
        const int jw = jst + k0w;
        // all of this warp's keys hold data and lie in [lo, pos]
        const bool all_in = jw >= kr.lo && jw + KPW - 1 <= kr.pos && (vmask & wmask) == wmask;
        // ---- scores of this lane's KPL keys for the GT heads
        float s;
        if constexpr (C::RED) {
            // Each partial score goes to shared memory as soon as it is
            // formed (row v = value v, column = lane within the key group;
            // 4-float chunks xor-swizzled by row, so that the stores and the
            // chunked row reads are free of bank conflicts); lane dl then
            // sums row dl.
            constexpr int RPB = 32 / LPK;  // rows per 32 banks
            auto swz = [](int v) { return (v / RPB) & (LPK / 4 - 1); };
            float *rd = red + (warp * KG + kg) * C::RED_KG;
            auto put = [&](int v, float x) { rd[v * LPK + (dl ^ (swz(v) << 2))] = x; };
#pragma unroll
            for (int r = 0; r < KPL; ++r) {
                float2 kf[NPR];
                load_chunk<INT8, C::CB>(kt + lane_base + koff(r), kf);
#pragma unroll
                for (int h = 0; h < GT; ++h) {
                    float2 a = __fmul2_rn(qf[h][0], kf[0]);
#pragma unroll
                    for (int e = 1; e < NPR; ++e)
                        a = __ffma2_rn(qf[h][e], kf[e], a);
                    put(h * KPL + r, a.x + a.y);
                }
            }
            __syncwarp();
            const float4 *row = reinterpret_cast<const float4 *>(rd + dl * LPK);
            const int sw = swz(dl);
            float t0 = 0.f, t1 = 0.f;
#pragma unroll
            for (int c = 0; c < LPK / 4; ++c) {
                const float4 x = row[c ^ sw];
                t0 += x.x + x.y;
                t1 += x.z + x.w;
            }
            s = t0 + t1;
        } else {
            float acc[NV];
#pragma unroll
            for (int r = 0; r < KPL; ++r) {
                float2 kf[NPR];
                load_chunk<INT8, C::CB>(kt + lane_base + koff(r), kf);
#pragma unroll
                for (int h = 0; h < GT; ++h) {
                    float2 a = __fmul2_rn(qf[h][0], kf[0]);
#pragma unroll
                    for (int e = 1; e < NPR; ++e)
                        a = __ffma2_rn(qf[h][e], kf[e], a);
                    acc[h * KPL + r] = a.x + a.y;
                }
            }
            s = reduce_scatter<NV, LPK>(acc, lane);
        }
        const int jm = jst + km;
        const bool ok = (vmask & km_bit) && jm >= kr.lo && jm <= kr.pos;
        if (per_token)
            s *= ksc[km];
        s = ok ? s : -INFINITY;
        if (!alias) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&kempty[st]);
        }
        // ---- online softmax over the warp's KPW keys
        float mx = s;
#pragma unroll
        for (int off = DUP; off < DUP * KPL; off <<= 1)
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, off));
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1)
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, off));
        // m is warp-uniform (every lane takes it from the same lanes), so the
        // rescale below is a uniform branch taken only when a max grows.
        float alpha[GT];
        bool grow = false;
        float m_mine = 0.f, a_mine = 1.f;
#pragma unroll
        for (int h = 0; h < GT; ++h) {
            const float tm = __shfl_sync(FULL_MASK, mx, h * DUP * KPL);
            const float mn = fmaxf(m[h], tm);
            alpha[h] = 1.f;
            if (mn > m[h]) {
                grow = true;
                alpha[h] = (m[h] == -INFINITY) ? 0.f : fast_exp2(m[h] - mn);
                m[h] = mn;
            }
            if (h == my_h) {
                m_mine = m[h];
                a_mine = alpha[h];
            }
        }
        const float pr = ok ? fast_exp2(s - m_mine) : 0.f;
        if (grow) {
            l_lane *= a_mine;
#pragma unroll
            for (int h = 0; h < GT; ++h) {
                const float2 a2 = make_float2(alpha[h], alpha[h]);
#pragma unroll
                for (int e = 0; e < NPR; ++e)
                    o[h][e] = __fmul2_rn(o[h][e], a2);
            }
        }
        l_lane += l_owner ? pr : 0.f;
        if (!alias && !__all_sync(FULL_MASK, mbar_wait(&vfull[st], par, p.err)))
            break;
        float pv = pr;
        if (per_token)
            pv = ok ? pr * vsc[km] : 0.f;
        // ---- P.V over this lane's KPL keys
        if constexpr (INT8 && GT >= 2) {
            // int8: the weights go through shared memory as (p, p) pairs
            // (one load per key for all heads, no register moves to form the
            // pairs), and stages whose keys all count skip the masking
            if (l_owner)
                pw[my_r * GT + my_h] = make_float2(pv, pv);
            __syncwarp();
            auto pv_key = [&](int r) {
                float2 w2[GT];
                if constexpr (GT == 1) {
                    w2[0] = pw[r];
                } else {
#pragma unroll
                    for (int h = 0; h < GT; h += 2) {
                        const float4 t = *reinterpret_cast<const float4 *>(pw + r * GT + h);
                        w2[h] = make_float2(t.x, t.y);
                        w2[h + 1] = make_float2(t.z, t.w);
                    }
                }
                float2 vf[NPR];
                load_chunk<INT8, C::CB>(vt + lane_base + koff(r), vf);
#pragma unroll
                for (int h = 0; h < GT; ++h)
#pragma unroll
                    for (int e = 0; e < NPR; ++e)
                        o[h][e] = __ffma2_rn(w2[h], vf[e], o[h][e]);
            };
            if (all_in) {
#pragma unroll
                for (int r = 0; r < KPL; ++r)
                    pv_key(r);
            } else {
#pragma unroll
                for (int r = 0; r < KPL; ++r) {
                    // masked key: its slot may hold stale data, do not touch it
                    const int k = kb + KG * r;
                    const int j = jst + k;
                    if ((vmask >> (k / C::P) & 1u) && j >= kr.lo && j <= kr.pos)
                        pv_key(r);
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < KPL; ++r) {
                float w[GT];
#pragma unroll
                for (int h = 0; h < GT; ++h)
                    w[h] = __shfl_sync(FULL_MASK, pv, (h * KPL + r) * DUP, LPK);
                if (!all_in) {
                    // masked key: its slot may hold stale data, do not touch it
                    const int k = kb + KG * r;
                    const int j = jst + k;
                    if (!(vmask >> (k / C::P) & 1u) || j < kr.lo || j > kr.pos)
                        continue;
                }
                float2 vf[NPR];
                load_chunk<INT8, C::CB>(vt + lane_base + koff(r), vf);
#pragma unroll
                for (int h = 0; h < GT; ++h) {
                    const float2 w2 = make_float2(w[h], w[h]);
#pragma unroll
                    for (int e = 0; e < NPR; ++e)
                        o[h][e] = __ffma2_rn(w2, vf[e], o[h][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(alias ? &kempty[st] : &vempty[st]);
    }

    // sum o over the key groups, l over the lanes of each head
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
        for (int h = 0; h < GT; ++h)
#pragma unroll
            for (int e = 0; e < NPR; ++e) {
                o[h][e].x += __shfl_xor_sync(FULL_MASK, o[h][e].x, off);
                o[h][e].y += __shfl_xor_sync(FULL_MASK, o[h][e].y, off);
            }
    {
        float ls = l_lane;
#pragma unroll
        for (int off = 1; off < DUP * KPL; off <<= 1)
            ls += __shfl_xor_sync(FULL_MASK, ls, off);
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1)
            ls += __shfl_xor_sync(FULL_MASK, ls, off);
        l_lane = ls;
    }
    float lh[GT];
#pragma unroll
    for (int h = 0; h < GT; ++h)
        lh[h] = __shfl_sync(FULL_MASK, l_lane, h * DUP * KPL);

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
    if (kg == 0) {
#pragma unroll
        for (int h = 0; h < GT; ++h)
#pragma unroll
            for (int e = 0; e < NPR; ++e)
                *reinterpret_cast<float2 *>(&mrg_o[(warp * GT + h) * D + lane_elem + 2 * e]) =
                    o[h][e];
    }
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
            const size_t prow = (static_cast<size_t>(b) * p.num_splits + split) * p.num_q_heads + hq;
            p.part_o[prow * D + d] = y;
            if (d == 0)
                p.part_lse[prow] =
                    L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
        }
    }
}

// The kernels.  One query head per CTA has its own entry with at most 80
// registers, so that five CTAs fit an SM (left to itself the compiler takes
// 81 for the int8 head_dim-128 instance, which then runs four CTAs per SM and
// measured 6% slower).  The int8 two-head instances are bounded to three
// CTAs per SM (at most 136 registers; 1% faster than the compiler's choice on
// the Gemma4 sliding layer with int8 KV).  The others keep the compiler's
// choice: an explicit bound of one CTA makes it take more registers (the
// bf16 two-head instance then runs four CTAs per SM instead of five and
// measured 1-2% slower on the Gemma4 sliding layer).
template <int D, int GT, bool INT8>
__global__ void __launch_bounds__(THREADS) decode_kernel(const DecodeParams p,
                                                         const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv)
{
    decode_body<D, GT, INT8>(p, &tmk, &tmv);
}

template <int D>
__global__ void __launch_bounds__(THREADS, 3) decode_kernel_i8x2(const DecodeParams p,
                                                                const __grid_constant__ CUtensorMap tmk,
                                                                const __grid_constant__ CUtensorMap tmv)
{
    decode_body<D, 2, true>(p, &tmk, &tmv);
}

template <int D, bool INT8>
__global__ void __launch_bounds__(THREADS, 5) decode_kernel_1h(const DecodeParams p,
                                                               const __grid_constant__ CUtensorMap tmk,
                                                               const __grid_constant__ CUtensorMap tmv)
{
    decode_body<D, 1, INT8>(p, &tmk, &tmv);
}

template <int D, int GT, bool INT8>
constexpr auto decode_entry()
{
    if constexpr (GT == 1)
        return decode_kernel_1h<D, INT8>;
    else if constexpr (GT == 2 && INT8)
        return decode_kernel_i8x2<D>;
    else
        return decode_kernel<D, GT, INT8>;
}

// Sequences ordered by decreasing number of paged blocks in their key range
// (counting sort, one CTA): CTAs are dispatched in grid order, so with more
// CTAs than fit at once the longest ranges start first and the short ones
// fill the last wave.  Ties come out in any order (the results do not depend
// on the order in which CTAs run).
constexpr int ORDER_BINS = 4096;

__global__ void __launch_bounds__(1024) seq_order_kernel(const int32_t *seq_lens, int batch,
                                                         int window, int len_cap,
                                                         int2 *order)
{
    __shared__ int hist[ORDER_BINS];
    __shared__ int wsum[32];
    pdl_launch_dependents();
    auto key = [&](int b) {
        const int len = min(seq_lens[b], len_cap);
        const KeyRange kr = key_range(len, window, 0);
        return ORDER_BINS - 1 - min(kr.nblk, ORDER_BINS - 1);  // longest first
    };
    for (int i = threadIdx.x; i < ORDER_BINS; i += 1024)
        hist[i] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += 1024)
        atomicAdd(&hist[key(b)], 1);
    __syncthreads();
    // exclusive prefix over the bins: 4 per thread, warp shuffles, then warps
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int v[4], sum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[j] = hist[threadIdx.x * 4 + j];
        sum += v[j];
    }
    int x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(FULL_MASK, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(FULL_MASK, w, off);
            if (lane >= off)
                w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    int run = x - sum + (wid > 0 ? wsum[wid - 1] : 0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        hist[threadIdx.x * 4 + j] = run;
        run += v[j];
    }
    __syncthreads();
    for (int b = threadIdx.x; b < batch; b += 1024)
        order[atomicAdd(&hist[key(b)], 1)] = make_int2(b, seq_lens[b]);
}

// ------------------------------------------------------------ host side
int decode_group_tile(int group)
{
    return group >= 4 ? 4 : (group >= 2 ? (group == 2 ? 2 : 4) : 1);
}

template <int D>
static int red_bytes_d(int int8, int gt)
{
    if (!int8)
        return 0;
    return gt == 1 ? Cfg<D, 1, true>::RED_BYTES
                   : (gt == 2 ? Cfg<D, 2, true>::RED_BYTES : Cfg<D, 4, true>::RED_BYTES);
}

static int red_bytes(int head_dim, int int8, int gt)
{
    switch (head_dim) {
    case 64: return red_bytes_d<64>(int8, gt);
    case 128: return red_bytes_d<128>(int8, gt);
    default: return red_bytes_d<256>(int8, gt);
    }
}

size_t decode_smem_bytes(int head_dim, int int8, int alias, int per_token, int group_tile,
                         int num_stages)
{
    const int tile = kBlock * head_dim * (int8 ? 1 : 2);
    const int bps = blocks_per_stage(tile, group_tile, int8 != 0);
    const size_t ring = static_cast<size_t>(num_stages) * (alias ? 1 : 2) *
                        slot_bytes(tile, bps, per_token);
    const size_t merge = (2 * NC * group_tile + static_cast<size_t>(NC) * group_tile * head_dim) *
                         sizeof(float);
    return BAR_BYTES + red_bytes(head_dim, int8, group_tile) + (ring > merge ? ring : merge);
}

// Let the kernel use the opt-in maximum of dynamic shared memory (once).
template <int D, int GT, bool INT8>
static cudaError_t configure_smem()
{
    static std::atomic<int> done{0};
    if (done.load(std::memory_order_acquire))
        return cudaSuccess;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_entry<D, GT, INT8>(),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e == cudaSuccess)
        done.store(1, std::memory_order_release);
    return e;
}

// Ring depth: the most CTAs per SM first (registers or shared memory limit
// them; the consumer warps' dependency chains, not bytes in flight, limit a
// CTA), then the deepest ring (2..8 stages) that keeps that many.
template <int D, int GT, bool INT8>
static int ring_stages_one(int alias, int per_token)
{
    static std::atomic<int> cache[2][2];
    int v = cache[alias][per_token].load(std::memory_order_relaxed);
    if (v)
        return v;
    if (configure_smem<D, GT, INT8>() != cudaSuccess)
        return 2;
    int best = 2, best_occ = -1;
    for (int ns = 2; ns <= 8; ++ns) {
        const size_t smem = decode_smem_bytes(D, INT8, alias, per_token, GT, ns);
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_entry<D, GT, INT8>(),
                                                          THREADS, smem) != cudaSuccess ||
            occ < 1)
            break;
        if (occ >= best_occ) {
            best_occ = occ;
            best = ns;
        }
    }
    cache[alias][per_token].store(best, std::memory_order_relaxed);
    return best;
}

template <int D>
static int ring_stages_d(int int8, int alias, int per_token, int gt)
{
    if (int8) {
        if (gt == 1) return ring_stages_one<D, 1, true>(alias, per_token);
        if (gt == 2) return ring_stages_one<D, 2, true>(alias, per_token);
        return ring_stages_one<D, 4, true>(alias, per_token);
    }
    if (gt == 1) return ring_stages_one<D, 1, false>(alias, per_token);
    if (gt == 2) return ring_stages_one<D, 2, false>(alias, per_token);
    return ring_stages_one<D, 4, false>(alias, per_token);
}

int decode_ring_stages(int head_dim, int int8, int alias, int per_token, int group_tile)
{
    alias = alias != 0;
    per_token = per_token != 0;
    switch (head_dim) {
    case 64: return ring_stages_d<64>(int8, alias, per_token, group_tile);
    case 128: return ring_stages_d<128>(int8, alias, per_token, group_tile);
    case 256: return ring_stages_d<256>(int8, alias, per_token, group_tile);
    default: return 2;
    }
}

template <int D, int GT, bool INT8>
static cudaError_t launch_one(const DecodeParams &p, const CUtensorMap &tmk,
                              const CUtensorMap &tmv, cudaStream_t s)
{
    const size_t smem =
        decode_smem_bytes(D, INT8, p.alias, INT8 && p.scale_mode == PKV_SCALE_PER_TOKEN, GT,
                          p.num_stages);
    cudaError_t e = configure_smem<D, GT, INT8>();
    if (e != cudaSuccess)
        return e;
    dim3 grid(p.num_splits, p.num_kv_heads * p.head_chunks, p.batch);
    // More CTAs than fit at once (a single pass with ragged lengths is what
    // gains): order the sequences longest first, if the caller gave room.
    bool order = false;
    if (p.order_ws && p.split_blocks == 0 && p.batch > 1) {
        int occ = 0, dev = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_entry<D, GT, INT8>(),
                                                          THREADS, smem) == cudaSuccess &&
            cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            order = static_cast<int64_t>(grid.x) * grid.y * grid.z > static_cast<int64_t>(occ) * sms;
    }
    if (!order) {
        decode_entry<D, GT, INT8>()<<<grid, THREADS, smem, s>>>(p, tmk, tmv);
        note_launch();
        return cudaGetLastError();
    }
    seq_order_kernel<<<1, 1024, 0, s>>>(p.seq_lens, p.batch, p.window,
                                        p.ring_blocks ? INT_MAX : p.max_blocks * kBlock,
                                        reinterpret_cast<int2 *>(p.order_ws));
    note_launch();
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    note_launch();
    DecodeParams q = p;
    q.seq_order = p.order_ws;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_entry<D, GT, INT8>(), q, tmk, tmv);
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

}  // namespace pkv
