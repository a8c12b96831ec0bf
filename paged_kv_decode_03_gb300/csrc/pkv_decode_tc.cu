// pkv_decode_tc.cu -- decode attention over a bf16 paged KV pool on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM), run as a
// persistent stream-K kernel.
//
// Same problem and sources as pkv_decode.cu: y = softmax(scale * q K^T) V
// over the keys [lo, pos] of each sequence ("CS336 · 第 10 课", KV-cache
// section; "实验五：Gemma4 端到端推理优化", sliding-window, GQA and Flash
// Attention sections: online softmax with running max/sum in fp32, blocks
// outside the window never read).  Partial states of one key range, cut
// between CTAs or split by the caller, merge by the same max/sum recurrence
// ("LLM推理优化底层原理" §3.1 step 2) in log-sum-exp form.
//
// Why tensor cores here: at head_dim 256 the bf16 inner products of 8-16
// query heads cost the CUDA cores more issue slots than HBM needs time to
// deliver the bytes, so both contractions move to tcgen05 and the CUDA cores
// only do the softmax.
//
// Work decomposition (stream-K).  An item is one (sequence, kv head, split)
// key range (one split when the caller does not split); the 128-key tiles of
// all items, in (sequence, kv head, split, tile) order, each item followed by
// KAPPA virtual tiles that stand for its fixed cost, form one sequence of W
// units.  CTA c takes the units [c*W/C, (c+1)*W/C), C = min(grid, W),
// starting with the first item with real tiles there (or an empty item
// starting there); up to 8192 sequences each CTA derives that from the
// lengths itself, for larger batches tc_plan_kernel (one CTA) records it.
// tc_plan_kernel always clears the cut items' tickets and checks the lengths;
// the decode kernel, launched behind it with programmatic dependent launch,
// waits for it only before taking its first ticket.  A CTA walks its items
// in order with one pipeline that never drains between them; an item it
// covers entirely is finished in place (the output, or that split's partial
// state), an item cut at CTA boundaries leaves one partial state per CTA
// (log-sum-exp and normalised o) and a ticket: the part that finishes last
// merges them.  No CTA waits for another.  Every SM gets the same number of
// units within one, whatever the mix of lengths, and the per-CTA start-up
// (TMEM allocation, first loads) is paid once per SM instead of once per
// item.
//
// One CTA per SM, 16 warps:
//   warps 8-13 (producers): TMA loads of 128-key tiles into a ring of six
//     32 KB units.  With K and V separate the ring is split into a K ring
//     (read only by the score warp) and a V ring (read only by the P.V
//     warp); with K == V one ring is read by both in the same order, and
//     only the score warp waits for the loads (the P.V warp reads a unit
//     after the softmax published P for it, which follows the score MMAs
//     on it).  Each waiter thus waits on every phase of the slots it reads,
//     which is what makes parity waits sound.  Producer warp w owns slot w and
//     issues its uses in order; several issuing warps are needed because
//     the rate of 2 KB TMA boxes scales with the number of issuing warps.
//     Producer 0 also loads each item's Q^T (TMA, 128-byte swizzle) into one
//     of two buffers.
//   warp 14 (one thread): S^T[128 keys x 16] = K Q^T (M=128, N=16 query
//     heads padded, K=16 per instruction) into TMEM;
//   warp 15 (one thread): O^T[128 dims x 16] += V^T P^T per 128-dim half,
//     accumulated in TMEM over all tiles of an item (two O buffers, one per
//     item in flight).  tcgen05.commit signals the mbarriers that free ring
//     units, Q and P buffers and hand a finished item to the epilogue.
//   warps 0-3 (softmax): thread t owns key t of the tile (TMEM lane t):
//     loads its 16 scores, masks keys outside [lo, pos] (from the item's
//     geometry alone: the softmax reads no block table), keeps running max /
//     sums in fp32 and writes P^T in bf16 (K-major, swizzled) for the P.V
//     MMA -- for fp32 output also the bf16 residual p - bf16(p), multiplied
//     in a second pass, which keeps the error near 2^-17.  The running max
//     changes only when a score exceeds it by more than 2^8 (any reference
//     at least the true maximum minus 8 gives the same result and keeps
//     p <= 256); when it changes after an item's first tile, the softmax
//     scales the item's O in TMEM by 2^(m_old - m_new) once the previous
//     tile's P.V is done, before it publishes the new P.
//   warps 4-7 (epilogue): per item, once its last P.V is done, read O^T from
//     TMEM (thread t owns output dims t and 128+t), divide by the sum, and
//     store the output row, the split's partial state, or this CTA's part of
//     a cut item -- off the softmax's path, while the next item streams.
//   The P.V warp zeroes the V rows of masked keys inside loaded blocks
//   (stale slots past pos, keys before the window start) before its MMAs
//   read them, so no stale value (not even a NaN) reaches the output.
//   Q^T rows past the group hold other heads' queries (or zeros past the
//   end of q); their score columns are masked and their P^T rows stay zero.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int SOFTMAX_WARPS = 4;   // warps 0-3; TMEM lanes 0-127
constexpr int EPI_WARP = 4;        // warps 4-7: the epilogue warpgroup
constexpr int PRODUCER_WARP = 8;   // first producer warp
constexpr int PRODUCER_WARPS = 6;  // one per ring unit; TMA issue rate scales with issuing warps
constexpr int MMA_WARP = PRODUCER_WARP + PRODUCER_WARPS;  // issues the score MMAs, owns TMEM
constexpr int PV_WARP = MMA_WARP + 1;                     // issues the P.V MMAs
constexpr int TC_WARPS = PV_WARP + 1;
constexpr int TC_THREADS = TC_WARPS * 32;
constexpr int NPAD = 16;          // N of every MMA: query heads padded to 16
constexpr int UNIT = 32768;       // 128 keys x 128 dims bf16
constexpr int CHUNK = 16384;      // 128 keys x 64 dims bf16 (one swizzled column)
constexpr int CTRL = 1024;        // barriers, TMEM address, flags, exchange
constexpr int QBUF = 8192;        // Q^T of one item: up to 4 columns x 16 heads x 128 B
constexpr int QBYTES = 2 * QBUF;  // two Q^T buffers
constexpr int PBYTES = 16384;     // P^T: 2 buffers x (hi, lo) x 128 keys x 16 heads x 2 B
constexpr int RING_OFF = CTRL + QBYTES + PBYTES;
constexpr uint32_t TMEM_COLS = 128;

// TMEM columns: S^T of tile parity sb, O^T half `half` of item parity ob.
__device__ __forceinline__ uint32_t s_col(int sb) { return sb * 16; }
__device__ __forceinline__ uint32_t o_col(int ob, int half) { return 32 + ob * 32 + half * 16; }

struct Flags {
    volatile int *abort;
};

// Bounded wait on an mbarrier phase; false (and the CTA's pipeline aborted)
// if it ran past its limit or another role aborted.  SPIN: the roles on the
// per-tile critical path poll; the epilogue, which waits most of the time,
// sleeps between polls.
template <bool SPIN>
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, const Flags &f,
                                              unsigned int *err)
{
    if (*f.abort)
        return false;
    const bool ok = SPIN ? mbar_wait_spin(bar, parity, err) : mbar_wait(bar, parity, err);
    if (!ok) {
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

// OR of a predicate over the 128 threads of named barrier `id`.
template <int ID>
__device__ __forceinline__ bool group_any(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(ID)
        : "memory");
    return r != 0;
}

// AND of a predicate over the 128 threads of named barrier `id`.
template <int ID>
__device__ __forceinline__ bool group_all(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "n"(ID)
        : "memory");
    return r != 0;
}

constexpr int BAR_SOFTMAX = 1;  // named barrier of warps 0-3
constexpr int BAR_EPI = 2;      // named barrier of warps 4-7

template <int ID>
__device__ __forceinline__ void group_sync()
{
    asm volatile("bar.sync %0, 128;" ::"n"(ID) : "memory");
}

// Sums over the 32 lanes of N values (N = 2..16) by halving exchanges: a
// lane keeps one half of its values and sends the other, so the whole
// reduction takes N - 1 + 5 - log2(N) shuffles instead of 5N.  Returns the
// full sum of value `head`, a function of the lane: lanes that differ only
// in their low 5 - log2(N) bits hold the same head.
template <int N>
__device__ __forceinline__ float warp_sum_scatter(const float (&in)[N], int lane, int &head)
{
    static_assert(N == 2 || N == 4 || N == 8 || N == 16, "N");
    constexpr int STEPS = N == 2 ? 1 : N == 4 ? 2 : N == 8 ? 3 : 4;
    float v[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        v[i] = in[i];
    head = 0;
#pragma unroll
    for (int k = 0; k < STEPS; ++k) {
        const int o = 16 >> k;
        const bool up = (lane & o) != 0;
        const int half = N >> (k + 1);
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL_MASK, send, o);
        }
        head = (head << 1) | (up ? 1 : 0);
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 >> STEPS; o > 0; o >>= 1)
        r += __shfl_xor_sync(FULL_MASK, r, o);
    return r;
}


// Virtual tiles charged per item for its fixed cost on the CTA's pipeline
// (the first tile's loads of the next item start behind the item's last
// ones; the result is written by the epilogue warps, off that path).
constexpr int KAPPA = 1;

// One (sequence, kv head, split) item and its key range.
struct Item {
    int b, g, s;   // position in (sequence, kv head, split) order
    int start;     // global index of its first tile
    int pos, lo;   // attended keys [lo, pos]
    int ub0, ub1;  // paged blocks [ub0, ub1) of this split
    int n, T;      // blocks and 128-key tiles
    int nsplit;    // splits of the sequence
};

// Key range of an item (the same arithmetic as the CUDA-core kernel's
// key_range; lengths past the block table are clipped there and reported by
// the plan kernel).
__device__ __forceinline__ void item_geom(const DecodeParams &p, Item &it)
{
    int len = p.seq_lens[it.b];
    const int cap = p.max_blocks * kBlock;
    if (p.ring_blocks == 0)  // a ring does not bound the length
        len = len > cap ? cap : len;
    it.pos = len - 1;
    it.lo = p.window > 0 ? max(0, it.pos - p.window) : 0;
    const int blk_lo = len > 0 ? it.lo / kBlock : 0;
    const int nblk = len > 0 ? it.pos / kBlock - blk_lo + 1 : 0;
    it.nsplit =
        (p.split_blocks > 0 && nblk > 0) ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    it.ub0 = blk_lo + it.s * p.split_blocks;
    it.ub1 = p.split_blocks > 0 ? min(it.ub0 + p.split_blocks, blk_lo + nblk) : blk_lo + nblk;
    it.n = max(0, it.ub1 - it.ub0);
    it.T = (it.n + 7) / 8;
}

__device__ __forceinline__ Item item_at(const DecodeParams &p, int4 e)
{
    Item it;
    it.b = e.x;
    it.g = e.y;
    it.s = e.z;
    it.start = e.w;
    it.T = 0;
    it.nsplit = 1;
    if (it.b < p.batch)
        item_geom(p, it);
    return it;
}

__device__ __forceinline__ void item_next(const DecodeParams &p, Item &it)
{
    it.start += it.T + KAPPA;
    if (++it.s >= it.nsplit) {
        it.s = 0;
        if (++it.g >= p.num_kv_heads) {
            it.g = 0;
            ++it.b;
        }
    }
    it.T = 0;
    it.nsplit = 1;
    if (it.b < p.batch)
        item_geom(p, it);
}

// CTA c's share of the W tiles.
__device__ __forceinline__ int tile_bound(int c, int W, int C)
{
    return static_cast<int>(static_cast<int64_t>(c) * W / C);
}


}  // namespace

// Units of sequence b in the stream-K walk: its tiles (whole splits of F
// tiles and a remainder, or one range) plus KAPPA per item, for every kv head.
__device__ __forceinline__ int seq_units(const DecodeParams &p, int b, int F)
{
    int len = p.seq_lens[b];
    const int cap = p.max_blocks * kBlock;
    if (p.ring_blocks == 0 && len > cap)
        len = cap;
    int tiles = 0, ns = 1;
    if (len > 0) {
        const int sb = p.split_blocks;
        const int pos = len - 1;
        const int lo = p.window > 0 ? max(0, pos - p.window) : 0;
        const int nblk = pos / kBlock - lo / kBlock + 1;
        if (sb > 0) {
            const int whole = nblk / sb, rem = nblk - whole * sb;
            tiles = whole * F + (rem + 7) / 8;
            ns = whole + (rem > 0 ? 1 : 0);
        } else {
            tiles = (nblk + 7) / 8;
        }
    }
    return (tiles + KAPPA * ns) * p.num_kv_heads;
}

// The item a CTA whose units start at x processes first: the first item
// whose real tiles reach into [x, ...), or an empty item starting there.
// soff = the sequences' first units (prefix sums, soff[batch] = W).
__device__ __forceinline__ int4 first_item_at(const DecodeParams &p, const int *soff, int x, int F)
{
    const int H = p.num_kv_heads, sb = p.split_blocks;
    // the sequence whose units hold x, then the item whose units hold it
    int lo_b = 0, hi_b = p.batch;
    while (lo_b < hi_b) {
        const int mid = (lo_b + hi_b) >> 1;
        if (soff[mid + 1] > x)
            hi_b = mid;
        else
            lo_b = mid + 1;
    }
    Item it;
    it.b = lo_b;
    it.g = 0;
    it.s = 0;
    it.start = soff[lo_b];
    item_geom(p, it);
    const int Eg = (soff[lo_b + 1] - it.start) / H;  // units per kv head
    const int rel = x - it.start;
    if (rel > 0) {
        it.g = rel / Eg;
        const int r2 = rel - it.g * Eg;
        it.s = sb > 0 ? min(r2 / (F + KAPPA), it.nsplit - 1) : 0;
        it.start += it.g * Eg + it.s * (F + KAPPA);
        item_geom(p, it);
        // x in this item's virtual tail: the CTA starts with the next item
        if (it.start + it.T <= x && !(it.T == 0 && it.start >= x))
            item_next(p, it);
    }
    return make_int4(it.b, it.g, it.s, it.start);
}

// ------------------------------------------------------------------ plan
// One CTA: units per sequence (tiles + KAPPA per item, all kv heads and
// splits), their prefix sums (workspace), and for each of the C CTAs the
// first item it processes: the first item whose real tiles reach into its
// units, or an empty item starting in them.  plan[0] = {W, C}; plan[1 + c] =
// {b, g, s, first unit of that item}; plan[1 + C] = {batch, 0, 0, W}.
constexpr int PLAN_SMEM_SEQS = 8192;  // prefix sums kept in shared memory up to this batch
constexpr int SELF_PLAN_SEQS = 8192;  // batches up to this size: each CTA plans its own walk

__global__ void __launch_bounds__(1024) tc_plan_kernel(const DecodeParams p, int grid)
{
    __shared__ int wsum[32];
    __shared__ int carry_s;
    __shared__ int soff_s[PLAN_SMEM_SEQS + 1];
    const bool in_smem = p.batch <= PLAN_SMEM_SEQS;
    int *soff = in_smem ? soff_s : p.tc_seqoff;
    pdl_launch_dependents();  // the decode kernel's prologue may start now
    for (int i = threadIdx.x; i < 2 * kTcMaxGrid; i += 1024)
        p.tc_flags[i] = 0;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int sb = p.split_blocks;
    const int F = sb > 0 ? (sb + 7) / 8 : 0;  // tiles of a whole split
    if (tid == 0)
        carry_s = 0;
    __syncthreads();
    for (int base = 0; base < p.batch; base += 1024) {
        const int b = base + tid;
        int v = 0;
        if (b < p.batch) {
            const int len = p.seq_lens[b];
            if (p.ring_blocks == 0 && len > p.max_blocks * kBlock)
                record_error(p.err, PKV_DEV_LEN_TABLE);
            if (len > p.max_seq_len)
                record_error(p.err, PKV_DEV_LEN_BOUND);
            v = seq_units(p, b, F);
        }
        int x = v;
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
        const int incl = x + (wid > 0 ? wsum[wid - 1] : 0);
        const int carry = carry_s;
        if (b < p.batch)
            soff[b] = carry + incl - v;
        __syncthreads();
        if (tid == 1023)
            carry_s = carry + incl;
        __syncthreads();
    }
    const int W = carry_s;  // >= KAPPA: every sequence has an item per kv head
    if (tid == 0)
        soff[p.batch] = W;
    __syncthreads();
    const int C = min(grid, W);
    if (tid == 0)
        p.tc_plan[0] = make_int4(W, C, 0, 0);
    for (int c = tid; c <= C; c += 1024) {
        int4 e;
        if (c == C) {
            e = make_int4(p.batch, 0, 0, W);
        } else {
            e = first_item_at(p, soff, tile_bound(c, W, C), F);
        }
        p.tc_plan[1 + c] = e;
    }
}


// ------------------------------------------------------------------ epilogue
// Partial-state row of part k of a cut item: the CTA holding its first tile
// (ca) has it as its last item (slot 1), the CTAs after it as their first
// item (slot 0).
__device__ __forceinline__ size_t part_row(int ca, int k)
{
    return (static_cast<size_t>(ca + k) * 2 + (k == 0 ? 1 : 0)) * NPAD;
}

// Merge of a cut item's parts by the epilogue warpgroup of the CTA whose
// part finished last: per head the weights exp(lse_k - max) / sum over the
// parts, then the weighted sum of the normalised partial outputs, written
// as the output row (one split) or as the split's partial state.  Thread t
// owns head t / 8 and every eighth 16-byte column of it; the parts'
// log-sum-exps are reduced by the 8 threads of a head.
template <int D>
__device__ __forceinline__ void merge_parts(const DecodeParams &p, const Item &it, int ca,
                                         int nparts, int t)
{
    constexpr int NV = D / 32;  // 16-byte columns per thread
    const int G = p.group;
    const int hh = t >> 3, grp = t & 7;
    float M = -INFINITY, Z = 0.f;
    if (hh < G) {
        for (int k = grp; k < nparts; k += 8) {
            const float l = __ldcg(&p.sub_lse[part_row(ca, k) + hh]);
            if (l == -INFINITY)
                continue;
            if (l > M) {
                Z = Z * expf(M - l) + 1.f;
                M = l;
            } else {
                Z += expf(l - M);
            }
        }
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
        const float M2 = __shfl_xor_sync(FULL_MASK, M, off);
        const float Z2 = __shfl_xor_sync(FULL_MASK, Z, off);
        const float Mn = fmaxf(M, M2);
        Z = Mn == -INFINITY ? 0.f
                            : (M == -INFINITY ? 0.f : Z * expf(M - Mn)) +
                                  (M2 == -INFINITY ? 0.f : Z2 * expf(M2 - Mn));
        M = Mn;
    }
    if (hh >= G)
        return;
    const float invZ = Z > 0.f ? 1.f / Z : 0.f;
    float4 acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i)
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    // one part per step: NV independent 16-byte loads in flight per thread
    for (int k = 0; k < nparts; ++k) {
        const size_t r = part_row(ca, k) + hh;
        const float l = __ldcg(&p.sub_lse[r]);
        const float4 *src = reinterpret_cast<const float4 *>(p.sub_o + r * D);
        float4 v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i)
            v[i] = __ldcg(src + grp + 8 * i);
        const float w = (l == -INFINITY || M == -INFINITY) ? 0.f : expf(l - M) * invZ;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            acc[i].x = fmaf(w, v[i].x, acc[i].x);
            acc[i].y = fmaf(w, v[i].y, acc[i].y);
            acc[i].z = fmaf(w, v[i].z, acc[i].z);
            acc[i].w = fmaf(w, v[i].w, acc[i].w);
        }
    }
    if (it.nsplit == 1) {
        const size_t o = (static_cast<size_t>(it.b) * p.num_q_heads + it.g * G + hh) * D;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int d = (grp + 8 * i) * 4;
            if (p.out_f32) {
                *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + o + d) = acc[i];
            } else {
                __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc[i].x, acc[i].y);
                __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc[i].z, acc[i].w);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t *>(&lo2);
                u.y = *reinterpret_cast<uint32_t *>(&hi2);
                *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + o + d) = u;
            }
        }
    } else {
        const size_t prow =
            (static_cast<size_t>(it.b) * p.num_splits + it.s) * p.num_q_heads + it.g * G + hh;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            *reinterpret_cast<float4 *>(&p.part_o[prow * D + (grp + 8 * i) * 4]) = acc[i];
        if (grp == 0)
            p.part_lse[prow] = Z > 0.f ? M + logf(Z) : -INFINITY;
    }
}

// ------------------------------------------------------------------ decode
template <int D, int GP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmq)
{
    constexpr int HALVES = D / 128;
    constexpr uint32_t QB = NPAD * D * 2;  // Q^T bytes of one item
    static_assert(D == 128 || D == 256, "head_dim");
    static_assert(GP == 2 || GP == 4 || GP == 8 || GP == 16, "padded group");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t *unit_full = reinterpret_cast<uint64_t *>(sm);  // [8]
    uint64_t *unit_empty = unit_full + 8;                    // [8]
    uint64_t *s_full = unit_full + 16;                       // [2] S^T of a tile in TMEM
    uint64_t *s_empty = s_full + 2;                          // [2] S^T read by the softmax
    uint64_t *p_full = s_full + 4;                           // [2] P^T of a tile written
    uint64_t *pv_done = s_full + 6;                          // [2] a tile's P.V complete
    uint64_t *o_full = s_full + 8;                           // [2] an item's O^T complete
    uint64_t *o_free = s_full + 10;                          // [2] an item's O^T read
    uint64_t *q_full = s_full + 12;                          // [2]
    uint64_t *q_empty = s_full + 14;                         // [2]
    uint64_t *epi_full = s_full + 16;                        // [2] an item's max and sums
    uint64_t *epi_empty = s_full + 18;                       // [2] ... read by the epilogue
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + 288);
    Flags flags{reinterpret_cast<volatile int *>(sm + 292)};
    volatile int *ticket_s = reinterpret_cast<volatile int *>(sm + 296);
    float *red = reinterpret_cast<float *>(sm + 320);        // [4][16] softmax exchange
    // running max per head and the last rescale factors: the same in every
    // softmax thread, so kept once in shared memory instead of in registers
    float *mrun_s = reinterpret_cast<float *>(sm + 576);     // [16]
    float *alpha_s = reinterpret_cast<float *>(sm + 640);    // [16]
    float *epi_m = reinterpret_cast<float *>(sm + 704);      // [2][16] an item's max (log2)
    float *epi_l = reinterpret_cast<float *>(sm + 832);      // [2][16] an item's sums
    uint8_t *qs = sm + CTRL;
    uint8_t *ps = sm + CTRL + QBYTES;
    uint8_t *units = sm + RING_OFF;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const bool alias = p.alias != 0;
    const int NU = p.num_stages;
    const bool precise = p.out_f32 != 0;  // P as bf16 hi + lo: two P.V passes

    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; ++i) {
            mbar_init(&unit_full[i], 1);
            mbar_init(&unit_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], SOFTMAX_WARPS);
            mbar_init(&p_full[i], SOFTMAX_WARPS);
            mbar_init(&pv_done[i], 1);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_free[i], 4);
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&epi_full[i], 1);
            mbar_init(&epi_empty[i], 4);
        }
        *flags.abort = 0;
        fence_barrier_init();
    }
    if (warp == MMA_WARP)
        tmem_alloc(tmem_slot, TMEM_COLS);
    if (warp < SOFTMAX_WARPS) {
        // P^T buffers start at zero: padded heads stay zero for the whole kernel
        for (int idx = threadIdx.x; idx < PBYTES / 16; idx += 128)
            reinterpret_cast<uint4 *>(ps)[idx] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The walk: up to SELF_PLAN_SEQS sequences each CTA lays out its own
    // share (the same arithmetic as tc_plan_kernel, the prefix sums in the
    // ring, which no load uses yet), so it starts streaming without waiting
    // for the plan kernel, which then only clears the tickets (awaited before
    // the first ticket is taken).  Larger batches read the plan kernel's.
    const int c = blockIdx.x;
    int W, C;
    int4 first;
    if (p.batch <= SELF_PLAN_SEQS) {
        int *soff = reinterpret_cast<int *>(units);
        int *wsum = reinterpret_cast<int *>(sm + 960);                  // [16]
        volatile int *carry_s = reinterpret_cast<volatile int *>(sm + 300);
        int4 *res = reinterpret_cast<int4 *>(units + 4 * (SELF_PLAN_SEQS + 4));
        const int tid = threadIdx.x;
        const int F = p.split_blocks > 0 ? (p.split_blocks + 7) / 8 : 0;
        if (tid == 0)
            *carry_s = 0;
        __syncthreads();
        for (int base = 0; base < p.batch; base += TC_THREADS) {
            const int b = base + tid;
            const int v = b < p.batch ? seq_units(p, b, F) : 0;
            int x = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(FULL_MASK, x, off);
                if (lane >= off)
                    x += y;
            }
            if (lane == 31)
                wsum[warp] = x;
            __syncthreads();
            if (warp == 0) {
                int w = lane < TC_WARPS ? wsum[lane] : 0;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(FULL_MASK, w, off);
                    if (lane >= off)
                        w += y;
                }
                if (lane < TC_WARPS)
                    wsum[lane] = w;
            }
            __syncthreads();
            const int incl = x + (warp > 0 ? wsum[warp - 1] : 0);
            const int carry = *carry_s;
            if (b < p.batch)
                soff[b] = carry + incl - v;
            __syncthreads();
            if (tid == TC_THREADS - 1)
                *carry_s = carry + incl;
            __syncthreads();
        }
        if (tid == 0) {
            const int w = *carry_s;
            soff[p.batch] = w;
            const int cc = min(static_cast<int>(gridDim.x), w);
            res[0] = make_int4(w, cc, 0, 0);
            res[1] = c < cc ? first_item_at(p, soff, tile_bound(c, w, cc), F)
                            : make_int4(p.batch, 0, 0, 0);
        }
        __syncthreads();
        W = res[0].x;
        C = res[0].y;
        first = res[1];
        __syncthreads();  // the ring is the producers' from here
    } else {
        pdl_wait();  // the plan kernel has completed
        const int4 hdr = p.tc_plan[0];
        W = hdr.x;
        C = hdr.y;
        first = c < C ? p.tc_plan[1 + c] : make_int4(p.batch, 0, 0, 0);
    }
    pdl_launch_dependents();  // a dependent kernel may be scheduled as SMs free up
    const bool active = c < C;  // CTAs past C only release their TMEM
    const int t0 = active ? tile_bound(c, W, C) : 0, t1 = active ? tile_bound(c + 1, W, C) : 0;

    constexpr int GL = GP < 16 ? GP : 16;  // TMEM columns per S or O half
    // Unit j (a 128-dim half of a 128-key tile, counted over the CTA's whole
    // walk) of the K stream lives in slot j % NKU, use j / NKU; of the V
    // stream in slot VBASE + j % NVU, use j / NVU.
    const int NKU = alias ? NU : NU / 2;
    const int NVU = alias ? NU : NU - NKU;
    const int VBASE = alias ? 0 : NKU;

    if (warp >= PRODUCER_WARP && warp < MMA_WARP) {
        // ------------------------------------------------------ producers
        const int slot = warp - PRODUCER_WARP;  // the ring slot this warp owns
        const bool vwarp = !alias && slot >= NKU;
        const int ring = vwarp ? NVU : NKU, rbase = vwarp ? VBASE : 0;
        if (slot < NU) {
            const CUtensorMap *map = vwarp ? &tmv : &tmk;
            if (lane == 0) {
                prefetch_tensormap(map);
                if (slot == 0)
                    prefetch_tensormap(&tmq);
            }
            const uint64_t pol = policy_evict_first();
            int j = 0, kq = 0, last_use = -1, q_last = -1;
            bool stop = false;
            Item it = item_at(p, first);
            for (; !stop && it.b < p.batch && it.start < t1; item_next(p, it)) {
                const int lt0 = max(0, t0 - it.start), lt1 = min(it.T, t1 - it.start);
                if (lt1 <= lt0)
                    continue;
                if (slot == 0) {
                    // Q^T of this item: 16 rows (heads g*G ...) x D dims
                    const int qb = kq & 1;
                    const bool room =
                        kq < 2 || wait_or_abort<true>(&q_empty[qb], ((kq >> 1) - 1) & 1, flags, p.err);
                    if (!__all_sync(FULL_MASK, room))
                        break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&q_full[qb], QB);
#pragma unroll
                        for (int col = 0; col < D / 64; ++col)
                            tma_load_2d(qs + qb * QBUF + col * 2048, &tmq, col * 64,
                                        it.b * p.num_q_heads + it.g * G, &q_full[qb]);
                    }
                    q_last = kq;
                }
                ++kq;
                const int32_t *bt_row = p.block_table + static_cast<size_t>(it.b) * p.max_blocks;
                TableCursor tc;
                tc.init(bt_row, it.ub0 + lt0 * 8, it.n - lt0 * 8, p.ring_blocks, lane);
                for (int i = lt0; i < lt1 && !stop; ++i) {
                    int row[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int blk = i * 8 + t;
                        const int phys = blk < it.n ? tc.get(blk - lt0 * 8, lane) : -1;
                        const bool valid =
                            static_cast<unsigned>(phys) < static_cast<unsigned>(p.num_blocks);
                        if (blk < it.n && !valid && lane == 0 && slot == 0)
                            record_error(p.err, PKV_DEV_BAD_BLOCK);
                        // an out-of-range row: the TMA fills the box with zeros
                        row[t] = valid ? phys * kBlock : p.num_blocks * kBlock;
                    }
                    for (int h = 0; h < HALVES; ++h) {
                        const int jj = j++;
                        if (rbase + jj % ring != slot)
                            continue;
                        const int use = jj / ring;
                        const bool room = use == 0 || wait_or_abort<true>(&unit_empty[slot], (use - 1) & 1,
                                                                          flags, p.err);
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
                            const int t = lane >> 1, cc = lane & 1;
                            int rt = row[0];
#pragma unroll
                            for (int k = 1; k < 8; ++k)
                                rt = (t == k) ? row[k] : rt;
                            tma_load_3d(units + slot * UNIT + cc * CHUNK + t * 2048, map,
                                        h * 128 + cc * 64, it.g, rt, &unit_full[slot], pol);
                        }
                        last_use = use;
                    }
                    __syncwarp();
                }
            }
            // Drain: do not retire with this warp's copies in flight.
            if (lane == 0) {
                if (last_use >= 0)
                    mbar_wait(&unit_full[slot], last_use & 1, p.err, 100000000ull);
                if (q_last >= 0)
                    mbar_wait(&q_full[q_last & 1], (q_last >> 1) & 1, p.err, 100000000ull);
            }
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------ score MMAs
        // tile i needs its item's Q^T, its K units and a free S buffer
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = umma_idesc_bf16(128, NPAD, false, false);
            const uint32_t u_base = smem_u32(units);
            int i_g = 0, j = 0, kq = 0;
            bool ok = true;
            Item it = item_at(p, first);
            for (; ok && it.b < p.batch && it.start < t1; item_next(p, it)) {
                const int lt0 = max(0, t0 - it.start), lt1 = min(it.T, t1 - it.start);
                if (lt1 <= lt0)
                    continue;
                const int qb = kq & 1;
                ok = wait_or_abort<true>(&q_full[qb], (kq >> 1) & 1, flags, p.err);
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t q_base = smem_u32(qs + qb * QBUF);
                for (int i = lt0; i < lt1 && ok; ++i, ++i_g) {
                    const int sb = i_g & 1;
                    if (i_g >= 2 &&
                        !wait_or_abort<true>(&s_empty[sb], ((i_g >> 1) - 1) & 1, flags, p.err)) {
                        ok = false;
                        break;
                    }
                    for (int h = 0; h < HALVES; ++h, ++j) {
                        const int slot = j % NKU;
                        ok = wait_or_abort<true>(&unit_full[slot], (j / NKU) & 1, flags, p.err);
                        if (!ok)
                            break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = umma_smem_desc(
                                u_base + slot * UNIT + (kk >> 2) * CHUNK + (kk & 3) * 32, 16, 1024);
                            const int kqd = h * 8 + kk;
                            const uint64_t bd = umma_smem_desc(
                                q_base + (kqd >> 2) * 2048 + (kqd & 3) * 32, 16, 1024);
                            umma_bf16(tmem + s_col(sb), a, bd, IDESC_QK, (h | kk) != 0);
                        }
                        if (!alias)
                            umma_commit(&unit_empty[slot]);  // K unit free once read
                    }
                    if (ok)
                        umma_commit(&s_full[sb]);
                }
                if (ok)
                    umma_commit(&q_empty[qb]);  // Q^T buffer free once its MMAs are done
                ++kq;
            }
        }
        __syncwarp();
    } else if (warp == PV_WARP) {
        // ------------------------------------------------------ P.V MMAs
        // tile i needs P^T and its V units; an item's first tile also needs
        // its O buffer (free once the epilogue has read the item two back).
        // The whole warp first zeroes V rows of masked keys inside loaded
        // blocks (only the block holding the window start and the block
        // holding pos can have them), lane 0 then issues the MMAs, which
        // accumulate into the item's O^T from its second tile on.
        constexpr uint32_t IDESC_PV = umma_idesc_bf16(128, NPAD, true, true);
        const uint32_t p_base = smem_u32(ps), u_base = smem_u32(units);
        int i_g = 0, j = 0, k = 0;
        bool ok = true;
        Item it = item_at(p, first);
        for (; ok && it.b < p.batch && it.start < t1; item_next(p, it)) {
            const int lt0 = max(0, t0 - it.start), lt1 = min(it.T, t1 - it.start);
            if (lt1 <= lt0)
                continue;
            const int ob = k & 1;
            {
                const bool go =
                    k < 2 || wait_or_abort<true>(&o_free[ob], ((k >> 1) - 1) & 1, flags, p.err);
                if (!__all_sync(FULL_MASK, go)) {
                    ok = false;
                    break;
                }
            }
            const int lo_blk = it.lo / kBlock, pos_blk = it.pos / kBlock;
            for (int i = lt0; i < lt1 && ok; ++i, ++i_g) {
                const int sb = i_g & 1;
                const bool go = wait_or_abort<true>(&p_full[sb], (i_g >> 1) & 1, flags, p.err);
                if (!__all_sync(FULL_MASK, go)) {
                    ok = false;
                    break;
                }
                const int tb0 = it.ub0 + i * 8;  // first block of the tile
                const int key0 = tb0 * kBlock;
                // rows [z0a, z0b) before lo and [z1a, z1b) after pos, in this tile
                int z0a = 0, z0b = 0, z1a = 0, z1b = 0;
                if (lo_blk >= tb0 && lo_blk < tb0 + 8 && lo_blk < it.ub1 && it.lo > lo_blk * kBlock) {
                    z0a = lo_blk * kBlock - key0;
                    z0b = it.lo - key0;
                }
                if (pos_blk >= tb0 && pos_blk < tb0 + 8 && pos_blk < it.ub1 &&
                    it.pos < pos_blk * kBlock + kBlock - 1) {
                    z1a = it.pos + 1 - key0;
                    z1b = (pos_blk + 1) * kBlock - key0;
                }
                for (int h = 0; h < HALVES; ++h, ++j) {
                    const int slot = VBASE + j % NVU;
                    // A separate V stream is waited for here.  With K == V the
                    // score warp waited for the unit, and its MMAs on it came
                    // before S, P and p_full.  Each half is issued on its own:
                    // one burst of 16 P.V MMAs delays the next tile's score
                    // MMAs queued behind it in the tensor pipe.
                    if (!alias) {
                        ok = wait_or_abort<true>(&unit_full[slot], (j / NVU) & 1, flags, p.err);
                        if (!__all_sync(FULL_MASK, ok)) {
                            ok = false;
                            break;
                        }
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
                                // P^T: MN-major, one 32-byte row of 16 heads
                                // per key, 8-key groups 256 B apart
                                const uint64_t bd = umma_smem_desc_sw32(
                                    p_base + sb * 8192 + pass * 4096 + kk * 512, 4096, 256);
                                umma_bf16(tmem + o_col(ob, h), a, bd, IDESC_PV,
                                          i > lt0 || pass > 0 || kk > 0);
                            }
                        }
                        umma_commit(&unit_empty[slot]);  // V (or K = V) unit free once read
                    }
                    __syncwarp();
                }
                if (!ok)
                    break;
                if (lane == 0) {
                    umma_commit(&pv_done[sb]);  // P^T buffer sb free; O through this tile
                    if (i == lt1 - 1)
                        umma_commit(&o_full[ob]);  // the item's O^T is final
                }
                __syncwarp();
            }
            ++k;
        }
    } else if (warp < SOFTMAX_WARPS) {
        // ------------------------------------------------------ softmax
        const int t = threadIdx.x;  // key row of the tile == TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float qk = p.qk_scale_log2;
        float lpart[GP];
        int i_g = 0, k = 0;
        Item it = item_at(p, first);
        for (; it.b < p.batch && it.start < t1; item_next(p, it)) {
            const int lt0 = max(0, t0 - it.start), lt1 = min(it.T, t1 - it.start);
            if (lt1 <= lt0)
                continue;
            const int ob = k & 1;
#pragma unroll
            for (int h = 0; h < GP; ++h)
                lpart[h] = 0.f;
            for (int i = lt0; i < lt1; ++i, ++i_g) {
                const int sb = i_g & 1;
                const bool first_tile = i == lt0;
                // key t of the tile: inside the item's blocks and in [lo, pos].
                // A block id outside the pool is not read here: the producer
                // reports it and its box arrives as zeros (keys of score 0,
                // V rows 0), so only that sequence's output is affected; no
                // global load stands in the softmax's path.
                const bool loaded = i * 8 + (t >> 4) < it.n;
                const int jk = (it.ub0 + i * 8) * kBlock + t;
                const bool ok = loaded && jk >= it.lo && jk <= it.pos;
                // ---- scores
                bool live = wait_or_abort<true>(&s_full[sb], (i_g >> 1) & 1, flags, p.err);
                tc_fence_after();
                float s[GL];
                if (live)
                    ld_cols<GL>(lane_base + s_col(sb), s);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s_empty[sb]);
                float sc[GP];
                // the item's first tile always sets the running max
                bool big = first_tile;
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    sc[h] = (live && ok && h < G) ? s[h] * qk : -INFINITY;
                    big |= sc[h] > mrun_s[h] + 8.f;  // no stores in between: loads overlap
                }
                // ---- running max: changed only when some score exceeds it by
                // more than 2^8.  group_any is also the barrier after which
                // red / mrun_s / alpha_s may be rewritten.
                const bool rescale = group_any<BAR_SOFTMAX>(big);
                if (rescale) {
#pragma unroll
                    for (int h = 0; h < GP; ++h) {
                        float v = sc[h];
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1)
                            v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, off));
                        if (lane == 0)
                            red[warp * 16 + h] = v;
                    }
                    group_sync<BAR_SOFTMAX>();
                    if (t < GP) {
                        const float tm =
                            fmaxf(fmaxf(red[t], red[16 + t]), fmaxf(red[32 + t], red[48 + t]));
                        const float mo = first_tile ? -INFINITY : mrun_s[t];
                        const float mn = fmaxf(mo, tm);
                        alpha_s[t] = mn == -INFINITY ? 1.f : fast_exp2(mo - mn);
                        mrun_s[t] = mn;
                    }
                    group_sync<BAR_SOFTMAX>();  // red is reused
                }
                // ---- P^T buffer sb was last read by the P.V of tile i_g - 2
                if (i_g >= 2)
                    live &= wait_or_abort<true>(&pv_done[sb], ((i_g >> 1) - 1) & 1, flags, p.err);
                if (rescale && !first_tile) {
                    // O^T through the previous tile is relative to the old max:
                    // scale it once that tile's P.V is done, before this P is
                    // published (the P.V warp waits for it)
                    live &= wait_or_abort<true>(&pv_done[sb ^ 1], ((i_g - 1) >> 1) & 1, flags, p.err);
                    tc_fence_after();
                    if (live) {
#pragma unroll
                        for (int hv = 0; hv < HALVES; ++hv) {
                            constexpr int NC = GL < 8 ? GL : 8;  // columns per TMEM access
#pragma unroll
                            for (int c0 = 0; c0 < GL; c0 += NC) {
                                float o[NC];
                                ld_cols<NC>(lane_base + o_col(ob, hv) + c0, o);
#pragma unroll
                                for (int h = 0; h < NC; ++h)
                                    o[h] *= alpha_s[c0 + h];
                                tmem_st<NC>(lane_base + o_col(ob, hv) + c0, o);
                            }
                        }
                    }
                    tc_fence_before();
                }
                // ---- probabilities, running sums, P^T (bf16, K-major, swizzled).
                // The maxima and rescale factors are read into registers
                // first: read inside the loop, behind its shared-memory
                // stores, every head would wait for its own load.
                float mr[GP], al[GP];
#pragma unroll
                for (int h4 = 0; h4 < GP; h4 += (GP >= 4 ? 4 : GP)) {
                    if constexpr (GP >= 4) {
                        const float4 m4 = *reinterpret_cast<const float4 *>(mrun_s + h4);
                        const float4 a4 = *reinterpret_cast<const float4 *>(alpha_s + h4);
                        mr[h4] = m4.x; mr[h4 + 1] = m4.y; mr[h4 + 2] = m4.z; mr[h4 + 3] = m4.w;
                        al[h4] = a4.x; al[h4 + 1] = a4.y; al[h4 + 2] = a4.z; al[h4 + 3] = a4.w;
                    } else {
                        const float2 m2 = *reinterpret_cast<const float2 *>(mrun_s + h4);
                        const float2 a2 = *reinterpret_cast<const float2 *>(alpha_s + h4);
                        mr[h4] = m2.x; mr[h4 + 1] = m2.y;
                        al[h4] = a2.x; al[h4 + 1] = a2.y;
                    }
                }
                // P^T is MN-major with the 32-byte swizzle: key t's 16 heads
                // are one 32-byte row (8-key groups of 256 B), its two 16-byte
                // halves swapped in rows 4-7 of a group; the thread writes
                // its row with one or two vector stores
                uint8_t *pb = ps + sb * 8192 + (t >> 3) * 256 + (t & 7) * 32;
                const int sw = (t >> 2) & 1;
                uint32_t whi[GP / 2], wlo[GP / 2];
#pragma unroll
                for (int h = 0; h < GP; h += 2) {
                    float pr2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        pr2[e] = sc[h + e] == -INFINITY ? 0.f : fast_exp2(sc[h + e] - mr[h + e]);
                        lpart[h + e] = rescale ? fmaf(lpart[h + e], al[h + e], pr2[e])
                                               : lpart[h + e] + pr2[e];
                    }
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(pr2[0], pr2[1]);
                    whi[h / 2] = *reinterpret_cast<const uint32_t *>(&hi);
                    if (precise) {
                        const float2 hf = __bfloat1622float2(hi);
                        const __nv_bfloat162 lo =
                            __floats2bfloat162_rn(pr2[0] - hf.x, pr2[1] - hf.y);
                        wlo[h / 2] = *reinterpret_cast<const uint32_t *>(&lo);
                    }
                }
                auto put_row = [&](uint8_t *row, const uint32_t(&w)[GP / 2]) {
                    if constexpr (GP >= 8) {
#pragma unroll
                        for (int c = 0; c < GP / 8; ++c)
                            *reinterpret_cast<uint4 *>(row + ((c ^ sw) << 4)) =
                                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    } else if constexpr (GP == 4) {
                        *reinterpret_cast<uint2 *>(row + (sw << 4)) = make_uint2(w[0], w[1]);
                    } else {
                        *reinterpret_cast<uint32_t *>(row + (sw << 4)) = w[0];
                    }
                };
                put_row(pb, whi);
                if (precise)
                    put_row(pb + 4096, wlo);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[sb]);
            }
            // ---- the item's sums over its keys and its max go to the
            // epilogue (slot ob, free once the epilogue has read item k - 2)
            {
                int hh;
                const float v = warp_sum_scatter<GP>(lpart, lane, hh);
                if ((lane & (32 / GP - 1)) == 0)
                    red[warp * 16 + hh] = v;
            }
            group_sync<BAR_SOFTMAX>();
            if (warp == 0) {
                if (t < GP) {
                    if (k >= 2)
                        wait_or_abort<true>(&epi_empty[ob], ((k >> 1) - 1) & 1, flags, p.err);
                    epi_l[ob * 16 + t] = (red[t] + red[16 + t]) + (red[32 + t] + red[48 + t]);
                    epi_m[ob * 16 + t] = mrun_s[t];
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&epi_full[ob]);
            }
            ++k;
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int t = threadIdx.x - EPI_WARP * 32;  // output dims t, 128 + t == TMEM lane t
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        int k = 0;
        Item it = item_at(p, first);
        for (; it.b < p.batch && it.start < t1; item_next(p, it)) {
            const int lt0 = max(0, t0 - it.start), lt1 = min(it.T, t1 - it.start);
            if (it.T == 0) {
                // no keys (length 0): a zero output row, written by the CTA
                // whose units hold the item's start
                if (it.start >= t0) {
                    const size_t row0 = static_cast<size_t>(it.b) * p.num_q_heads + it.g * G;
                    for (int idx = t; idx < G * D; idx += 128) {
                        if (p.out_f32)
                            reinterpret_cast<float *>(p.out)[row0 * D + idx] = 0.f;
                        else
                            reinterpret_cast<__nv_bfloat16 *>(p.out)[row0 * D + idx] =
                                __float2bfloat16_rn(0.f);
                    }
                }
                continue;
            }
            if (lt1 <= lt0)
                continue;
            const int ob = k & 1;
            bool live = wait_or_abort<false>(&epi_full[ob], (k >> 1) & 1, flags, p.err);
            live = live && wait_or_abort<false>(&o_full[ob], (k >> 1) & 1, flags, p.err);
            tc_fence_after();
            float o[HALVES][GL];
            if (live) {
#pragma unroll
                for (int hv = 0; hv < HALVES; ++hv)
                    ld_cols<GL>(lane_base + o_col(ob, hv), o[hv]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&o_free[ob]);  // O^T is in registers now
            ++k;
            if (!group_all<BAR_EPI>(live))
                break;  // uniform over the warpgroup
            // 1 / L of head h and its log-sum-exp (natural log), from the
            // slot the softmax filled; the slot is released after the stores
            const float *Ls = epi_l + ob * 16, *Ms = epi_m + ob * 16;
            auto inv_of = [&](int h) {
                const float L = Ls[h];
                return L > 0.f ? 1.f / L : 0.f;
            };
            auto release_slot = [&]() {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&epi_empty[ob]);
            };
            const bool whole = lt0 == 0 && lt1 == it.T;
            const bool single = whole && it.nsplit == 1;
            if (single) {
                const size_t row0 = static_cast<size_t>(it.b) * p.num_q_heads + it.g * G;
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    if (h >= G)
                        continue;
                    const float inv = inv_of(h);
#pragma unroll
                    for (int hv = 0; hv < HALVES; ++hv) {
                        const size_t e = (row0 + h) * D + hv * 128 + t;
                        const float y = o[hv][h] * inv;
                        if (p.out_f32)
                            reinterpret_cast<float *>(p.out)[e] = y;
                        else
                            reinterpret_cast<__nv_bfloat16 *>(p.out)[e] = __float2bfloat16_rn(y);
                    }
                }
                release_slot();
                continue;
            }
            // a split's partial state (whole split) or this CTA's part of a cut item
            const int slot = lt0 > 0 ? 0 : 1;
            const size_t prow = whole ? (static_cast<size_t>(it.b) * p.num_splits + it.s) *
                                                p.num_q_heads + it.g * G
                                      : (static_cast<size_t>(c) * 2 + slot) * NPAD;
            float *dst_o = whole ? p.part_o : p.sub_o;
            float *dst_l = whole ? p.part_lse : p.sub_lse;
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                if (h >= G)
                    continue;
                const float inv = inv_of(h);
#pragma unroll
                for (int hv = 0; hv < HALVES; ++hv)
                    dst_o[(prow + h) * D + hv * 128 + t] = o[hv][h] * inv;
            }
            if (t < G) {
                const float L = Ls[t];
                dst_l[prow + t] = L > 0.f ? (Ms[t] + log2f(L)) * LN2 : -INFINITY;
            }
            release_slot();
            if (whole)
                continue;
            // cut item: publish this part, take a ticket; the last part merges
            int ca = c, cz = c;
            while (ca > 0 && tile_bound(ca, W, C) > it.start)
                --ca;
            const int u_last = it.start + it.T - 1;
            while (cz + 1 < C && tile_bound(cz + 1, W, C) <= u_last)
                ++cz;
            const int nparts = cz - ca + 1;
            __threadfence();
            group_sync<BAR_EPI>();
            if (t == 0) {
                pdl_wait();  // the plan kernel has cleared the tickets
                *ticket_s = atomicAdd(&p.tc_flags[ca], 1) == nparts - 1;
            }
            group_sync<BAR_EPI>();
            const bool last = *ticket_s != 0;
            if (last) {
                __threadfence();
                merge_parts<D>(p, it, ca, nparts, t);
            }
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

size_t decode_tc_scratch_bytes(int batch, int head_dim)
{
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    return up(sizeof(int4) * (2 + kTcMaxGrid)) + up(sizeof(int) * 2 * kTcMaxGrid) +
           up(sizeof(int) * (static_cast<size_t>(batch) + 1)) +
           up(sizeof(float) * kTcMaxGrid * 2 * NPAD) +
           sizeof(float) * kTcMaxGrid * 2 * NPAD * static_cast<size_t>(head_dim);
}

void decode_tc_bind_scratch(DecodeParams &p, void *scratch, int batch)
{
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    char *s = static_cast<char *>(scratch);
    p.tc_plan = reinterpret_cast<int4 *>(s);
    s += up(sizeof(int4) * (2 + kTcMaxGrid));
    p.tc_flags = reinterpret_cast<int *>(s);
    s += up(sizeof(int) * 2 * kTcMaxGrid);
    p.tc_seqoff = reinterpret_cast<int *>(s);
    s += up(sizeof(int) * (static_cast<size_t>(batch) + 1));
    p.sub_lse = reinterpret_cast<float *>(s);
    s += up(sizeof(float) * kTcMaxGrid * 2 * NPAD);
    p.sub_o = reinterpret_cast<float *>(s);
}

int decode_tc_grid()
{
    static std::atomic<int> cached{0};
    int v = cached.load(std::memory_order_relaxed);
    if (v)
        return v;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 1;
    v = sms < kTcMaxGrid ? sms : kTcMaxGrid;
    cached.store(v, std::memory_order_relaxed);
    return v;
}

template <int D, int GP>
static cudaError_t launch_tc_one(const DecodeParams &p, const CUtensorMap &tmk,
                                 const CUtensorMap &tmv, const CUtensorMap &tmq, int grid,
                                 cudaStream_t s)
{
    const size_t smem = decode_tc_smem_bytes(p.num_stages);
    auto kern = decode_tc_kernel<D, GP>;
    static std::atomic<int> configured{0};
    if (static_cast<int>(smem) > configured.load(std::memory_order_relaxed)) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured.store(static_cast<int>(smem), std::memory_order_relaxed);
    }
    // no CTA waits for another (cut items merge by ticket), so the launch
    // needs no co-residency guarantee
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv, tmq);
}

template <int D>
static cudaError_t launch_tc_d(const DecodeParams &p, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, const CUtensorMap &tmq, int gp, int grid,
                               cudaStream_t s)
{
    switch (gp) {
    case 2: return launch_tc_one<D, 2>(p, tmk, tmv, tmq, grid, s);
    case 4: return launch_tc_one<D, 4>(p, tmk, tmv, tmq, grid, s);
    case 8: return launch_tc_one<D, 8>(p, tmk, tmv, tmq, grid, s);
    case 16: return launch_tc_one<D, 16>(p, tmk, tmv, tmq, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_tc(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                             const CUtensorMap &tmq, int head_dim, cudaStream_t s)
{
    const int gp = decode_tc_group_pad(p.group);
    const int grid = decode_tc_grid();
    tc_plan_kernel<<<1, 1024, 0, s>>>(p, grid);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    if (head_dim == 128)
        e = launch_tc_d<128>(p, tmk, tmv, tmq, gp, grid, s);
    else if (head_dim == 256)
        e = launch_tc_d<256>(p, tmk, tmv, tmq, gp, grid, s);
    else
        e = cudaErrorInvalidValue;
    return e;
}

}  // namespace pkv

