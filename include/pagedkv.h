/*
 * pagedkv.h -- C ABI of libpagedkv.so: single-token decode attention over a
 * paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The problem (sources by page title and section):
 *  - "CS336 · 第 10 课" (inference lecture guide), KV-cache section: at each
 *    decode step the new token's K/V are appended to the cache and its query
 *    attends over every cached key, a = softmax(q K^T / sqrt(d_h)), y = a V.
 *  - "推理优化与 AI Infra" (tiniestgpt notes), section 2: the cache is a pool
 *    of physical blocks k_cache[block][slot][head][dim] reached through
 *    block_table[seq][i]; section 5: int8 KV with per_token or per_head
 *    scales, dequantised after the gather; section 8: static step buffers
 *    (block_table, seq_lens, slot ids) and a host-side integer bound on the
 *    KV length so that no device value is read on the host.
 *  - "实验五：Gemma4 端到端推理优化" (Lab5-Gemma4): sections 滑动窗口注意力
 *    (window [i-w, i]), 分组查询注意力 (query heads share KV heads), the
 *    model overview (W_K = W_V on global layers: K and V one tensor), and
 *    Flash Attention (online softmax with running max/sum, blocks outside
 *    the window skipped, a separate narrow-query decode kernel).
 *
 * Conventions for every call:
 *  - All pointers are DEVICE pointers unless stated; the caller allocates and
 *    owns every buffer.  The library allocates no device memory and keeps no
 *    state except a thread-local error string, an error word in device
 *    memory (pkv_device_status), per-device launch attributes and the fixed
 *    scratch array of paged_decode_attention_noalloc.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  No call synchronises or reads device data on
 *    the host, so the calls may be captured in a CUDA graph.
 *  - Return value: 0 (PKV_OK) on success; a negative PKV_E_* code when an
 *    argument is rejected on the host (nothing is launched; the message is in
 *    pkv_last_error()); a positive cudaError_t when a launch fails.
 *  - Errors the host cannot see (a block id outside the pool, a length
 *    beyond the block table or beyond max_seq_len, a slot outside the pool)
 *    are detected in the kernels and set a bit in the device error word,
 *    read with pkv_device_status() after the stream has been synchronised.
 *    Nothing outside the pool or the block table is read or written: keys
 *    past the block table and tokens with a slot outside the pool are
 *    skipped; a block id outside the pool is never dereferenced (the
 *    CUDA-core kernel skips its keys, the tensor-core kernel reads them as
 *    zero vectors), so the output of a sequence that names one is
 *    unspecified.  Other sequences are unaffected.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

/* element type of the pool */
#define PKV_BF16 0
#define PKV_INT8 1
/* int8 scale granularity (tiniestgpt notes, section 5: per_token / per_head) */
#define PKV_SCALE_NONE 0
#define PKV_SCALE_PER_TOKEN 1
#define PKV_SCALE_PER_HEAD 2
/* output element type */
#define PKV_OUT_BF16 0
#define PKV_OUT_F32 1
/* split_tokens value asking the library to choose the split length */
#define PKV_SPLIT_AUTO (-1)

/* host-side status codes */
#define PKV_OK 0
#define PKV_E_NULL (-1)        /* a required pointer is NULL */
#define PKV_E_SHAPE (-2)       /* inconsistent sizes (e.g. H_q % H_kv != 0) */
#define PKV_E_UNSUPPORTED (-3) /* head_dim / block_size / dtype not built */
#define PKV_E_WORKSPACE (-4)   /* workspace missing or too small */
#define PKV_E_ALIGN (-5)       /* a pointer violates its alignment rule */
#define PKV_E_ARG (-6)         /* any other invalid argument */
#define PKV_E_DRIVER (-7)      /* tensor-map encoding / device query failed */

/* device error word bits (pkv_device_status) */
#define PKV_DEV_BAD_BLOCK 1u    /* block_table entry outside [0, num_blocks) */
#define PKV_DEV_LEN_TABLE 2u    /* seq_len > max_blocks_per_seq * block_size */
#define PKV_DEV_BAD_SLOT 4u     /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEV_TIMEOUT 8u      /* a pipeline wait ran past its limit */
#define PKV_DEV_LEN_BOUND 16u   /* seq_len > max_seq_len given on the host */
#define PKV_DEV_BAD_POSITION 32u /* a RoPE position >= num_positions of its table */

/* Pairing of dims in a rotary embedding (paged_kv_append_rope). */
#define PKV_ROPE_HALVES 0      /* pair i = dims (i, i + head_dim / 2) */
#define PKV_ROPE_INTERLEAVED 1 /* pair i = dims (2i, 2i + 1) */

/*
 * One layer's KV pool (tiniestgpt notes, section 2; one pool per layer).
 *   k, v:  [num_blocks][block_size][num_kv_heads][head_dim], elements bf16 or
 *          int8 (dtype).  16-byte aligned.  v == NULL or v == k means K and V
 *          are one tensor (Lab5-Gemma4 model overview: W_K = W_V on global
 *          layers); it is then read once per key.
 *   k_scale, v_scale: fp32 scale tables of an int8 pool.
 *          PKV_SCALE_PER_TOKEN: [num_blocks * block_size], indexed by slot,
 *          written by paged_kv_append, 16-byte aligned;
 *          PKV_SCALE_PER_HEAD:  [num_kv_heads], set by the caller (static).
 *          Unused (may be NULL) for bf16 pools; v_scale unused when K == V.
 *   block_size must be 16; head_dim must be 64, 128 or 256.
 *   ring_blocks: 0 = paged layout: row b of a block table lists the
 *          sequence's blocks in logical order (entry j holds positions
 *          [16j, 16j+16)).  > 0 = ring layout of a sliding-window layer
 *          (Lab5-Gemma4, Ring KV Cache: position t in slot t mod W of a fixed
 *          ring, W = ring_blocks * block_size): row b lists the sequence's
 *          ring, and position t lives in entry (t mod W) / 16 at offset
 *          t mod 16, overwriting a position W earlier.  A decode with window
 *          w over a ring needs W >= w + 1 (the w + 1 keys of [pos-w, pos]);
 *          a sequence uses min(len, W) slots whatever its length.
 */
typedef struct pkv_pool {
    void *k;
    void *v;
    float *k_scale;
    float *v_scale;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t dtype;      /* PKV_BF16 | PKV_INT8 */
    int32_t scale_mode; /* PKV_SCALE_* (PKV_SCALE_NONE only for bf16) */
    int32_t ring_blocks; /* 0 = paged; > 0 = ring of this many blocks per sequence */
} pkv_pool;

/*
 * paged_kv_append -- write each new token's K and V into its slot.
 * (CS336 lecture 10, KV-cache section: "append new K/V"; tiniestgpt notes,
 * sections 2 and 8: slot ids; section 5: int8 quantisation with
 * scale = max|x|/127, x_q = round(x/scale) from the CS336 guide's int8
 * section.)
 *   k, v:          [num_tokens][num_kv_heads][head_dim] bf16, 16-byte
 *                  aligned; v ignored (may be NULL) when the pool has K == V.
 *   slot_mapping:  [num_tokens] int64, 8-byte aligned; token t goes to block
 *                  slot / block_size, offset slot % block_size; a negative
 *                  slot is padding and is skipped.
 *   bf16 pool: bit copy.  int8 per token: scale = max|x| / 127 over the
 *   token's num_kv_heads*head_dim values (fp32, IEEE division), stored at
 *   scale[slot]; q = clamp(round_half_even(x / scale), -127, 127); a zero
 *   scale stores zeros.  Non-finite inputs: NaN is ignored by max|x| and
 *   stored as code 0; +-inf makes the token's scale inf (every code of that
 *   token 0) or, under a per-head scale, saturates to +-127.  int8 per
 *   head: the same rounding with the caller's static scale[h].  K and V are
 *   quantised separately.
 *   Tokens that map to the same slot race (the last writer is unspecified).
 */
PKV_API int paged_kv_append(const void *k, const void *v, const int64_t *slot_mapping,
                            int32_t num_tokens, const pkv_pool *pool, void *stream);

/*
 * paged_kv_slot_mapping -- slot ids of num_tokens new tokens under the
 * pool's layout, computed on the device (so that a captured step needs only
 * positions, not host-computed slots): token i of sequence seq_ids[i] (or i
 * when seq_ids is NULL) at absolute position positions[i] goes to
 *   paged (ring_blocks 0):  block_table[seq][pos / 16] * 16 + pos % 16
 *   ring:                   block_table[seq][(pos mod W) / 16] * 16 + pos % 16
 * (Lab5-Gemma4, Paged Attention and Ring KV Cache sections).  A negative
 * position gives slot -1 (padding, which paged_kv_append skips); a table
 * entry past max_blocks_per_seq or outside [0, num_blocks) gives -1 and sets
 * PKV_DEV_BAD_BLOCK.
 *   block_table: [batch][max_blocks_per_seq] int32; seq_ids: [num_tokens]
 *   int32 or NULL; positions: [num_tokens] int64; slot_mapping (output):
 *   [num_tokens] int64, 8-byte aligned.  All device pointers.
 */
PKV_API int paged_kv_slot_mapping(const pkv_pool *pool, const int32_t *block_table,
                                  int32_t max_blocks_per_seq, const int32_t *seq_ids,
                                  const int64_t *positions, int32_t num_tokens,
                                  int64_t *slot_mapping, void *stream);

/*
 * Rotary position embedding fused with the append.  The Lab5-Gemma4 model
 * overview names p-RoPE on the global layers but gives no formula; the
 * rotation is RoFormer's (Su et al., "RoFormer: Enhanced Transformer with
 * Rotary Position Embedding", section 3.2 and the element-wise form of
 * section 3.4.2): pair i of a vector at position m turns by m * theta_i,
 *     a' = a cos(m theta_i) - b sin(m theta_i),
 *     b' = a sin(m theta_i) + b cos(m theta_i),
 * and p-RoPE (Barbero et al., "Round and Round We Go! What makes Rotary
 * Positional Encodings useful?") keeps only the highest frequencies: the
 * first rotary_pairs pairs of a decreasing theta table turn, the others pass
 * unchanged.  theta is the caller's (RoFormer: theta_i = base^(-2i/D)).
 *
 * paged_rope_cos_sin_table -- the (cos, sin) table of every position.
 *   theta:  [rotary_pairs] fp64, radians per position, 8-byte aligned.
 *   table (output): [num_positions][rotary_pairs] pairs of fp32,
 *          table[m][i] = (fp32(cos(m theta_i)), fp32(sin(m theta_i))), the
 *          angle one fp64 product and its cosine and sine fp64 values
 *          rounded once to fp32; 8-byte aligned.  Computed once per model.
 */
PKV_API int paged_rope_cos_sin_table(const double *theta, int32_t rotary_pairs,
                                     int64_t num_positions, float *table, void *stream);

/*
 * paged_kv_append_rope -- rotate each new token's q and k by its position,
 * write the rotated q to q_out and append the rotated k (and the unrotated
 * v) as paged_kv_append does (bf16 copy or int8 quantisation of the rotated
 * values).  With K and V one tensor the stored (rotated) row serves as both.
 *   q:         [num_tokens][num_q_heads][head_dim] bf16, 16-byte aligned, or
 *              NULL (k only); q_out: same shape, may be q (in place).
 *   k, v, slot_mapping, pool: as paged_kv_append.
 *   positions: [num_tokens] int64, 8-byte aligned.  A negative position is
 *              padding: q_out gets the q row unchanged and nothing is
 *              appended.  A position >= num_positions is treated the same
 *              and sets PKV_DEV_BAD_POSITION.  A token with a valid position
 *              and a negative slot has its q rotated and appends nothing.
 *   table:     from paged_rope_cos_sin_table (num_positions rows of
 *              rotary_pairs entries); rotary_pairs in [0, head_dim / 2].
 *   layout:    PKV_ROPE_HALVES or PKV_ROPE_INTERLEAVED.
 * Arithmetic: with (c, s) from the table, t = b * s, a' = fma(a, c, -t),
 * t = b * c, b' = fma(a, s, t) in fp32, each rounded once to bf16 (nearest,
 * ties to even); the stored bits are fixed by it.  Dims that do not turn are
 * copied bit for bit; a non-finite input gives a non-finite output.
 */
PKV_API int paged_kv_append_rope(const void *q, void *q_out, int32_t num_q_heads, const void *k,
                                 const void *v, const int64_t *positions,
                                 const int64_t *slot_mapping, int32_t num_tokens,
                                 const float *table, int64_t num_positions,
                                 int32_t rotary_pairs, int32_t layout, const pkv_pool *pool,
                                 void *stream);

/*
 * paged_decode_split_tokens -- the split length paged_decode_attention uses
 * for split_tokens.  PKV_SPLIT_AUTO resolves to 4096 keys for GQA groups of
 * 8 or more and 2048 otherwise, or to 0 (a single pass) when the longest key
 * range (max_seq_len, window) fits in one split.  Returns 0 for a single
 * pass, a positive multiple of block_size, or a negative PKV_E_* code.
 */
PKV_API int32_t paged_decode_split_tokens(int32_t batch, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t block_size,
                                          int32_t max_seq_len, int32_t window,
                                          int32_t split_tokens);

/*
 * paged_decode_num_splits -- the most key splits a sequence of length at
 * most max_seq_len can have for a resolved split length (>= 1).
 */
PKV_API int32_t paged_decode_num_splits(int32_t block_size, int32_t max_seq_len, int32_t window,
                                        int32_t split_tokens);

/*
 * paged_decode_workspace_bytes -- device scratch paged_decode_attention
 * uses for these sizes: the largest of the split partials (when the key
 * ranges are split: partial log-sum-exp [batch][num_splits][num_q_heads]
 * fp32, then, 256-byte aligned, partial outputs
 * [batch][num_splits][num_q_heads][head_dim] fp32), the tensor-core kernel's
 * scratch (paged_decode_partial_workspace_bytes) and, for a single pass on
 * CUDA cores, (sequence, length) int32 pairs of the batch longest first (used
 * when the grid exceeds one wave; a single pass given no workspace runs in
 * batch order).  0 only for batch 0.
 */
PKV_API size_t paged_decode_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t block_size, int32_t max_seq_len,
                                            int32_t window, int32_t split_tokens);

/*
 * paged_decode_partial_workspace_bytes -- device scratch of the tensor-core
 * kernel (bf16 pools, head_dim 128 or 256, 8 to 16 query heads per KV head),
 * which paged_decode_split_partial needs as its workspace and which
 * paged_decode_workspace_bytes includes: the stream-K plan (one entry per
 * SM and a prefix sum per sequence) and the partial states of key ranges
 * cut between SMs.  0 for shapes that run on the CUDA-core kernel.
 */
PKV_API size_t paged_decode_partial_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                                    int32_t num_kv_heads, int32_t head_dim);

/*
 * paged_decode_attention -- one decode step of one layer: for every sequence
 * b and query head h,
 *     out[b][h] = softmax_j(softmax_scale * <q[b][h], K_b[j]>) V_b[j]
 * over the keys j in [lo, pos], pos = seq_lens[b] - 1,
 * lo = window > 0 ? max(0, pos - window) : 0 (Lab5-Gemma4 sliding-window
 * section: position i sees [i-w, i]; window 0 = global causal layer).
 * K_b[j] is row j % block_size of physical block
 * block_table[b][j / block_size], kv head h / (num_q_heads / num_kv_heads)
 * (consecutive query heads share a KV head).  int8 values are dequantised
 * after the gather.  Online softmax in fp32 (Lab5-Gemma4, Flash Attention
 * section): scores are never written to memory.  Blocks outside [lo, pos]
 * are never read.
 *   q:            [batch][num_q_heads][head_dim] bf16, 16-byte aligned.
 *   block_table:  [batch][max_blocks_per_seq] int32 (for a ring pool, each
 *                 row is the sequence's ring; max_blocks_per_seq >=
 *                 ring_blocks, and lengths are not bounded by the table).
 *   seq_lens:     [batch] int32, length including the token appended this
 *                 step; 0 gives a zero output row.
 *   max_seq_len:  host upper bound on every seq_lens[b] (tiniestgpt notes,
 *                 section 8); it sizes the grid.
 *   split_tokens: 0 = single pass; > 0 = split each key range into pieces
 *                 of this many keys (multiple of block_size) and merge them
 *                 with a log-sum-exp combine; PKV_SPLIT_AUTO = library's
 *                 choice.  The tensor-core kernel balances the key ranges
 *                 across SMs itself and ignores it (same result up to
 *                 rounding).
 *   workspace:    device scratch of paged_decode_workspace_bytes(...) bytes,
 *                 256-byte aligned.  Required (PKV_E_WORKSPACE without it)
 *                 when the call splits the key ranges or runs on the
 *                 tensor-core kernel (paged_decode_uses_tensor_cores);
 *                 optional for a single pass on the CUDA-core kernel, which
 *                 then takes the sequences in batch order instead of longest
 *                 first.  Calls on one stream may share it; concurrent calls
 *                 may not.
 *   out:          [batch][num_q_heads][head_dim], bf16 (out_dtype
 *                 PKV_OUT_BF16) or fp32 (PKV_OUT_F32), 16-byte aligned.
 */
PKV_API int paged_decode_attention(const void *q, const pkv_pool *pool, const int32_t *block_table,
                                   int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                   int32_t batch, int32_t num_q_heads, int32_t max_seq_len,
                                   int32_t window, float softmax_scale, int32_t split_tokens,
                                   void *workspace, size_t workspace_bytes, void *out,
                                   int32_t out_dtype, void *stream);

/*
 * paged_prefill_attention -- attention of a chunk of new tokens per sequence
 * (q_len > 1: chunked prefill, or the gamma + 1 tokens a speculative step
 * verifies).  Lab5-Gemma4, Flash Attention section: prefill's q_len > 1
 * beside decode's q_len = 1, causal and sliding-window masks over the
 * cache's history, GQA without repeated K/V, the partial last tile;
 * tiniestgpt notes, section 7: the verify step feeds gamma + 1 tokens.
 * Sequence b's chunk is its last n_b = q_start[b+1] - q_start[b] tokens,
 * already appended to the pool (seq_lens include them): query row
 * q_start[b] + i is the token at position seq_lens[b] - n_b + i, and for
 * each query head h
 *     out[row][h] = softmax_j(softmax_scale * <q[row][h], K_b[j]>) V_b[j]
 * over the keys j in [lo, pos] of its own position pos (lo = pos - window
 * on sliding layers, else 0): causal within the chunk.  A chunk of one
 * token is the decode.
 *   q:          [total_q][num_q_heads][head_dim] bf16, 16-byte aligned.
 *   q_start:    [batch + 1] int32, non-decreasing, q_start[0] = 0,
 *               q_start[batch] = total_q.
 *   max_q_len:  host bound on every n_b (sizes the grid); a chunk longer
 *               than it, or than its sequence, sets PKV_DEV_LEN_BOUND.
 *   pool:       bf16 only (PKV_E_UNSUPPORTED for int8), paged or ring (a
 *               ring must hold window + max_q_len slots: the chunk's first
 *               query still sees keys its last token's slot would
 *               overwrite in a smaller ring); num_q_heads / num_kv_heads in
 *               {1, 2, 4, 8, 16}.
 *   other arguments as for paged_decode_attention; out: [total_q]
 *   [num_q_heads][head_dim], bf16 or fp32.  No workspace.
 */
PKV_API int paged_prefill_attention(const void *q, const int32_t *q_start, int32_t total_q,
                                    int32_t max_q_len, const pkv_pool *pool,
                                    const int32_t *block_table, int32_t max_blocks_per_seq,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t max_seq_len, int32_t window, float softmax_scale,
                                    void *out, int32_t out_dtype, void *stream);

/*
 * paged_decode_split_partial -- the first step of the split-KV path: every
 * (sequence, query head, split s) attends over keys
 * [lo + s*split_tokens', ...) where split_tokens' counts from the block
 * holding lo (splits are block-aligned: split s covers logical blocks
 * lo/bs + s*split_tokens/bs ... of the sequence, clipped to [lo, pos]).
 * For a sequence whose range has a single split the final output row is
 * written to `out` directly; otherwise partial_lse[b][s][h] (natural log of
 * the sum of exp(score)) and partial_o[b][s][h][:] (the split's normalised
 * output) are written: split-major, so that one split's query heads are
 * contiguous.  split_tokens must be a positive multiple of
 * block_size; num_splits >= paged_decode_num_splits(...); both partial
 * arrays 16-byte aligned.  workspace: device
 * scratch of paged_decode_partial_workspace_bytes(...) bytes, 256-byte
 * aligned (NULL allowed when that is 0).
 */
PKV_API int paged_decode_split_partial(const void *q, const pkv_pool *pool,
                                       const int32_t *block_table, int32_t max_blocks_per_seq,
                                       const int32_t *seq_lens, int32_t batch,
                                       int32_t num_q_heads, int32_t max_seq_len, int32_t window,
                                       float softmax_scale, int32_t split_tokens,
                                       float *partial_lse, float *partial_o, int32_t num_splits,
                                       void *workspace, size_t workspace_bytes, void *out,
                                       int32_t out_dtype, void *stream);

/*
 * paged_decode_lse_combine -- the second step: for each sequence with more
 * than one split and each query head,
 *     L = log sum_s exp(lse_s),   out = sum_s exp(lse_s - L) o_s
 * (the online-softmax merge of Lab5-Gemma4's Flash Attention section applied
 * to whole splits).  Sequences with one split are left untouched.  The
 * split count of each sequence is recomputed from seq_lens, window,
 * block_size and split_tokens exactly as paged_decode_split_partial does.
 */
PKV_API int paged_decode_lse_combine(const float *partial_lse, const float *partial_o,
                                     const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                     int32_t head_dim, int32_t block_size, int32_t window,
                                     int32_t split_tokens, int32_t num_splits, void *out,
                                     int32_t out_dtype, void *stream);

/*
 * paged_decode_attention_noalloc -- paged_decode_attention for callers that
 * cannot allocate device memory and so cannot pass a workspace: a plugin
 * whose host framework gives it only its inputs and outputs, an engine that
 * has already reserved all of HBM for its KV pool, or a latency-critical
 * loop in which cudaMalloc/cudaFree would synchronise the device.  None of
 * the pages has a counterpart; this is a library convenience.
 *   Same arguments and result as paged_decode_attention, minus the
 *   workspace.  The split-KV partials (and the tensor-core kernel's
 *   scratch) go to a fixed array of
 *   PKV_STATIC_SCRATCH_BYTES in device memory that every GPU which loads the
 *   library holds until the process exits.  Sizes whose scratch would not
 *   fit are rejected with PKV_E_WORKSPACE before anything is launched.
 *   Nothing here calls cudaMalloc, cudaFree or any allocating routine.
 *   The first call on a device looks the array's address up on that device
 *   (cudaGetSymbolAddress, the device current); make that first call before
 *   any stream capture.  The address is kept for the life of the process:
 *   after cudaDeviceReset (or any reset of the device's primary context) the
 *   array is gone and this entry point must not be called again.  The same
 *   holds for every call of this library, which caches the address of its
 *   device error word the same way.  All calls share the one array and it keeps the
 *   previous call's contents (no part of it needs to start at zero: every
 *   partial is written before it is read), so calls that overlap on the GPU
 *   -- on two streams, or from two threads -- race and must be serialised by
 *   the caller.
 */
#define PKV_STATIC_SCRATCH_BYTES (32u << 20) /* 32 MiB per device */
PKV_API int paged_decode_attention_noalloc(const void *q, const pkv_pool *pool,
                                           const int32_t *block_table, int32_t max_blocks_per_seq,
                                           const int32_t *seq_lens, int32_t batch,
                                           int32_t num_q_heads, int32_t max_seq_len,
                                           int32_t window, float softmax_scale,
                                           int32_t split_tokens, void *out, int32_t out_dtype,
                                           void *stream);

/*
 * One layer of a decode step (paged_decode_step).  Every layer has its own
 * pool, query, new token and output; the layers share the step's layout
 * (block table, lengths, slot ids), as the layers of one model do.
 */
typedef struct pkv_layer {
    pkv_pool pool;       /* this layer's pool */
    const void *q;       /* [batch][num_q_heads][head_dim] bf16, 16-byte aligned */
    const void *k_new;   /* [batch][num_kv_heads][head_dim] bf16: each sequence's new token */
    const void *v_new;   /* likewise for V; ignored (may be NULL) when the pool has K == V */
    void *out;           /* [batch][num_q_heads][head_dim], bf16 or fp32 (out_dtype) */
    int32_t window;      /* 0 = global causal layer; > 0 = sliding window (keys [pos-w, pos]) */
    float softmax_scale;
    /* Optional RoPE fused with the append (paged_kv_append_rope).  With
     * rope_table not NULL, q is rotated into q_rotated and k_new is rotated
     * before it is stored, each sequence's new token at position
     * seq_lens[b] - 1, and the decode reads q_rotated.  All zero: no RoPE. */
    const float *rope_table;   /* [rope_num_positions][rope_pairs] (cos, sin) pairs */
    int64_t rope_num_positions;
    int32_t rope_pairs;        /* rotated pairs, <= head_dim / 2 */
    int32_t rope_layout;       /* PKV_ROPE_HALVES or PKV_ROPE_INTERLEAVED */
    void *q_rotated;           /* [batch][num_q_heads][head_dim] bf16, 16-byte aligned; may be q */
} pkv_layer;

/*
 * paged_decode_step_workspace_bytes -- device scratch paged_decode_step
 * needs for these layers: the largest paged_decode_workspace_bytes of any
 * layer (the layers run one after another on one stream and share it).
 * `layers` is a host array.  0 if layers is NULL or num_layers <= 0.
 */
PKV_API size_t paged_decode_step_workspace_bytes(const pkv_layer *layers, int32_t num_layers,
                                                 int32_t batch, int32_t num_q_heads,
                                                 int32_t max_seq_len, int32_t split_tokens);

/*
 * paged_decode_step -- one decode step of a whole model's attention: for
 * each layer in order, paged_kv_append of the layer's new tokens at
 * slot_mapping (paged_kv_append_rope at positions seq_lens[b] - 1 for a
 * layer with a RoPE table), then paged_decode_attention over the layer's
 * pool, all enqueued on `stream` by one call.  (tiniestgpt notes, section 8: a decode
 * step over static block_table / seq_lens / slot_ids buffers with a host-side
 * length bound, captured once as a CUDA graph and replayed; CS336 lecture 10,
 * local/global section: sliding-window layers interleaved with global ones.)
 *   layers:        host array of num_layers descriptors (read during the
 *                  call only).
 *   slot_mapping:  [batch] int64 device array, the new token's slot per
 *                  sequence (negative = padding, skipped), shared by all
 *                  layers; block_table, seq_lens, max_seq_len, split_tokens
 *                  as for paged_decode_attention, shared by all layers.
 *   workspace:     paged_decode_step_workspace_bytes(...) bytes, 256-byte
 *                  aligned (shared by the layers; see paged_decode_attention
 *                  for when it is required).
 * Every layer's arguments are validated before anything is launched; a
 * launch that fails part-way leaves the earlier layers enqueued.  Allocates
 * nothing and reads no device data on the host, so a whole step can be
 * captured in one CUDA graph.  pkv_last_launch_count() counts every kernel
 * of the step.
 */
PKV_API int paged_decode_step(const pkv_layer *layers, int32_t num_layers,
                              const int64_t *slot_mapping, const int32_t *block_table,
                              int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                              int32_t num_q_heads, int32_t max_seq_len, int32_t split_tokens,
                              void *workspace, size_t workspace_bytes, int32_t out_dtype,
                              void *stream);

/*
 * paged_decode_uses_tensor_cores -- 1 if decodes over this pool with
 * num_q_heads query heads run on the tensor-core kernel (bf16 pool,
 * head_dim 128 or 256, 8 to 16 query heads per KV head; PKV_DISABLE_TC=1 /
 * PKV_FORCE_TC=1 in the environment override it), 0 if on the CUDA-core
 * kernel, or a negative PKV_E_* code for an invalid pool.  Host only.
 */
PKV_API int32_t paged_decode_uses_tensor_cores(const pkv_pool *pool, int32_t num_q_heads);

/*
 * pkv_check_bounded_wait -- diagnostic of the failure path every pipeline
 * wait of this library takes: one CTA of `threads` threads waits, with the
 * kernels' own bounded wait (spin = 0: the sleeping wait; 1: the polling
 * wait), on an mbarrier phase that nothing completes.  Each wait gives up
 * after limit_ns nanoseconds (1 us .. 2 s), sets PKV_DEV_TIMEOUT in the
 * device error word and the kernel returns; out[t] = 1 for every thread
 * whose wait gave up.  Nothing faults and the context stays usable.  Read
 * the result after synchronising (pkv_device_status).  out: [threads] int32
 * device array.
 */
PKV_API int pkv_check_bounded_wait(uint64_t limit_ns, int32_t spin, int32_t *out,
                                   int32_t threads, void *stream);

/* Number of kernels the calling thread's last call of this library launched. */
PKV_API int32_t pkv_last_launch_count(void);

/* Message of the last host-side error on this thread ("" if none). */
PKV_API const char *pkv_last_error(void);

/*
 * pkv_device_status -- the device error word (PKV_DEV_* bits) of the
 * current device, optionally clearing it.  This call synchronises the
 * device; call it after the stream's work has finished.  Returns a
 * negative PKV_E_* code if the device cannot be queried.
 */
PKV_API int pkv_device_status(int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
