// pkv_internal.h -- host-side interface between the C-ABI layer and the
// kernel launchers.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kBlock = 16;  // tokens per paged block (block_size)

// Parameters of the decode kernels (passed by value to the kernel).
struct DecodeParams {
    const uint16_t *q;        // [B][H_q][D] bf16 bits
    const int32_t *block_table;
    const int32_t *seq_lens;
    const float *k_scale;
    const float *v_scale;
    float *part_lse;          // [B][num_splits][H_q]
    float *part_o;            // [B][num_splits][H_q][D]
    void *out;                // [B][H_q][D]
    int32_t max_blocks;       // block_table row length
    int32_t ring_blocks;      // 0: paged; > 0: logical block j lives in entry j % ring_blocks
    int32_t scale_mode;
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;            // H_q / H_kv
    int32_t head_chunks;      // CTAs per kv head along the query group
    int32_t num_blocks;       // pool blocks
    int32_t window;
    int32_t max_seq_len;
    int32_t split_blocks;     // paged blocks per split; 0 = single pass
    int32_t num_splits;       // grid extent along splits
    int32_t alias;            // K and V are one tensor
    int32_t out_f32;
    int32_t num_stages;       // smem ring depth
    float qk_scale_log2;      // softmax_scale * log2(e)
    unsigned int *err;        // device error word
    int32_t head_dim;
    // tensor-core kernel only (workspace): stream-K plan and partial states
    int4 *tc_plan;            // [0] = {W, C}; [1 + c] = CTA c's first item; [1 + C] = end
    int32_t *tc_seqoff;       // [batch + 1] first tile of each sequence
    float *sub_lse;           // [grid][2][16] partial states of items cut at CTA boundaries
    float *sub_o;             // [grid][2][16][head_dim]
    int32_t *tc_flags;        // [grid][2] tickets of cut items, by first CTA (cleared by the plan)
    // CUDA-core kernel: (sequence, length) pairs longest first (NULL = in
    // order), and the workspace that may hold them ([batch] int2; NULL = none)
    const int32_t *seq_order;
    int32_t *order_ws;
};

// Parameters of the chunk (q_len > 1) attention kernel.
struct PrefillParams {
    const uint16_t *q;        // [total][H_q][D] bf16
    const int32_t *q_start;   // [B + 1] first query row of each sequence's chunk
    const int32_t *block_table;
    const int32_t *seq_lens;
    void *out;                // [total][H_q][D]
    unsigned int *err;
    int32_t max_blocks;
    int32_t ring_blocks;
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t num_blocks;
    int32_t window;
    int32_t max_seq_len;
    int32_t max_q_len;        // host bound on any chunk's length (sizes the grid)
    int32_t alias;
    int32_t out_f32;
    int32_t num_buffers;      // K/V tile buffers
    float qk_scale_log2;
};

struct CombineParams {
    const float *part_lse;    // [B][num_splits][H_q]
    const float *part_o;      // [B][num_splits][H_q][D]
    const int32_t *seq_lens;
    void *out;
    int32_t batch;
    int32_t num_q_heads;
    int32_t head_dim;
    int32_t window;
    int32_t split_blocks;
    int32_t num_splits;
    int32_t out_f32;
};

// CUDA-core decode kernel family (TMA-fed smem ring, one CTA per
// (split, kv head, head chunk, sequence)).
int decode_group_tile(int group);  // query heads per CTA for a GQA group
size_t decode_smem_bytes(int head_dim, int int8, int alias, int per_token, int group_tile,
                         int num_stages);
int decode_ring_stages(int head_dim, int int8, int alias, int per_token, int group_tile);
cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                          int head_dim, int int8, int group_tile, cudaStream_t s);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t s);

// Tensor-core decode kernel (bf16 pools, head_dim 128/256, group <= 16):
// persistent stream-K over the 128-key tiles of all (sequence, kv head,
// split) items, one CTA per SM (at most kTcMaxGrid); num_stages = ring units
// of 32 KB.  Launches the plan and the (cooperative) decode kernel; needs
// decode_tc_scratch_bytes of workspace bound with decode_tc_bind_scratch.
constexpr int kTcMaxGrid = 256;
int decode_tc_group_pad(int group);  // 0 if the group is too large
size_t decode_tc_smem_bytes(int num_units);
size_t decode_tc_scratch_bytes(int batch, int head_dim);
void decode_tc_bind_scratch(DecodeParams &p, void *scratch, int batch);
int decode_tc_grid();
cudaError_t launch_decode_tc(const DecodeParams &p, const CUtensorMap &tmk,
                             const CUtensorMap &tmv, const CUtensorMap &tmq, int head_dim,
                             cudaStream_t s);
// Chunk attention (tensor cores, bf16 pools): K/V tile buffers that fit, the
// shared memory of a launch, and the launch itself.
int prefill_num_buffers(int head_dim, int alias);
size_t prefill_smem_bytes(int head_dim, int alias, int num_buffers);
cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           const CUtensorMap &tmq, int head_dim, cudaStream_t s);

// Count one kernel launch of the current API call (pkv_last_launch_count).
void note_launch();

}  // namespace pkv
