// pkv_write.h -- host-side interface of the KV-writing kernels (append,
// RoPE fused with the append, device slot mapping) and of the bounded-wait
// diagnostic, all in pkv_append.cu.  Not installed; not part of the public
// ABI.  Kept apart from pkv_internal.h so that the decode kernels' sources
// do not change when these do.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

struct AppendParams {
    const uint16_t *k;
    const uint16_t *v;
    const int64_t *slot_mapping;
    void *pool_k;
    void *pool_v;
    float *k_scale;
    float *v_scale;
    int32_t num_tokens;
    int32_t row;              // num_kv_heads * head_dim
    int32_t head_dim;
    int64_t num_slots;
    int32_t scale_mode;
    int32_t alias;
    unsigned int *err;
};

// RoPE fused with the append (with AppendParams): q rotated into q_out, k
// rotated before it is stored.
struct RopeParams {
    const uint16_t *q;        // [T][H_q][D] bf16 or NULL (no q)
    uint16_t *q_out;          // same shape; may be q
    const int64_t *positions; // [T], or NULL: token t of sequence t at seq_lens[t] - 1
    const int32_t *seq_lens;  // [T] when positions is NULL
    const float2 *table;      // [num_positions][pairs] (cos, sin)
    int64_t num_positions;
    int32_t num_q_heads;
    int32_t pairs;            // rotated pairs, <= D / 2
    int32_t layout;           // PKV_ROPE_HALVES or PKV_ROPE_INTERLEAVED
};

cudaError_t launch_append(const AppendParams &p, int int8, cudaStream_t s);
size_t append_rope_smem_bytes(int row, int pairs);
cudaError_t launch_append_rope(const AppendParams &p, const RopeParams &r, int int8,
                               cudaStream_t s);
cudaError_t launch_rope_table(const double *theta, int pairs, int64_t num_positions,
                              float *table, cudaStream_t s);
cudaError_t launch_bounded_wait(uint64_t limit_ns, int spin, int *out, int threads,
                                unsigned int *err, cudaStream_t s);
cudaError_t launch_slot_mapping(const int32_t *block_table, int max_blocks, int ring_blocks,
                                int num_blocks, const int32_t *seq_ids, const int64_t *positions,
                                int num_tokens, int64_t *slots, unsigned int *err, cudaStream_t s);

}  // namespace pkv
