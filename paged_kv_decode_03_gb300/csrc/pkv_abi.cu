// pkv_abi.cu -- the extern "C" entry points declared in include/pagedkv.h:
// argument validation on the host, TMA tensor-map encoding, split-length
// resolution and kernel launches.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_write.h"

namespace pkv {

// Device error word (PKV_DEV_* bits), one per device that loads the
// library.  Kernels receive its address as a parameter.
static __device__ unsigned int g_error_word = 0;

// Address of g_error_word on the current device (looked up once per device).
static unsigned int *error_word_ptr()
{
    static std::mutex mu;
    static unsigned int *ptrs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess)
            return nullptr;
        ptrs[dev] = static_cast<unsigned int *>(p);
    }
    return ptrs[dev];
}

static thread_local std::string t_last_error;
static thread_local int t_launches = 0;  // kernels launched by this thread's last call

void note_launch() { ++t_launches; }

static int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

static int cuda_fail(cudaError_t e, const char *what)
{
    t_last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return static_cast<int>(e);
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Tensor map over a pool [num_blocks*block_size][H_kv][D] (innermost first:
// D, H_kv, rows); box = {chunk elements, 1 head, block_size rows}.
static int encode_pool_map(CUtensorMap *map, void *base, const pkv_pool &pool)
{
    auto fn = encode_fn();
    if (!fn)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled is unavailable");
    const int es = pool.dtype == PKV_INT8 ? 1 : 2;
    const int che = pool.head_dim * es > 256 ? 256 / es : pool.head_dim;
    cuuint64_t dims[3] = {(cuuint64_t)pool.head_dim, (cuuint64_t)pool.num_kv_heads,
                          (cuuint64_t)pool.num_blocks * (cuuint64_t)pool.block_size};
    cuuint64_t strides[2] = {(cuuint64_t)pool.head_dim * es,
                             (cuuint64_t)pool.num_kv_heads * pool.head_dim * es};
    cuuint32_t box[3] = {(cuuint32_t)che, 1u, (cuuint32_t)pool.block_size};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                    3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PKV_OK;
}

// Tensor map for the tensor-core kernel: box = {64 dims, 1 head,
// block_size rows} with the 128-byte swizzle that tcgen05.mma expects of a
// K-major (and, read transposed, MN-major) bf16 operand.
static int encode_pool_map_tc(CUtensorMap *map, void *base, const pkv_pool &pool)
{
    auto fn = encode_fn();
    if (!fn)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)pool.head_dim, (cuuint64_t)pool.num_kv_heads,
                          (cuuint64_t)pool.num_blocks * (cuuint64_t)pool.block_size};
    cuuint64_t strides[2] = {(cuuint64_t)pool.head_dim * 2,
                             (cuuint64_t)pool.num_kv_heads * pool.head_dim * 2};
    cuuint32_t box[3] = {64u, 1u, (cuuint32_t)pool.block_size};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled (swizzled) failed (%d)", (int)r);
    return PKV_OK;
}

// Tensor map over q [batch*num_q_heads][head_dim] bf16 for the tensor-core
// kernel: box = {64 dims, 16 rows} with the 128-byte swizzle, i.e. one
// 64-dim column of Q^T for 16 query heads as the K-major B operand.
static int encode_q_map(CUtensorMap *map, const void *q, int32_t rows, int32_t head_dim)
{
    auto fn = encode_fn();
    if (!fn)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    cuuint32_t box[2] = {64u, 16u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
    return PKV_OK;
}

// Tensor map over the chunk queries q [total][H_q][D] bf16 for the chunk
// attention kernel: box = {64 dims, G heads, 128 / G tokens} with the
// 128-byte swizzle, i.e. 128 query rows (token, head) of one kv head's group
// as the K-major A operand.
static int encode_chunk_q_map(CUtensorMap *map, const void *q, int32_t total, int32_t num_q_heads,
                              int32_t head_dim, int32_t group)
{
    auto fn = encode_fn();
    if (!fn)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)total};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_q_heads * head_dim * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)group, (cuuint32_t)(128 / group)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(PKV_E_DRIVER, "cuTensorMapEncodeTiled (chunk q) failed (%d)", (int)r);
    return PKV_OK;
}

static bool env_flag(const char *name)
{
    const char *e = getenv(name);
    return e && e[0] == '1';
}

// Whether shapes alone allow the tensor-core kernel (and so its workspace):
// head_dim 128 or 256 and 8 to 16 query heads per KV head (any group up to
// 16 with PKV_FORCE_TC=1).
static bool tc_shape(int group, int head_dim)
{
    if ((head_dim != 128 && head_dim != 256) || group < 1 || decode_tc_group_pad(group) == 0)
        return false;
    if (env_flag("PKV_DISABLE_TC"))
        return false;
    return group >= 8 || env_flag("PKV_FORCE_TC");
}

// Whether a decode runs on the tensor-core kernel: bf16 pool, head_dim 128
// or 256, and 8 to 16 query heads per KV head.  Below 8 heads the CUDA-core
// kernel keeps up with HBM and, with several CTAs per SM, measures faster.
// PKV_DISABLE_TC=1 forces the CUDA-core kernel and PKV_FORCE_TC=1 the
// tensor-core kernel for any group <= 16 (both read at every call).
static bool use_tc(const pkv_pool *pool, int group)
{
    if (pool->dtype != PKV_BF16 || (pool->head_dim != 128 && pool->head_dim != 256))
        return false;
    return tc_shape(group, pool->head_dim);
}

// ---------------------------------------------------------- validation
static int check_pool(const pkv_pool *pool)
{
    if (!pool)
        return fail(PKV_E_NULL, "pool is NULL");
    if (!pool->k)
        return fail(PKV_E_NULL, "pool->k is NULL");
    if (pool->block_size != kBlock)
        return fail(PKV_E_UNSUPPORTED, "block_size %d not supported (16 only)", pool->block_size);
    if (pool->head_dim != 64 && pool->head_dim != 128 && pool->head_dim != 256)
        return fail(PKV_E_UNSUPPORTED, "head_dim %d not supported (64, 128, 256)", pool->head_dim);
    if (pool->num_kv_heads <= 0 || pool->num_blocks <= 0)
        return fail(PKV_E_SHAPE, "num_kv_heads and num_blocks must be positive");
    if ((int64_t)pool->num_blocks * pool->block_size > INT32_MAX)
        return fail(PKV_E_SHAPE, "pool has more than 2^31 slots");
    if (pool->dtype != PKV_BF16 && pool->dtype != PKV_INT8)
        return fail(PKV_E_UNSUPPORTED, "dtype %d", pool->dtype);
    if (pool->ring_blocks < 0)
        return fail(PKV_E_ARG, "ring_blocks %d < 0", pool->ring_blocks);
    if (!aligned(pool->k, 16) || (pool->v && !aligned(pool->v, 16)))
        return fail(PKV_E_ALIGN, "pool k/v must be 16-byte aligned");
    const bool alias = pool->v == nullptr || pool->v == pool->k;
    if (pool->dtype == PKV_BF16) {
        if (pool->scale_mode != PKV_SCALE_NONE)
            return fail(PKV_E_ARG, "bf16 pools take no scales");
    } else {
        if (pool->scale_mode != PKV_SCALE_PER_TOKEN && pool->scale_mode != PKV_SCALE_PER_HEAD)
            return fail(PKV_E_ARG, "int8 pools need per-token or per-head scales");
        if (!pool->k_scale || (!alias && !pool->v_scale))
            return fail(PKV_E_NULL, "int8 pool scale table is NULL");
        if (pool->scale_mode == PKV_SCALE_PER_TOKEN &&
            (!aligned(pool->k_scale, 16) || (!alias && !aligned(pool->v_scale, 16))))
            return fail(PKV_E_ALIGN, "per-token scale tables must be 16-byte aligned");
        if (!aligned(pool->k_scale, 4) || (!alias && !aligned(pool->v_scale, 4)))
            return fail(PKV_E_ALIGN, "scale tables must be 4-byte aligned");
    }
    return PKV_OK;
}

// Ring depth override for tuning builds (-DPKV_RING_STAGES=n); 0, the
// product's value, = automatic.
#ifndef PKV_RING_STAGES
#define PKV_RING_STAGES 0
#endif
static constexpr int stages_override()
{
    return PKV_RING_STAGES < 0 ? 0 : (PKV_RING_STAGES > 16 ? 16 : PKV_RING_STAGES);
}

// Most paged blocks the key range of a length-<=L sequence can touch.
static int64_t max_range_blocks(int P, int64_t L, int window)
{
    if (L <= 0)
        return 0;
    const int64_t keys = window > 0 ? (L < window + 1 ? L : (int64_t)window + 1) : L;
    const int64_t whole = (L + P - 1) / P;
    const int64_t span = (keys + P - 2) / P + 1;
    return whole < span ? whole : span;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

PKV_API const char *pkv_last_error(void) { return t_last_error.c_str(); }

PKV_API int32_t pkv_last_launch_count(void) { return t_launches; }

PKV_API int pkv_device_status(int32_t clear)
{
    unsigned int w = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&w, g_error_word, sizeof w);
    if (e != cudaSuccess)
        return fail(PKV_E_DRIVER, "reading the device error word: %s", cudaGetErrorString(e));
    if (clear) {
        unsigned int z = 0;
        e = cudaMemcpyToSymbol(g_error_word, &z, sizeof z);
        if (e != cudaSuccess)
            return fail(PKV_E_DRIVER, "clearing the device error word: %s", cudaGetErrorString(e));
    }
    return static_cast<int>(w);
}

PKV_API int pkv_check_bounded_wait(uint64_t limit_ns, int32_t spin, int32_t *out,
                                   int32_t threads, void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (!out || !aligned(out, 4))
        return fail(PKV_E_NULL, "out is NULL or misaligned");
    if (threads < 1 || threads > 1024)
        return fail(PKV_E_ARG, "threads %d", threads);
    if (limit_ns < 1000 || limit_ns > 2000000000ull)
        return fail(PKV_E_ARG, "limit_ns must be in [1 us, 2 s]");
    unsigned int *err = error_word_ptr();
    if (!err)
        return fail(PKV_E_DRIVER, "cannot resolve the device error word");
    cudaError_t e = launch_bounded_wait(limit_ns, spin, out, threads, err,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "bounded-wait check launch");
    return PKV_OK;
}

PKV_API int32_t paged_decode_uses_tensor_cores(const pkv_pool *pool, int32_t num_q_heads)
{
    t_last_error.clear();
    t_launches = 0;
    if (int rc = check_pool(pool))
        return rc;
    if (num_q_heads <= 0 || num_q_heads % pool->num_kv_heads)
        return fail(PKV_E_SHAPE, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    num_q_heads, pool->num_kv_heads);
    return use_tc(pool, num_q_heads / pool->num_kv_heads) ? 1 : 0;
}

PKV_API int paged_kv_append(const void *k, const void *v, const int64_t *slot_mapping,
                            int32_t num_tokens, const pkv_pool *pool, void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (int rc = check_pool(pool))
        return rc;
    if (num_tokens < 0)
        return fail(PKV_E_ARG, "num_tokens < 0");
    if (num_tokens == 0)
        return PKV_OK;
    const bool alias = pool->v == nullptr || pool->v == pool->k;
    if (!k || !slot_mapping || (!alias && !v))
        return fail(PKV_E_NULL, "k, v or slot_mapping is NULL");
    if (!aligned(k, 16) || (!alias && !aligned(v, 16)) || !aligned(slot_mapping, 8))
        return fail(PKV_E_ALIGN, "k/v must be 16-byte and slot_mapping 8-byte aligned");
    AppendParams p{};
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(alias ? k : v);
    p.slot_mapping = slot_mapping;
    p.pool_k = pool->k;
    p.pool_v = alias ? pool->k : pool->v;
    p.k_scale = pool->k_scale;
    p.v_scale = alias ? pool->k_scale : pool->v_scale;
    p.num_tokens = num_tokens;
    p.row = pool->num_kv_heads * pool->head_dim;
    p.head_dim = pool->head_dim;
    p.num_slots = (int64_t)pool->num_blocks * pool->block_size;
    p.scale_mode = pool->scale_mode;
    p.alias = alias;
    p.err = error_word_ptr();
    if (!p.err)
        return fail(PKV_E_DRIVER, "cannot resolve the device error word");
    cudaError_t e = launch_append(p, pool->dtype == PKV_INT8, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "append launch");
    return PKV_OK;
}

PKV_API int paged_rope_cos_sin_table(const double *theta, int32_t rotary_pairs,
                                     int64_t num_positions, float *table, void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (rotary_pairs < 0 || num_positions < 0)
        return fail(PKV_E_ARG, "rotary_pairs or num_positions < 0");
    if (rotary_pairs == 0 || num_positions == 0)
        return PKV_OK;
    if (!theta || !table)
        return fail(PKV_E_NULL, "theta or table is NULL");
    if (!aligned(theta, 8) || !aligned(table, 8))
        return fail(PKV_E_ALIGN, "theta and table must be 8-byte aligned");
    cudaError_t e = launch_rope_table(theta, rotary_pairs, num_positions, table,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "RoPE table launch");
    return PKV_OK;
}

}  // extern "C"

// RoPE fused with the append at positions[t], or (positions NULL, the decode
// step) at seq_lens[t] - 1.  Host checks, then one launch.
static int append_rope_impl(const void *q, void *q_out, int32_t num_q_heads, const void *k,
                            const void *v, const int64_t *positions, const int32_t *seq_lens,
                            const int64_t *slot_mapping, int32_t num_tokens, const float *table,
                            int64_t num_positions, int32_t rotary_pairs, int32_t layout,
                            const pkv_pool *pool, void *stream)
{
    if (int rc = check_pool(pool))
        return rc;
    if (num_tokens < 0)
        return fail(PKV_E_ARG, "num_tokens < 0");
    if (rotary_pairs < 0 || 2 * rotary_pairs > pool->head_dim)
        return fail(PKV_E_ARG, "rotary_pairs %d outside [0, head_dim / 2]", rotary_pairs);
    if (layout != PKV_ROPE_HALVES && layout != PKV_ROPE_INTERLEAVED)
        return fail(PKV_E_ARG, "unknown RoPE layout %d", layout);
    if (num_positions < 0)
        return fail(PKV_E_ARG, "num_positions < 0");
    if (q && num_q_heads <= 0)
        return fail(PKV_E_ARG, "num_q_heads <= 0");
    if (num_tokens == 0)
        return PKV_OK;
    const bool alias = pool->v == nullptr || pool->v == pool->k;
    if (!k || !slot_mapping || !(positions || seq_lens) || (!alias && !v) || (q && !q_out) ||
        (rotary_pairs > 0 && num_positions > 0 && !table))
        return fail(PKV_E_NULL, "k, v, q_out, positions, slot_mapping or table is NULL");
    if (!aligned(k, 16) || (!alias && !aligned(v, 16)) || !aligned(slot_mapping, 8) ||
        (positions && !aligned(positions, 8)) || (q && (!aligned(q, 16) || !aligned(q_out, 16))) ||
        (table && !aligned(table, 8)))
        return fail(PKV_E_ALIGN, "q/q_out/k/v must be 16-byte, positions/slot_mapping/table "
                                 "8-byte aligned");
    AppendParams p{};
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(alias ? k : v);
    p.slot_mapping = slot_mapping;
    p.pool_k = pool->k;
    p.pool_v = alias ? pool->k : pool->v;
    p.k_scale = pool->k_scale;
    p.v_scale = alias ? pool->k_scale : pool->v_scale;
    p.num_tokens = num_tokens;
    p.row = pool->num_kv_heads * pool->head_dim;
    p.head_dim = pool->head_dim;
    p.num_slots = (int64_t)pool->num_blocks * pool->block_size;
    p.scale_mode = pool->scale_mode;
    p.alias = alias;
    p.err = error_word_ptr();
    if (!p.err)
        return fail(PKV_E_DRIVER, "cannot resolve the device error word");
    if (append_rope_smem_bytes(p.row, rotary_pairs) > 227 * 1024)
        return fail(PKV_E_SHAPE, "a token's K row (%d elements) is too large", p.row);
    RopeParams r{};
    r.q = static_cast<const uint16_t *>(q);
    r.q_out = static_cast<uint16_t *>(q_out);
    r.positions = positions;
    r.seq_lens = seq_lens;
    r.table = reinterpret_cast<const float2 *>(table);
    r.num_positions = num_positions;
    r.num_q_heads = q ? num_q_heads : 0;
    r.pairs = rotary_pairs;
    r.layout = layout;
    cudaError_t e = launch_append_rope(p, r, pool->dtype == PKV_INT8,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "append (RoPE) launch");
    return PKV_OK;
}

extern "C" {

PKV_API int paged_kv_append_rope(const void *q, void *q_out, int32_t num_q_heads, const void *k,
                                 const void *v, const int64_t *positions,
                                 const int64_t *slot_mapping, int32_t num_tokens,
                                 const float *table, int64_t num_positions,
                                 int32_t rotary_pairs, int32_t layout, const pkv_pool *pool,
                                 void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (!positions && num_tokens > 0)
        return fail(PKV_E_NULL, "positions is NULL");
    return append_rope_impl(q, q_out, num_q_heads, k, v, positions, nullptr, slot_mapping,
                            num_tokens, table, num_positions, rotary_pairs, layout, pool, stream);
}

PKV_API int paged_kv_slot_mapping(const pkv_pool *pool, const int32_t *block_table,
                                  int32_t max_blocks_per_seq, const int32_t *seq_ids,
                                  const int64_t *positions, int32_t num_tokens,
                                  int64_t *slot_mapping, void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (int rc = check_pool(pool))
        return rc;
    if (num_tokens < 0 || max_blocks_per_seq <= 0)
        return fail(PKV_E_ARG, "num_tokens < 0 or max_blocks_per_seq <= 0");
    if (num_tokens == 0)
        return PKV_OK;
    if (!block_table || !positions || !slot_mapping)
        return fail(PKV_E_NULL, "block_table, positions or slot_mapping is NULL");
    if (!aligned(block_table, 4) || !aligned(positions, 8) || !aligned(slot_mapping, 8) ||
        (seq_ids && !aligned(seq_ids, 4)))
        return fail(PKV_E_ALIGN, "misaligned block_table, seq_ids, positions or slot_mapping");
    if (pool->ring_blocks > max_blocks_per_seq)
        return fail(PKV_E_SHAPE, "block table rows (%d) shorter than the ring (%d blocks)",
                    max_blocks_per_seq, pool->ring_blocks);
    unsigned int *err = error_word_ptr();
    if (!err)
        return fail(PKV_E_DRIVER, "cannot resolve the device error word");
    cudaError_t e = launch_slot_mapping(block_table, max_blocks_per_seq, pool->ring_blocks,
                                        pool->num_blocks, seq_ids, positions, num_tokens,
                                        slot_mapping, err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "slot mapping launch");
    return PKV_OK;
}

PKV_API int32_t paged_decode_num_splits(int32_t block_size, int32_t max_seq_len, int32_t window,
                                        int32_t split_tokens)
{
    if (block_size <= 0 || split_tokens <= 0 || split_tokens % block_size)
        return 1;
    const int64_t nblk = max_range_blocks(block_size, max_seq_len, window);
    const int64_t sb = split_tokens / block_size;
    const int64_t ns = (nblk + sb - 1) / sb;
    return ns < 1 ? 1 : static_cast<int32_t>(ns);
}

PKV_API int32_t paged_decode_split_tokens(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t block_size, int32_t max_seq_len, int32_t window,
                                          int32_t split_tokens)
{
    if (block_size <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || batch < 0)
        return fail(PKV_E_ARG, "bad sizes");
    if (split_tokens >= 0) {
        if (split_tokens % block_size)
            return fail(PKV_E_ARG, "split_tokens %d is not a multiple of block_size", split_tokens);
        return split_tokens;
    }
    if (split_tokens != PKV_SPLIT_AUTO)
        return fail(PKV_E_ARG, "split_tokens %d", split_tokens);
    // Auto: split each sequence's key range into pieces of a fixed length --
    // 4096 keys for GQA groups of 8 or more (tensor-core kernel, one CTA per
    // SM), 2048 otherwise -- and run a single pass (no combine) when the
    // longest range fits in one piece.  Sequences shorter than a piece take
    // one CTA whatever their neighbours' lengths, which keeps ragged batches
    // balanced without knowing the lengths on the host.
    const int group = num_q_heads / num_kv_heads;
    const int64_t piece = group >= 8 ? 4096 : 2048;
    const int64_t nblk = max_range_blocks(block_size, max_seq_len, window);
    if (nblk * block_size <= piece)
        return 0;
    return static_cast<int32_t>(piece);
}

PKV_API size_t paged_decode_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_dim,
                                            int32_t block_size, int32_t max_seq_len,
                                            int32_t window, int32_t split_tokens)
{
    const int32_t st = paged_decode_split_tokens(batch, num_q_heads, num_kv_heads, block_size,
                                                 max_seq_len, window, split_tokens);
    size_t need = 0;
    if (st > 0) {
        const size_t ns = paged_decode_num_splits(block_size, max_seq_len, window, st);
        const size_t rows = (size_t)batch * num_q_heads * ns;
        const size_t lse = (rows * sizeof(float) + 255) / 256 * 256;
        need = lse + rows * head_dim * sizeof(float);
    }
    const size_t tc = paged_decode_partial_workspace_bytes(batch, num_q_heads, num_kv_heads,
                                                           head_dim);
    // a single pass on CUDA cores orders the sequences longest first in here
    const size_t order = batch > 0 ? (2 * sizeof(int32_t) * (size_t)batch + 255) / 256 * 256 : 0;
    need = need > tc ? need : tc;
    return need > order ? need : order;
}

PKV_API size_t paged_decode_partial_workspace_bytes(int32_t batch, int32_t num_q_heads,
                                                    int32_t num_kv_heads, int32_t head_dim)
{
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
        return 0;
    if (!tc_shape(num_q_heads / num_kv_heads, head_dim))
        return 0;
    return decode_tc_scratch_bytes(batch, head_dim);
}

static int check_decode_args(const void *q, const pkv_pool *pool, const int32_t *block_table,
                             int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                             int32_t num_q_heads, int32_t max_seq_len, int32_t window, void *out,
                             int32_t out_dtype)
{
    if (int rc = check_pool(pool))
        return rc;
    if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0)
        return fail(PKV_E_SHAPE, "batch, num_q_heads, max_blocks_per_seq or max_seq_len invalid");
    if (num_q_heads % pool->num_kv_heads)
        return fail(PKV_E_SHAPE, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    num_q_heads, pool->num_kv_heads);
    if (batch > 65535)
        return fail(PKV_E_UNSUPPORTED, "batch > 65535");
    if (window < 0)
        return fail(PKV_E_ARG, "window < 0");
    if (pool->ring_blocks > 0) {
        // a ring holds the last W = ring_blocks * block_size positions: the
        // inclusive window's w + 1 keys must fit
        if (window == 0)
            return fail(PKV_E_ARG, "a ring layout needs a sliding window (window > 0)");
        if ((int64_t)pool->ring_blocks * pool->block_size < (int64_t)window + 1)
            return fail(PKV_E_SHAPE, "ring of %d slots is shorter than the window's %d keys",
                        pool->ring_blocks * pool->block_size, window + 1);
        if (max_blocks_per_seq < pool->ring_blocks)
            return fail(PKV_E_SHAPE, "block table rows (%d) shorter than the ring (%d blocks)",
                        max_blocks_per_seq, pool->ring_blocks);
    } else if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * pool->block_size) {
        return fail(PKV_E_SHAPE, "max_seq_len exceeds max_blocks_per_seq * block_size");
    }
    if (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_F32)
        return fail(PKV_E_ARG, "out_dtype %d", out_dtype);
    if (!q || !block_table || !seq_lens || !out)
        return fail(PKV_E_NULL, "q, block_table, seq_lens or out is NULL");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return fail(PKV_E_ALIGN, "q/out must be 16-byte aligned");
    return PKV_OK;
}

static int run_decode(const void *q, const pkv_pool *pool, const int32_t *block_table,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                      int32_t num_q_heads, int32_t max_seq_len, int32_t window,
                      float softmax_scale, int32_t split_tokens, float *part_lse, float *part_o,
                      int32_t num_splits, void *out, int32_t out_dtype, void *workspace,
                      size_t workspace_bytes, cudaStream_t s)
{
    const bool alias = pool->v == nullptr || pool->v == pool->k;
    const int group = num_q_heads / pool->num_kv_heads;
    const bool tc = use_tc(pool, group);
    if (tc) {
        const size_t need = decode_tc_scratch_bytes(batch, pool->head_dim);
        if (!workspace || workspace_bytes < need)
            return fail(PKV_E_WORKSPACE,
                        "the tensor-core kernel needs a workspace of %zu bytes, %zu given", need,
                        workspace ? workspace_bytes : (size_t)0);
        if (!aligned(workspace, 256))
            return fail(PKV_E_ALIGN, "workspace must be 256-byte aligned");
    }
    auto encode = tc ? encode_pool_map_tc : encode_pool_map;
    CUtensorMap tmk, tmv;
    if (int rc = encode(&tmk, pool->k, *pool))
        return rc;
    if (alias)
        tmv = tmk;
    else if (int rc = encode(&tmv, pool->v, *pool))
        return rc;
    const int gt = tc ? group : decode_group_tile(group);
    DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.k_scale = pool->k_scale;
    p.v_scale = alias ? pool->k_scale : pool->v_scale;
    p.part_lse = part_lse;
    p.part_o = part_o;
    p.out = out;
    p.max_blocks = max_blocks_per_seq;
    p.ring_blocks = pool->ring_blocks;
    p.scale_mode = pool->scale_mode;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = pool->num_kv_heads;
    p.group = group;
    p.head_chunks = tc ? 1 : (group + gt - 1) / gt;
    p.num_blocks = pool->num_blocks;
    p.window = window;
    p.max_seq_len = max_seq_len;
    p.split_blocks = split_tokens > 0 ? split_tokens / pool->block_size : 0;
    p.num_splits = split_tokens > 0 ? num_splits : 1;
    p.alias = alias;
    p.out_f32 = out_dtype == PKV_OUT_F32;
    // Ring depth: the most CTAs per SM, then the deepest ring that keeps
    // them (decode_ring_stages); a tuning build's PKV_RING_STAGES overrides
    // it within the opt-in shared-memory limit of one CTA.
    {
        const int i8 = pool->dtype == PKV_INT8;
        const int pt = i8 && pool->scale_mode == PKV_SCALE_PER_TOKEN;
        int ns = stages_override();
        if (ns) {
            while (ns > 2 && decode_smem_bytes(pool->head_dim, i8, alias, pt, gt, ns) > 227u * 1024u)
                --ns;
        } else if (!tc) {
            ns = decode_ring_stages(pool->head_dim, i8, alias, pt, gt);
        }
        p.num_stages = ns < 2 ? 2 : ns;
    }
    p.qk_scale_log2 = softmax_scale * LOG2E;
    p.head_dim = pool->head_dim;
    // a single pass on CUDA cores may order the sequences longest first in
    // the caller's workspace
    if (!tc && split_tokens == 0 && workspace && aligned(workspace, 8) &&
        workspace_bytes >= 2 * sizeof(int32_t) * static_cast<size_t>(batch))
        p.order_ws = static_cast<int32_t *>(workspace);
    p.err = error_word_ptr();
    if (!p.err)
        return fail(PKV_E_DRIVER, "cannot resolve the device error word");
    if ((int64_t)p.num_kv_heads * p.head_chunks > 65535)
        return fail(PKV_E_UNSUPPORTED, "too many kv heads");
    if (tc) {
        // ring of 32 KB units: 6 by default (one CTA per SM), PKV_RING_STAGES overrides
        int nu = stages_override() ? stages_override() : 6;
        while (nu > 2 && decode_tc_smem_bytes(nu) > 227u * 1024u)
            --nu;
        p.num_stages = nu < 6 ? nu : 6;  // one producer warp per ring unit
        CUtensorMap tmq;
        if (int rc = encode_q_map(&tmq, q, batch * num_q_heads, pool->head_dim))
            return rc;
        decode_tc_bind_scratch(p, workspace, batch);
        cudaError_t e = launch_decode_tc(p, tmk, tmv, tmq, pool->head_dim, s);
        if (e != cudaSuccess)
            return cuda_fail(e, "tensor-core decode launch");
        return PKV_OK;
    }
    cudaError_t e = launch_decode(p, tmk, tmv, pool->head_dim, pool->dtype == PKV_INT8, gt, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "decode launch");
    return PKV_OK;
}

PKV_API int paged_prefill_attention(const void *q, const int32_t *q_start, int32_t total_q,
                                    int32_t max_q_len, const pkv_pool *pool,
                                    const int32_t *block_table, int32_t max_blocks_per_seq,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t max_seq_len, int32_t window, float softmax_scale,
                                    void *out, int32_t out_dtype, void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (int rc = check_decode_args(q, pool, block_table, max_blocks_per_seq, seq_lens, batch,
                                   num_q_heads, max_seq_len, window, out, out_dtype))
        return rc;
    if (!q_start)
        return fail(PKV_E_NULL, "q_start is NULL");
    if (!aligned(q_start, 4))
        return fail(PKV_E_ALIGN, "q_start must be 4-byte aligned");
    if (total_q < 0 || max_q_len < 0)
        return fail(PKV_E_SHAPE, "total_q or max_q_len < 0");
    if (pool->dtype != PKV_BF16)
        return fail(PKV_E_UNSUPPORTED, "chunk attention needs a bf16 pool (tensor-core operands)");
    // a ring must hold the first query's window and the whole chunk at once
    if (pool->ring_blocks > 0 &&
        (int64_t)pool->ring_blocks * pool->block_size < (int64_t)window + max_q_len)
        return fail(PKV_E_SHAPE, "ring of %d slots cannot hold a %d-token chunk and its window %d",
                    pool->ring_blocks * pool->block_size, max_q_len, window);
    const int group = num_q_heads / pool->num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16)
        return fail(PKV_E_UNSUPPORTED, "chunk attention: %d query heads per kv head (1..16, "
                    "a power of two)", group);
    if (pool->num_kv_heads > 65535)
        return fail(PKV_E_UNSUPPORTED, "too many kv heads");
    if (batch == 0 || total_q == 0 || max_q_len == 0)
        return PKV_OK;
    if ((int64_t)max_q_len * group > (int64_t)128 * 65535)
        return fail(PKV_E_UNSUPPORTED, "max_q_len too large");
    const bool alias = pool->v == nullptr || pool->v == pool->k;
    CUtensorMap tmk, tmv, tmq;
    if (int rc = encode_pool_map_tc(&tmk, pool->k, *pool))
        return rc;
    if (alias)
        tmv = tmk;
    else if (int rc = encode_pool_map_tc(&tmv, pool->v, *pool))
        return rc;
    if (int rc = encode_chunk_q_map(&tmq, q, total_q, num_q_heads, pool->head_dim, group))
        return rc;
    PrefillParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.q_start = q_start;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.err = error_word_ptr();
    if (!p.err)
        return fail(PKV_E_DRIVER, "cannot resolve the device error word");
    p.max_blocks = max_blocks_per_seq;
    p.ring_blocks = pool->ring_blocks;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = pool->num_kv_heads;
    p.group = group;
    p.num_blocks = pool->num_blocks;
    p.window = window;
    p.max_seq_len = max_seq_len;
    p.max_q_len = max_q_len;
    p.alias = alias;
    p.out_f32 = out_dtype == PKV_OUT_F32;
    p.num_buffers = prefill_num_buffers(pool->head_dim, alias);
    p.qk_scale_log2 = softmax_scale * LOG2E;
    cudaError_t e = launch_prefill(p, tmk, tmv, tmq, pool->head_dim,
                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "chunk attention launch");
    return PKV_OK;
}

PKV_API int paged_decode_split_partial(const void *q, const pkv_pool *pool,
                                       const int32_t *block_table, int32_t max_blocks_per_seq,
                                       const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                       int32_t max_seq_len, int32_t window, float softmax_scale,
                                       int32_t split_tokens, float *partial_lse, float *partial_o,
                                       int32_t num_splits, void *workspace,
                                       size_t workspace_bytes, void *out, int32_t out_dtype,
                                       void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (int rc = check_decode_args(q, pool, block_table, max_blocks_per_seq, seq_lens, batch,
                                   num_q_heads, max_seq_len, window, out, out_dtype))
        return rc;
    if (split_tokens <= 0 || split_tokens % pool->block_size)
        return fail(PKV_E_ARG, "split_tokens must be a positive multiple of block_size");
    const int32_t need = paged_decode_num_splits(pool->block_size, max_seq_len, window, split_tokens);
    if (num_splits < need)
        return fail(PKV_E_WORKSPACE, "num_splits %d < %d needed", num_splits, need);
    if (num_splits > 1024)
        return fail(PKV_E_UNSUPPORTED, "more than 1024 splits");
    if (!partial_lse || !partial_o)
        return fail(PKV_E_NULL, "partial buffers are NULL");
    if (!aligned(partial_lse, 16) || !aligned(partial_o, 16))
        return fail(PKV_E_ALIGN, "partial_lse and partial_o must be 16-byte aligned");
    if (batch == 0)
        return PKV_OK;
    return run_decode(q, pool, block_table, max_blocks_per_seq, seq_lens, batch, num_q_heads,
                      max_seq_len, window, softmax_scale, split_tokens, partial_lse, partial_o,
                      num_splits, out, out_dtype, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

PKV_API int paged_decode_lse_combine(const float *partial_lse, const float *partial_o,
                                     const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                     int32_t head_dim, int32_t block_size, int32_t window,
                                     int32_t split_tokens, int32_t num_splits, void *out,
                                     int32_t out_dtype, void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (!partial_lse || !partial_o || !seq_lens || !out)
        return fail(PKV_E_NULL, "NULL argument");
    if (block_size != kBlock)
        return fail(PKV_E_UNSUPPORTED, "block_size %d", block_size);
    if (batch < 0 || num_q_heads <= 0 || head_dim <= 0 || num_splits <= 0 || num_splits > 1024 ||
        batch > 65535)
        return fail(PKV_E_SHAPE, "bad sizes");
    if (split_tokens <= 0 || split_tokens % block_size)
        return fail(PKV_E_ARG, "split_tokens must be a positive multiple of block_size");
    if (window < 0 || (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_F32))
        return fail(PKV_E_ARG, "window or out_dtype");
    if (batch == 0)
        return PKV_OK;
    CombineParams p{};
    p.part_lse = partial_lse;
    p.part_o = partial_o;
    p.seq_lens = seq_lens;
    p.out = out;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.head_dim = head_dim;
    p.window = window;
    p.split_blocks = split_tokens / block_size;
    p.num_splits = num_splits;
    p.out_f32 = out_dtype == PKV_OUT_F32;
    cudaError_t e = launch_combine(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "combine launch");
    return PKV_OK;
}

PKV_API int paged_decode_attention(const void *q, const pkv_pool *pool, const int32_t *block_table,
                                   int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                   int32_t batch, int32_t num_q_heads, int32_t max_seq_len,
                                   int32_t window, float softmax_scale, int32_t split_tokens,
                                   void *workspace, size_t workspace_bytes, void *out,
                                   int32_t out_dtype, void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (int rc = check_decode_args(q, pool, block_table, max_blocks_per_seq, seq_lens, batch,
                                   num_q_heads, max_seq_len, window, out, out_dtype))
        return rc;
    const int32_t st = paged_decode_split_tokens(batch, num_q_heads, pool->num_kv_heads,
                                                 pool->block_size, max_seq_len, window,
                                                 split_tokens);
    if (st < 0)
        return st;
    if (batch == 0)
        return PKV_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The tensor-core kernel balances the key ranges across SMs itself
    // (stream-K) and writes the outputs without a split pass.
    if (st == 0 || use_tc(pool, num_q_heads / pool->num_kv_heads))
        return run_decode(q, pool, block_table, max_blocks_per_seq, seq_lens, batch, num_q_heads,
                          max_seq_len, window, softmax_scale, 0, nullptr, nullptr, 1, out,
                          out_dtype, workspace, workspace_bytes, s);
    const int32_t ns = paged_decode_num_splits(pool->block_size, max_seq_len, window, st);
    if (ns > 1024)
        return fail(PKV_E_UNSUPPORTED, "more than 1024 splits; use a longer split_tokens");
    const size_t need = paged_decode_workspace_bytes(batch, num_q_heads, pool->num_kv_heads,
                                                     pool->head_dim, pool->block_size,
                                                     max_seq_len, window, st);
    if (!workspace || workspace_bytes < need)
        return fail(PKV_E_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace_bytes);
    if (!aligned(workspace, 256))
        return fail(PKV_E_ALIGN, "workspace must be 256-byte aligned");
    const size_t rows = (size_t)batch * num_q_heads * ns;
    float *lse = static_cast<float *>(workspace);
    float *po = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                          (rows * sizeof(float) + 255) / 256 * 256);
    if (int rc = run_decode(q, pool, block_table, max_blocks_per_seq, seq_lens, batch, num_q_heads,
                            max_seq_len, window, softmax_scale, st, lse, po, ns, out, out_dtype,
                            nullptr, 0, s))
        return rc;
    CombineParams c{};
    c.part_lse = lse;
    c.part_o = po;
    c.seq_lens = seq_lens;
    c.out = out;
    c.batch = batch;
    c.num_q_heads = num_q_heads;
    c.head_dim = pool->head_dim;
    c.window = window;
    c.split_blocks = st / pool->block_size;
    c.num_splits = ns;
    c.out_f32 = out_dtype == PKV_OUT_F32;
    cudaError_t e = launch_combine(c, s);
    if (e != cudaSuccess)
        return cuda_fail(e, "combine launch");
    return PKV_OK;
}

PKV_API size_t paged_decode_step_workspace_bytes(const pkv_layer *layers, int32_t num_layers,
                                                 int32_t batch, int32_t num_q_heads,
                                                 int32_t max_seq_len, int32_t split_tokens)
{
    size_t need = 0;
    if (!layers || num_layers <= 0)
        return 0;
    for (int32_t l = 0; l < num_layers; ++l) {
        const pkv_pool &pl = layers[l].pool;
        const size_t n = paged_decode_workspace_bytes(batch, num_q_heads, pl.num_kv_heads,
                                                      pl.head_dim, pl.block_size, max_seq_len,
                                                      layers[l].window, split_tokens);
        need = n > need ? n : need;
    }
    return need;
}

PKV_API int paged_decode_step(const pkv_layer *layers, int32_t num_layers,
                              const int64_t *slot_mapping, const int32_t *block_table,
                              int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                              int32_t num_q_heads, int32_t max_seq_len, int32_t split_tokens,
                              void *workspace, size_t workspace_bytes, int32_t out_dtype,
                              void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (!layers || num_layers <= 0)
        return fail(PKV_E_ARG, "no layers");
    if (!slot_mapping)
        return fail(PKV_E_NULL, "slot_mapping is NULL");
    if (!aligned(slot_mapping, 8))
        return fail(PKV_E_ALIGN, "slot_mapping must be 8-byte aligned");
    // validate every layer before anything is enqueued
    for (int32_t l = 0; l < num_layers; ++l) {
        const pkv_layer &L = layers[l];
        if (int rc = check_decode_args(L.q, &L.pool, block_table, max_blocks_per_seq, seq_lens,
                                       batch, num_q_heads, max_seq_len, L.window, L.out,
                                       out_dtype))
            return fail(rc, "layer %d: %s", l, std::string(t_last_error).c_str());
        const bool alias = L.pool.v == nullptr || L.pool.v == L.pool.k;
        if (!L.k_new || (!alias && !L.v_new))
            return fail(PKV_E_NULL, "layer %d: k_new or v_new is NULL", l);
        if (!aligned(L.k_new, 16) || (!alias && !aligned(L.v_new, 16)))
            return fail(PKV_E_ALIGN, "layer %d: k_new/v_new must be 16-byte aligned", l);
        if (L.rope_table) {
            if (L.rope_pairs < 0 || 2 * L.rope_pairs > L.pool.head_dim || L.rope_num_positions < 0 ||
                (L.rope_layout != PKV_ROPE_HALVES && L.rope_layout != PKV_ROPE_INTERLEAVED))
                return fail(PKV_E_ARG, "layer %d: RoPE pairs, positions or layout out of range", l);
            if (!L.q_rotated)
                return fail(PKV_E_NULL, "layer %d: q_rotated is NULL", l);
            if (!aligned(L.q_rotated, 16) || !aligned(L.rope_table, 8))
                return fail(PKV_E_ALIGN, "layer %d: q_rotated (16 B) or rope_table (8 B) misaligned",
                            l);
        }
        const int32_t st = paged_decode_split_tokens(batch, num_q_heads, L.pool.num_kv_heads,
                                                     L.pool.block_size, max_seq_len, L.window,
                                                     split_tokens);
        if (st < 0)
            return fail(st, "layer %d: %s", l, std::string(t_last_error).c_str());
        const bool needs_ws = use_tc(&L.pool, num_q_heads / L.pool.num_kv_heads) || st > 0;
        const size_t need = paged_decode_workspace_bytes(batch, num_q_heads, L.pool.num_kv_heads,
                                                         L.pool.head_dim, L.pool.block_size,
                                                         max_seq_len, L.window, st);
        if (needs_ws && batch > 0 && (!workspace || workspace_bytes < need))
            return fail(PKV_E_WORKSPACE, "layer %d: workspace of %zu bytes needed, %zu given", l,
                        need, workspace ? workspace_bytes : (size_t)0);
        if (needs_ws && workspace && !aligned(workspace, 256))
            return fail(PKV_E_ALIGN, "workspace must be 256-byte aligned");
    }
    int launches = 0;
    for (int32_t l = 0; l < num_layers; ++l) {
        const pkv_layer &L = layers[l];
        int rc;
        if (L.rope_table) {
            t_launches = 0;
            rc = append_rope_impl(L.q, L.q_rotated, num_q_heads, L.k_new, L.v_new, nullptr,
                                  seq_lens, slot_mapping, batch, L.rope_table,
                                  L.rope_num_positions, L.rope_pairs, L.rope_layout, &L.pool,
                                  stream);
        } else {
            rc = paged_kv_append(L.k_new, L.v_new, slot_mapping, batch, &L.pool, stream);
        }
        launches += t_launches;
        if (rc == PKV_OK) {
            rc = paged_decode_attention(L.rope_table ? L.q_rotated : L.q, &L.pool, block_table,
                                        max_blocks_per_seq, seq_lens,
                                        batch, num_q_heads, max_seq_len, L.window,
                                        L.softmax_scale, split_tokens, workspace, workspace_bytes,
                                        L.out, out_dtype, stream);
            launches += t_launches;
        }
        if (rc != PKV_OK) {
            t_launches = launches;
            return fail(rc, "layer %d: %s", l, std::string(t_last_error).c_str());
        }
    }
    t_launches = launches;
    return PKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory.
//
// paged_decode_attention needs a caller-provided workspace whenever it splits
// the key range.  Some callers have no way to provide one: a plugin whose
// host framework hands it only its input and output buffers, an engine that
// reserved all of HBM up front for its KV pool, or a latency-critical loop in
// which cudaMalloc/cudaFree would synchronise the device.  For them the split
// partials live in the fixed array below, which every device that loads this
// library holds until the process exits.
namespace pkv {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  The host-side
// name g_static_scratch is only a stand-in; the address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static void *static_scratch_ptr()
{
    static std::mutex mu;
    static void *ptrs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        fail(PKV_E_DRIVER, "cannot query the current device");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            fail(PKV_E_DRIVER, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
            return nullptr;
        }
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

}  // namespace pkv

extern "C" PKV_API int paged_decode_attention_noalloc(
    const void *q, const pkv_pool *pool, const int32_t *block_table, int32_t max_blocks_per_seq,
    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_seq_len,
    int32_t window, float softmax_scale, int32_t split_tokens, void *out, int32_t out_dtype,
    void *stream)
{
    t_last_error.clear();
    t_launches = 0;
    if (int rc = check_decode_args(q, pool, block_table, max_blocks_per_seq, seq_lens, batch,
                                   num_q_heads, max_seq_len, window, out, out_dtype))
        return rc;
    const int32_t st = paged_decode_split_tokens(batch, num_q_heads, pool->num_kv_heads,
                                                 pool->block_size, max_seq_len, window,
                                                 split_tokens);
    if (st < 0)
        return st;
    // The scratch paged_decode_attention itself needs on the path it takes:
    // the tensor-core kernel's scratch (it balances the key ranges itself
    // and ignores the split length), the split partials on the CUDA-core
    // kernel, or the optional length order of a CUDA-core single pass.
    size_t need;
    if (use_tc(pool, num_q_heads / pool->num_kv_heads))
        need = decode_tc_scratch_bytes(batch, pool->head_dim);
    else if (st > 0)
        need = paged_decode_workspace_bytes(batch, num_q_heads, pool->num_kv_heads,
                                            pool->head_dim, pool->block_size, max_seq_len,
                                            window, st);
    else
        need = batch > 0 ? (2 * sizeof(int32_t) * (size_t)batch + 255) / 256 * 256 : 0;
    if (need > kStaticScratchBytes)
        return fail(PKV_E_WORKSPACE,
                    "these sizes need %zu bytes of scratch but the static scratch holds %zu "
                    "(PKV_STATIC_SCRATCH_BYTES); use a longer split_tokens, a smaller batch, "
                    "or paged_decode_attention with a workspace",
                    need, kStaticScratchBytes);
    void *ws = nullptr;
    if (need > 0 && !(ws = static_scratch_ptr()))
        return PKV_E_DRIVER;
    // The whole array is offered: on each path paged_decode_attention
    // checks the workspace against the same figure as `need` above.
    return paged_decode_attention(q, pool, block_table, max_blocks_per_seq, seq_lens, batch,
                                  num_q_heads, max_seq_len, window, softmax_scale, st, ws,
                                  need > 0 ? kStaticScratchBytes : 0, out, out_dtype, stream);
}
