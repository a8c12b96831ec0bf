/*
 * pkv_oracle.c -- CPU oracle for paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; it exists so that tests, the smoke check and the CPU
 * baseline of the benchmark can compare the CUDA kernels against a plain,
 * slow, obviously correct definition.  It shares no source, header, table or
 * constant with the CUDA code.
 *
 * Sources followed (page title, section):
 *   [CS336-L10]  "CS336 · 第 10 课" (inference lecture guide): the decode
 *                attention formula in the KV-cache section, a =
 *                softmax(Q_new [K_1..K_n;K_new]^T / sqrt(d_h)), y = a [V..];
 *                and the int8 quantisation section, scale = max|x|/127,
 *                x_q = round(x/scale).
 *   [Lab5]       "实验五：Gemma4 端到端推理优化" (hpc101 Lab5-Gemma4):
 *                section 滑动窗口注意力 (mask M: lower-triangular on global
 *                layers, band [i-w, i] on sliding layers); section 分组查询注意力
 *                (query heads share a KV head by repetition); section
 *                Paged Attention (block pool + block table; first correct
 *                version gathers the blocks in logical order and reuses
 *                dense attention).
 *   [tiniestgpt] "推理优化与 AI Infra" notes: section 2 (pool layout
 *                k_cache[block][slot][head][dim], block_table[seq][i]) and
 *                section 5 (KV int8, per_token or per_head scales,
 *                dequantise after the gather).
 *   RoPE         the pages name p-RoPE on global layers ([Lab5] model
 *                overview) without a formula; the rotation follows RoFormer
 *                (Su et al.) and p-RoPE (Barbero et al.), cited at
 *                oracle_rope below.
 *
 * Arithmetic: attention in fp64 throughout.  The quantiser is fp32 because
 * the stored scale is an fp32 number (one fp32 division for the scale, one
 * fp32 division per element, round-half-to-even).  The stored RoPE output is
 * bf16, so its rounding is taken in the precision the library states (fp32
 * table and fp32 fused multiply-adds); oracle_rope_exact is the fp64 form.
 *
 * Parity status of each function is stated beside it; all are pinned by the
 * CPU tests in tests/test_oracle_pins.py (RoPE: tests/test_rope_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Pool description used by the oracle only (its own struct, not the
 * library's).  Layout of k and v: [num_blocks][block_size][num_kv_heads]
 * [head_dim], elements bf16 bit patterns (uint16) or int8.  v == NULL means
 * K and V are one tensor (shared W_K = W_V on global layers, [Lab5] model
 * overview). */
typedef struct {
    void *k;
    void *v;
    float *k_scale; /* per-token: [num_blocks*block_size]; per-head: [num_kv_heads] */
    float *v_scale;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t is_int8;    /* 0: bf16 elements, 1: int8 elements */
    int32_t scale_mode; /* 0: none, 1: per token, 2: per kv head */
    int32_t ring_blocks; /* 0: paged (the table lists every logical block);
                          * > 0: ring of ring_blocks blocks per sequence */
} oracle_pool;

enum { OR_OK = 0, OR_E_ARG = -1, OR_E_BLOCK = -2, OR_E_SLOT = -3 };

/* bf16 bit pattern -> exact float: bf16 is the upper half of an fp32. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* Quantiser ([CS336-L10] quantisation: scale = max(abs(x))/127,            */
/* x_q = round(x/scale)).  Readings: round = IEEE round-half-to-even; the   */
/* result is saturated to [-127, 127] (a static per-head scale can be       */
/* exceeded); a zero scale quantises everything to 0; a quotient that is    */
/* not a number (a NaN input, or inf/inf under an infinite per-token scale) */
/* has no code and is stored as 0 (the pages are silent on non-finite x).   */
/* ------------------------------------------------------------------------ */
static int8_t quantize_one(float x, float scale)
{
    if (scale == 0.0f)
        return 0;
    float y = x / scale;     /* one IEEE fp32 division */
    if (isnan(y))
        return 0;
    float r = nearbyintf(y); /* default rounding mode: half to even */
    if (r > 127.0f)
        r = 127.0f;
    if (r < -127.0f)
        r = -127.0f;
    return (int8_t)r;
}

/* Per-token scale of one row of n bf16 values: max|x| / 127 in fp32. */
float oracle_per_token_scale(const uint16_t *x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(bf16_bits_to_float(x[i]));
        if (a > amax)
            amax = a;
    }
    return amax / 127.0f;
}

/* Quantise n bf16 values with the given scale. */
void oracle_quantize(const uint16_t *x, int64_t n, float scale, int8_t *q)
{
    for (int64_t i = 0; i < n; ++i)
        q[i] = quantize_one(bf16_bits_to_float(x[i]), scale);
}

/* ------------------------------------------------------------------------ */
/* Append: write token t's K and V rows ([num_kv_heads][head_dim], bf16)     */
/* into slot slot_mapping[t] of the pool, i.e. block slot/P, offset slot%P   */
/* ([tiniestgpt] section 2 layout; slot ids are the static step buffer of   */
/* section 8).  A negative slot is padding and is skipped.  int8 pools      */
/* quantise per token (scale written at index slot) or per head (scale read */
/* from the table).  With K and V as one tensor only k is written.           */
/* ------------------------------------------------------------------------ */
int oracle_append(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                  int32_t num_tokens, const oracle_pool *pool)
{
    const int64_t row = (int64_t)pool->num_kv_heads * pool->head_dim;
    const int64_t nslots = (int64_t)pool->num_blocks * pool->block_size;
    const int alias = (pool->v == NULL || pool->v == pool->k);
    if (pool->is_int8 && pool->scale_mode == 0)
        return OR_E_ARG;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= nslots)
            return OR_E_SLOT;
        int64_t blk = slot / pool->block_size;
        int64_t off = slot % pool->block_size;
        int64_t base = (blk * pool->block_size + off) * row; /* element offset */
        for (int which = 0; which < (alias ? 1 : 2); ++which) {
            const uint16_t *src = (which == 0 ? k : v) + (int64_t)t * row;
            void *dst = (which == 0 ? pool->k : pool->v);
            float *tbl = (which == 0 ? pool->k_scale : pool->v_scale);
            if (!pool->is_int8) {
                memcpy((uint16_t *)dst + base, src, (size_t)row * sizeof(uint16_t));
            } else if (pool->scale_mode == 1) {
                float s = oracle_per_token_scale(src, row);
                tbl[slot] = s;
                oracle_quantize(src, row, s, (int8_t *)dst + base);
            } else {
                for (int32_t h = 0; h < pool->num_kv_heads; ++h)
                    oracle_quantize(src + (int64_t)h * pool->head_dim, pool->head_dim, tbl[h],
                                    (int8_t *)dst + base + (int64_t)h * pool->head_dim);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Rotary position embedding, for RoPE fused with the append.  [Lab5] model  */
/* overview names p-RoPE on Gemma4's global layers but gives no formula;    */
/* the definition followed is RoFormer's (Su et al., "RoFormer: Enhanced    */
/* Transformer with Rotary Position Embedding", section 3.2, general form,  */
/* and its element-wise form in section 3.4.2): the vector at position m is */
/* cut into two-dimensional pairs and pair i turns by the angle m*theta_i,  */
/*     a' = a cos(m theta_i) - b sin(m theta_i),                             */
/*     b' = a sin(m theta_i) + b cos(m theta_i).                             */
/* p-RoPE (Barbero et al., "Round and Round We Go! What makes Rotary        */
/* Positional Encodings useful?", its p-RoPE) drops the lowest frequencies;  */
/* read here as: the first rotary_pairs pairs (the highest frequencies of a */
/* decreasing theta table) turn and the rest pass unchanged.  theta_i is a  */
/* table the caller gives.  Pair i is dims (i, i + D/2) (layout 0, halves)  */
/* or (2i, 2i + 1) (layout 1, RoFormer's own interleaving).                 */
/*                                                                          */
/* Precision: the rotated values are stored as bf16 and, in int8 pools,     */
/* quantised, so a rounding decides stored bits.  Both sides take it in the */
/* same precision, the one the library states: cos and sin of the fp64      */
/* angle m * theta_i rounded once to fp32 (the table), then in fp32         */
/* t = b * s, a' = fma(a, c, -t) and t = b * c, b' = fma(a, s, t), each     */
/* rounded to bf16 (nearest, ties to even).  oracle_rope_exact is the fp64  */
/* rotation without any rounding, for the pins.                             */
/* ------------------------------------------------------------------------ */
enum { OR_E_POS = -4 };

/* fp32 -> bf16 bit pattern, round to nearest, ties to even (NaN kept quiet). */
uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x0040u);
    return (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}

/* 1 if the fp64 value v lies so close to the midpoint between two fp32
 * numbers that another faithful fp64 cos or sin (a few ulps away) could round
 * to the other one. */
static int near_f32_midpoint(double v)
{
    float f = (float)v;
    double d = v - (double)f;
    if (d == 0.0 || v == 0.0)
        return 0;
    float g = nextafterf(f, d > 0 ? INFINITY : -INFINITY);
    double mid = 0.5 * ((double)f + (double)g);
    double ulp = ldexp(1.0, ilogb(v) - 52);
    return fabs(v - mid) <= 8.0 * ulp;
}

/* table[m][i] = (fp32(cos(m theta_i)), fp32(sin(m theta_i))), m < npos,
 * i < pairs; the angle is one fp64 product.  ambiguous[m][i] (may be NULL)
 * flags entries whose rounding another faithful cos / sin could change. */
void oracle_rope_table(const double *theta, int32_t pairs, int64_t npos, float *table,
                       uint8_t *ambiguous)
{
    for (int64_t m = 0; m < npos; ++m)
        for (int32_t i = 0; i < pairs; ++i) {
            double ang = (double)m * theta[i];
            double c = cos(ang), s = sin(ang);
            int64_t e = m * pairs + i;
            table[2 * e] = (float)c;
            table[2 * e + 1] = (float)s;
            if (ambiguous)
                ambiguous[e] = (uint8_t)(near_f32_midpoint(c) || near_f32_midpoint(s));
        }
}

static void pair_dims(int32_t i, int32_t head_dim, int32_t layout, int32_t *ia, int32_t *ib)
{
    if (layout == 0) {
        *ia = i;
        *ib = i + head_dim / 2;
    } else {
        *ia = 2 * i;
        *ib = 2 * i + 1;
    }
}

/* x, y: [num_tokens][heads][head_dim] bf16 bits; token t sits at position
 * pos[t].  A negative position (padding) or one past the table copies the
 * row unchanged; the latter also makes the call return OR_E_POS.  y may be
 * x. */
int oracle_rope(const uint16_t *x, uint16_t *y, int64_t num_tokens, int32_t heads,
                int32_t head_dim, const int64_t *pos, const float *table, int64_t npos,
                int32_t pairs, int32_t layout)
{
    if (pairs < 0 || 2 * pairs > head_dim || (head_dim & 1))
        return OR_E_ARG;
    int rc = OR_OK;
    const int64_t row = (int64_t)heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const uint16_t *xr = x + t * row;
        uint16_t *yr = y + t * row;
        int64_t m = pos[t];
        if (yr != xr)
            memcpy(yr, xr, (size_t)row * sizeof(uint16_t));
        if (m < 0)
            continue;
        if (m >= npos) {
            rc = OR_E_POS;
            continue;
        }
        for (int32_t h = 0; h < heads; ++h) {
            const uint16_t *xh = xr + (int64_t)h * head_dim;
            uint16_t *yh = yr + (int64_t)h * head_dim;
            for (int32_t i = 0; i < pairs; ++i) {
                int32_t ia, ib;
                pair_dims(i, head_dim, layout, &ia, &ib);
                const float a = bf16_bits_to_float(xh[ia]), b = bf16_bits_to_float(xh[ib]);
                const float c = table[2 * (m * pairs + i)], s = table[2 * (m * pairs + i) + 1];
                /* plain float products are single IEEE fp32 roundings here
                 * (no contraction: built with -ffp-contract=off) */
                const float t1 = b * s;
                const float ap = fmaf(a, c, -t1);
                const float t2 = b * c;
                const float bp = fmaf(a, s, t2);
                yh[ia] = oracle_f32_to_bf16(ap);
                yh[ib] = oracle_f32_to_bf16(bp);
            }
        }
    }
    return rc;
}

/* The same rotation in fp64 with no rounding: x, y [head_dim], position m. */
void oracle_rope_exact(const double *x, double *y, int32_t head_dim, double m,
                       const double *theta, int32_t pairs, int32_t layout)
{
    for (int32_t d = 0; d < head_dim; ++d)
        y[d] = x[d];
    for (int32_t i = 0; i < pairs; ++i) {
        int32_t ia, ib;
        pair_dims(i, head_dim, layout, &ia, &ib);
        double c = cos(m * theta[i]), s = sin(m * theta[i]);
        y[ia] = x[ia] * c - x[ib] * s;
        y[ib] = x[ia] * s + x[ib] * c;
    }
}

/* ------------------------------------------------------------------------ */
/* Gather: logical key j of sequence b, kv head g, element d, dequantised    */
/* to fp64 ([Lab5] Paged Attention: logical block j/P -> physical block     */
/* block_table[b][j/P], slot j%P; [tiniestgpt] section 5: dequantise after  */
/* the gather).                                                             */
/* ------------------------------------------------------------------------ */
static double kv_value(const oracle_pool *pool, int is_v, int64_t phys, int64_t off, int32_t g,
                       int32_t d)
{
    const void *base = is_v && pool->v ? pool->v : pool->k;
    const float *tbl = is_v && pool->v ? pool->v_scale : pool->k_scale;
    int64_t idx = ((phys * pool->block_size + off) * pool->num_kv_heads + g) * pool->head_dim + d;
    if (!pool->is_int8)
        return (double)bf16_bits_to_float(((const uint16_t *)base)[idx]);
    double s = pool->scale_mode == 1 ? (double)tbl[phys * pool->block_size + off]
                                     : (double)tbl[g];
    return (double)((const int8_t *)base)[idx] * s;
}

/* Mask M of [Lab5] 滑动窗口注意力: the query at position pos sees key j iff
 * j <= pos (causal, global layers) and, on a sliding layer of window w,
 * j >= pos - w (the band [i-w, i]). */
static int mask_allows(int64_t j, int64_t pos, int32_t window)
{
    if (j > pos)
        return 0;
    if (window > 0 && j < pos - window)
        return 0;
    return 1;
}

/* Table entry and offset of the slot that holds position j of a sequence.
 * Paged ([Lab5] Paged Attention): entry j / P, offset j % P.
 * Ring ([Lab5] Ring KV Cache: the KV of absolute position t lives in slot
 * t mod W of a fixed ring of W slots): slot r = j mod W with
 * W = ring_blocks * P, i.e. entry r / P, offset r % P. */
static void slot_of_position(const oracle_pool *pool, int64_t j, int64_t *entry, int64_t *off)
{
    const int64_t P = pool->block_size;
    if (pool->ring_blocks > 0) {
        const int64_t W = (int64_t)pool->ring_blocks * P;
        const int64_t r = j % W;
        *entry = r / P;
        *off = r % P;
    } else {
        *entry = j / P;
        *off = j % P;
    }
}

/* Physical block of logical key j of sequence b (its offset in *off), or -1
 * if out of range. */
static int64_t phys_block(const oracle_pool *pool, const int32_t *block_table,
                          int32_t max_blocks_per_seq, int32_t b, int64_t j, int64_t *off)
{
    int64_t lb;
    slot_of_position(pool, j, &lb, off);
    if (lb >= max_blocks_per_seq)
        return -1;
    int32_t p = block_table[(int64_t)b * max_blocks_per_seq + lb];
    if (p < 0 || p >= pool->num_blocks)
        return -1;
    return p;
}

/* Slot ids of n tokens (sequence seq[i], absolute position pos[i]) under
 * the pool's layout: block_table[seq][entry] * P + offset, or -1 for a
 * negative position or a table entry that names no block of the pool. */
void oracle_slot_mapping(const oracle_pool *pool, const int32_t *block_table,
                         int32_t max_blocks_per_seq, const int32_t *seq, const int64_t *pos,
                         int64_t n, int64_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t off;
        int64_t p = pos[i] < 0 ? -1
                               : phys_block(pool, block_table, max_blocks_per_seq, seq[i], pos[i],
                                            &off);
        out[i] = p < 0 ? -1 : p * pool->block_size + off;
    }
}

/* One output row (sequence b, query head h) of masked softmax attention over
 * the keys j in [key_begin, key_end) that the mask allows.  Returns the
 * log-sum-exp of the allowed scores (natural log; -inf when no key is
 * allowed) and writes y = softmax(s) V into o (zeros when empty).
 *
 * s_j = softmax_scale * <q, K_j> ([CS336-L10] decode formula, with the
 * caller's scale in place of 1/sqrt(d_h)); query head h reads kv head
 * h / (H_q / H_kv) ([Lab5] 分组查询注意力: consecutive query heads share a KV
 * head, the same as repeating each KV head G times).  Softmax with the
 * maximum subtracted, all in fp64. */
static int attend_row_at(const uint16_t *qrow, const oracle_pool *pool,
                         const int32_t *block_table, int32_t max_blocks_per_seq, int64_t len,
                         int64_t pos, int32_t num_q_heads, int32_t window, double softmax_scale,
                         int32_t b, int32_t h, int64_t key_begin, int64_t key_end,
                         double *lse_out, double *o);

static int attend_row(const uint16_t *q, const oracle_pool *pool, const int32_t *block_table,
                      int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_q_heads,
                      int32_t window, double softmax_scale, int32_t b, int32_t h,
                      int64_t key_begin, int64_t key_end, double *lse_out, double *o)
{
    const int64_t len = seq_lens[b];
    return attend_row_at(q + ((int64_t)b * num_q_heads + h) * pool->head_dim, pool, block_table,
                         max_blocks_per_seq, len, len - 1, num_q_heads, window, softmax_scale, b,
                         h, key_begin, key_end, lse_out, o);
}

/* The same for a query row qrow at absolute position pos of a sequence whose
 * cache holds len keys (pos <= len - 1): keys j <= pos (and j >= pos - w on
 * a sliding layer), so a query sees the keys before it and itself -- causal
 * within a chunk of several new tokens ([Lab5] Flash Attention: q_len > 1 in
 * prefill; [Lab5] 滑动窗口注意力: mask M). */
static int attend_row_at(const uint16_t *qrow, const oracle_pool *pool,
                         const int32_t *block_table, int32_t max_blocks_per_seq, int64_t len,
                         int64_t pos, int32_t num_q_heads, int32_t window, double softmax_scale,
                         int32_t b, int32_t h, int64_t key_begin, int64_t key_end,
                         double *lse_out, double *o)
{
    const int32_t D = pool->head_dim;
    const int32_t G = num_q_heads / pool->num_kv_heads;
    const int32_t g = h / G;

    for (int32_t d = 0; d < D; ++d)
        o[d] = 0.0;
    *lse_out = -INFINITY;
    if (key_begin < 0)
        key_begin = 0;
    if (key_end > len)
        key_end = len;
    if (key_end <= key_begin)
        return OR_OK;

    int64_t n = key_end - key_begin;
    double *s = (double *)malloc((size_t)n * sizeof(double));
    if (!s)
        return OR_E_ARG;
    double m = -INFINITY;
    int rc = OR_OK;
    for (int64_t i = 0; i < n; ++i) {
        int64_t j = key_begin + i;
        s[i] = -INFINITY; /* M_j = -inf outside the mask */
        if (!mask_allows(j, pos, window))
            continue;
        int64_t off;
        int64_t p = phys_block(pool, block_table, max_blocks_per_seq, b, j, &off);
        if (p < 0) {
            rc = OR_E_BLOCK;
            break;
        }
        double acc = 0.0;
        for (int32_t d = 0; d < D; ++d)
            acc += (double)bf16_bits_to_float(qrow[d]) * kv_value(pool, 0, p, off, g, d);
        s[i] = softmax_scale * acc;
        if (s[i] > m)
            m = s[i];
    }
    if (rc == OR_OK && m > -INFINITY) {
        double z = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            if (s[i] == -INFINITY)
                continue;
            int64_t j = key_begin + i;
            int64_t off;
            int64_t p = phys_block(pool, block_table, max_blocks_per_seq, b, j, &off);
            double e = exp(s[i] - m);
            z += e;
            for (int32_t d = 0; d < D; ++d)
                o[d] += e * kv_value(pool, 1, p, off, g, d);
        }
        for (int32_t d = 0; d < D; ++d)
            o[d] /= z;
        *lse_out = m + log(z);
    }
    free(s);
    return rc;
}

static int check_shapes(const oracle_pool *pool, int32_t num_q_heads)
{
    if (pool->num_kv_heads <= 0 || pool->head_dim <= 0 || pool->block_size <= 0 ||
        num_q_heads <= 0 || num_q_heads % pool->num_kv_heads != 0)
        return OR_E_ARG;
    if (pool->is_int8 && pool->scale_mode == 0)
        return OR_E_ARG;
    if (pool->ring_blocks < 0)
        return OR_E_ARG;
    return OR_OK;
}

/* Decode attention for the listed rows (pairs (b, h); rows == NULL means all
 * B*H_q rows in order).  out: [nrows][head_dim] fp64.  Each row attends over
 * all keys 0..len_b-1 that the mask allows ([Lab5] Paged Attention: gather
 * the sequence's blocks in logical order, then dense attention). */
int oracle_decode(const uint16_t *q, const oracle_pool *pool, const int32_t *block_table,
                  int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                  int32_t num_q_heads, int32_t window, double softmax_scale, const int32_t *rows,
                  int32_t nrows, double *out, int32_t num_threads)
{
    int rc = check_shapes(pool, num_q_heads);
    if (rc)
        return rc;
    if (!rows)
        nrows = batch * num_q_heads;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : bad)
#endif
    for (int32_t r = 0; r < nrows; ++r) {
        int32_t b = rows ? rows[2 * r] : r / num_q_heads;
        int32_t h = rows ? rows[2 * r + 1] : r % num_q_heads;
        double lse;
        int e = attend_row(q, pool, block_table, max_blocks_per_seq, seq_lens, num_q_heads, window,
                           softmax_scale, b, h, 0, seq_lens[b],
                           &lse, out + (int64_t)r * pool->head_dim);
        if (e)
            bad |= 1;
    }
    (void)num_threads;
    return bad ? OR_E_BLOCK : OR_OK;
}

/* Attention of a chunk of new tokens per sequence (chunked prefill, or the
 * gamma + 1 tokens a speculative step verifies: tiniestgpt notes, section 7).
 * Sequence b's query tokens are rows q_start[b] .. q_start[b+1]-1 of
 * q [total][num_q_heads][head_dim]; they are the sequence's last n_b tokens,
 * so token i sits at position seq_lens[b] - n_b + i and attends the keys
 * allowed at that position (causal within the chunk, windowed on sliding
 * layers).  out: [total][num_q_heads][head_dim] fp64. */
int oracle_prefill(const uint16_t *q, const oracle_pool *pool, const int32_t *block_table,
                   int32_t max_blocks_per_seq, const int32_t *seq_lens, const int32_t *q_start,
                   int32_t batch, int32_t num_q_heads, int32_t window, double softmax_scale,
                   double *out, int32_t num_threads)
{
    int rc = check_shapes(pool, num_q_heads);
    if (rc)
        return rc;
    const int32_t D = pool->head_dim;
    const int64_t total = q_start[batch];
    int bad = 0;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : bad)
#endif
    for (int64_t r = 0; r < total * num_q_heads; ++r) {
        const int64_t row = r / num_q_heads;
        const int32_t h = (int32_t)(r % num_q_heads);
        int32_t b = 0;
        while (q_start[b + 1] <= row)
            ++b;
        const int64_t n = q_start[b + 1] - q_start[b];
        const int64_t len = seq_lens[b];
        const int64_t pos = len - n + (row - q_start[b]);
        double lse;
        int e = pos < 0 ? OR_E_ARG
                        : attend_row_at(q + (row * num_q_heads + h) * D, pool, block_table,
                                        max_blocks_per_seq, len, pos, num_q_heads, window,
                                        softmax_scale, b, h, 0, pos + 1, &lse,
                                        out + r * D);
        if (e)
            bad |= 1;
    }
    (void)num_threads;
    return bad ? OR_E_ARG : OR_OK;
}

/* Partial attention of every row (b, h) over its own key range
 * [key_begin[b], key_end[b]) (intersected with the mask): writes the
 * log-sum-exp lse[b][h] and the normalised partial output o[b][h][:].  This
 * is the state that split-KV passes to a combine step. */
int oracle_partial(const uint16_t *q, const oracle_pool *pool, const int32_t *block_table,
                   int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t batch,
                   int32_t num_q_heads, int32_t window, double softmax_scale,
                   const int64_t *key_begin, const int64_t *key_end, double *lse, double *o,
                   int32_t num_threads)
{
    int rc = check_shapes(pool, num_q_heads);
    if (rc)
        return rc;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads) reduction(| : bad)
#endif
    for (int32_t r = 0; r < batch * num_q_heads; ++r) {
        int32_t b = r / num_q_heads, h = r % num_q_heads;
        int e = attend_row(q, pool, block_table, max_blocks_per_seq, seq_lens, num_q_heads, window,
                           softmax_scale, b, h, key_begin[b], key_end[b], lse + r,
                           o + (int64_t)r * pool->head_dim);
        if (e)
            bad |= 1;
    }
    (void)num_threads;
    return bad ? OR_E_BLOCK : OR_OK;
}

/* Merge n partial states (lse_i, o_i) of one row: L = log sum_i exp(lse_i),
 * y = sum_i exp(lse_i - L) o_i.  Partials with lse = -inf carry no weight.
 * The rule is the online-softmax merge of two (max, sum, output) states
 * ([Lab5] Flash Attention section: running max m, sum l and unnormalised
 * output o, final O = o / l) applied to whole key ranges. */
void oracle_lse_combine(const double *lse, const double *o, int32_t n, int32_t head_dim,
                        double *out, double *lse_total)
{
    double m = -INFINITY;
    for (int32_t i = 0; i < n; ++i)
        if (lse[i] > m)
            m = lse[i];
    for (int32_t d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (m == -INFINITY) {
        *lse_total = -INFINITY;
        return;
    }
    double z = 0.0;
    for (int32_t i = 0; i < n; ++i)
        if (lse[i] > -INFINITY)
            z += exp(lse[i] - m);
    double L = m + log(z);
    for (int32_t i = 0; i < n; ++i) {
        if (lse[i] == -INFINITY)
            continue;
        double w = exp(lse[i] - L);
        for (int32_t d = 0; d < head_dim; ++d)
            out[d] += w * o[(int64_t)i * head_dim + d];
    }
    *lse_total = L;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
