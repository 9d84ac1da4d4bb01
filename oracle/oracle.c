/*
 * oracle.c -- plain, slow, fp64 CPU reference for one paged-KV engine step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library; both sides receive the same seeded inputs from the workload
 * generator and nothing else.
 *
 * What it computes (the step traced on the page "vLLM 推理流程分析"):
 *   1. slot_mapping for every scheduled token                 (§5.1.2)
 *   2. the KV-cache scatter (reshape_and_cache_flash)          (§6.3)
 *      and the zeroing of newly allocated blocks              (§4, §5.1.1)
 *   3. causal GQA attention of every scheduled query token over its
 *      request's context, read through block_table            (§6.2, §10.1-10.2)
 * and, for the partition pins, attention restricted to one key range with
 * the (m, l, o) partial it produces plus the merge of several partials
 * (page "vLLM 源码完全拆解（十六）", section "第三条走读路径：KV 页表怎样变成 GPU
 * 上的真实地址": per-partition local (m_r, l_r, o_r) merged with exponential
 * rescaling; page and partition boundaries must not change the result).
 *
 * Conventions (each is a reading of the pages, listed in the design notes):
 *   - K and V caches are separate arrays, each [num_blocks][block_size][Hkv][D]
 *     of IEEE bfloat16 bit patterns (uint16).                 (§6.2 layout)
 *   - query q is [T][Hq][D] bf16; query head h reads kv head h / (Hq/Hkv).
 *   - the query token i of request r sits at absolute position
 *     num_computed[r] + i and sees keys 0..position (bottom-right causal).
 *   - a negative slot means "do not write this token".
 *   - softmax uses the natural exponential; scores are scale * <q, k>.
 *   - all arithmetic is IEEE double; inputs are widened exactly from bf16.
 *
 * Parity pins (tests/test_oracle_pins.py) tie every function here to facts
 * the pages state or to mathematics: worked slot examples, closed forms,
 * invariances, and a dense brute force on tiny inputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_METADATA 1
#define ORACLE_BAD_BLOCK 2
#define ORACLE_NO_MEMORY 3

double oracle_e4m3_value(uint8_t code);

/* bf16 -> double, exact: a bf16 pattern is the top half of an IEEE binary32. */
static double bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

double oracle_bf16_value(uint16_t bits) { return bf16_to_double(bits); }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops from now on (n >= 1); for timing the oracle
 * on one core and on all of them. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Step 1 -- slot_mapping ("vLLM 推理流程分析" §5.1.2, compute_slot_mapping;
 * also "vLLM 源码完全拆解（十六）", third walk-through: logical position p
 * splits into logical block p / S and offset p % S, the block table gives the
 * physical block, slot = physical * S + offset).
 *
 * Token i of request r has position num_computed[r] + i (§5.1.2 positions).
 * Returns ORACLE_BAD_METADATA if a needed block-table column is out of range.
 */
int oracle_slot_mapping(int32_t num_reqs, const int32_t *query_start_loc,
                        const int32_t *num_computed, const int32_t *block_table,
                        int32_t max_blocks_per_req, int32_t block_size,
                        int64_t *slot_mapping) {
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t first = query_start_loc[r];
        int32_t count = query_start_loc[r + 1] - first;
        for (int32_t i = 0; i < count; ++i) {
            int64_t position = (int64_t)num_computed[r] + i;
            int64_t logical_block = position / block_size;
            int64_t offset = position % block_size;
            if (logical_block >= max_blocks_per_req) return ORACLE_BAD_METADATA;
            int64_t physical = block_table[(int64_t)r * max_blocks_per_req + logical_block];
            slot_mapping[first + i] = physical * block_size + offset;
        }
    }
    return ORACLE_OK;
}

/*
 * Step 2 -- the cache write ("vLLM 推理流程分析" §6.3, reshape_and_cache_flash):
 * token t's key and value vectors (all kv heads, all dims) are copied bit for
 * bit into slot slot_mapping[t] of the key and value caches.  A slot is a row
 * of Hkv*D elements because the cache is [num_blocks][block_size][Hkv][D].
 * Negative slots are skipped.  Returns ORACLE_BAD_BLOCK for a slot past the
 * end of the cache (nothing is written for that token).
 */
int oracle_write_kv(int32_t num_tokens, int32_t num_heads_kv, int32_t head_dim,
                    const uint16_t *key, const uint16_t *value,
                    const int64_t *slot_mapping, uint16_t *key_cache,
                    uint16_t *value_cache, int64_t num_slots) {
    int status = ORACLE_OK;
    int64_t row = (int64_t)num_heads_kv * head_dim;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { status = ORACLE_BAD_BLOCK; continue; }
        for (int64_t e = 0; e < row; ++e) {
            key_cache[slot * row + e] = key[(int64_t)t * row + e];
            value_cache[slot * row + e] = value[(int64_t)t * row + e];
        }
    }
    return status;
}

/*
 * Zeroing of newly allocated cache blocks ("vLLM 推理流程分析" §4: the
 * scheduler output lists new_block_ids_to_zero, blocks whose old contents must
 * be cleared; §5.1.1: _update_states zeroes them so that cache positions not
 * yet written are never read as stale KV).  Every byte of the K and V entries
 * of each listed block becomes 0 (+0 in bf16, code 0x00 in E4M3); ids < 0 are
 * skipped; an id past the cache is skipped and reported.
 */
int oracle_zero_blocks(int32_t num_ids, const int32_t *block_ids, int64_t num_blocks, int64_t block_bytes,
                       uint8_t *key_cache, uint8_t *value_cache) {
    int status = ORACLE_OK;
    for (int32_t i = 0; i < num_ids; ++i) {
        int64_t b = block_ids[i];
        if (b < 0) continue;
        if (b >= num_blocks) { status = ORACLE_BAD_BLOCK; continue; }
        memset(key_cache + b * block_bytes, 0, (size_t)block_bytes);
        memset(value_cache + b * block_bytes, 0, (size_t)block_bytes);
    }
    return status;
}

/*
 * FP8 KV cache ("vLLM 推理流程分析" §6.3: reshape_and_cache_flash takes
 * kv_cache_dtype, k_scale and v_scale and converts to FP8 when the cache is
 * quantised).  Reading: the cache holds OCP E4M3 codes (1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; largest finite 448, no infinities,
 * S.1111.111 is NaN) of x / scale, with one float scale per tensor; a read
 * returns code_value * scale.  The quotient is formed in IEEE binary32 (the
 * precision the write kernel uses), then rounded to the nearest E4M3 value,
 * ties to even, saturating to +-448.
 */
double oracle_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);              /* subnormal: m * 2^-9 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isinf(x)) return (uint8_t)(sign | 0x7E);     /* saturates like any large value */
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    /* spacing of the E4M3 grid around a: 2^-9 below the smallest normal
     * 2^-6, else 2^(exponent - 3) */
    int ex;
    frexp(a, &ex);                                    /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                                   /* floor(log2(a)) */
    double quantum = e < -6 ? ldexp(1.0, -9) : ldexp(1.0, e - 3);
    double v = rint(a / quantum) * quantum;           /* nearest, ties to even */
    if (v > 448.0) v = 448.0;                         /* saturate to the largest finite */
    if (v == 0.0) return sign;
    frexp(v, &ex);
    e = ex - 1;
    uint8_t bits;
    if (e < -6) {
        bits = (uint8_t)(v / ldexp(1.0, -9));         /* subnormal mantissa */
    } else {
        int mant = (int)((v / ldexp(1.0, e) - 1.0) * 8.0);
        bits = (uint8_t)(((e + 7) << 3) | mant);
    }
    return (uint8_t)(sign | bits);
}

static float fp8_quotient(uint16_t bits, float scale) {
    return (float)bf16_to_double(bits) / scale;       /* binary32 division */
}

/* Step 2 with an FP8 cache: caches are [num_slots][Hkv*D] E4M3 codes. */
int oracle_write_kv_fp8(int32_t num_tokens, int32_t num_heads_kv, int32_t head_dim,
                        const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                        uint8_t *key_cache, uint8_t *value_cache, int64_t num_slots,
                        float k_scale, float v_scale) {
    int status = ORACLE_OK;
    int64_t row = (int64_t)num_heads_kv * head_dim;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_slots) { status = ORACLE_BAD_BLOCK; continue; }
        for (int64_t e = 0; e < row; ++e) {
            key_cache[slot * row + e] = oracle_e4m3_encode(fp8_quotient(key[(int64_t)t * row + e], k_scale));
            value_cache[slot * row + e] = oracle_e4m3_encode(fp8_quotient(value[(int64_t)t * row + e], v_scale));
        }
    }
    return status;
}

/* Metadata check shared by the attention entry points: q_len from the
 * prefix sums ("vLLM 源码完全拆解（十六）", fourth walk-through: c_i tokens of
 * request i, query_start_loc its prefix sum) and seq_len = num_computed +
 * num_scheduled ("vLLM 推理流程分析" §5.1.2). */
static int check_metadata(int32_t num_reqs, const int32_t *qsl, const int32_t *seq_lens,
                          const int32_t *num_computed, int32_t max_blocks_per_req,
                          int32_t block_size) {
    if (qsl[0] != 0) return ORACLE_BAD_METADATA;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t q_len = qsl[r + 1] - qsl[r];
        if (q_len < 0) return ORACLE_BAD_METADATA;
        if (num_computed[r] < 0) return ORACLE_BAD_METADATA;
        if (num_computed[r] + q_len != seq_lens[r]) return ORACLE_BAD_METADATA;
        if (((int64_t)seq_lens[r] + block_size - 1) / block_size > max_blocks_per_req)
            return ORACLE_BAD_METADATA;
    }
    return ORACLE_OK;
}

/* Gather request r's keys and values for positions [0, length) into
 * contiguous float arrays [length][Hkv][D] (bf16 -> float is exact).  This is
 * the logical->physical translation of "vLLM 请求生命周期" §7 (logical block
 * [0,1,2] -> block table -> physical [7,12,19]). */
static int gather_context(int32_t r, int32_t length, int32_t num_heads_kv, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks, const int32_t *block_table,
                          int32_t max_blocks_per_req, const void *key_cache,
                          const void *value_cache, int kv_fp8, float *k_ctx, float *v_ctx) {
    int64_t row = (int64_t)num_heads_kv * head_dim;
    for (int32_t j = 0; j < length; ++j) {
        int32_t physical = block_table[(int64_t)r * max_blocks_per_req + j / block_size];
        if (physical < 0 || physical >= num_blocks) return ORACLE_BAD_BLOCK;
        int64_t slot = (int64_t)physical * block_size + j % block_size;
        for (int64_t e = 0; e < row; ++e) {
            /* an E4M3 code's value is exact in binary32; its scale is applied
             * in fp64 by the caller */
            k_ctx[(int64_t)j * row + e] = kv_fp8
                ? (float)oracle_e4m3_value(((const uint8_t *)key_cache)[slot * row + e])
                : (float)bf16_to_double(((const uint16_t *)key_cache)[slot * row + e]);
            v_ctx[(int64_t)j * row + e] = kv_fp8
                ? (float)oracle_e4m3_value(((const uint8_t *)value_cache)[slot * row + e])
                : (float)bf16_to_double(((const uint16_t *)value_cache)[slot * row + e]);
        }
    }
    return ORACLE_OK;
}

/*
 * Attention of one query vector against keys [key_begin, key_end) of a
 * gathered context, in fp64 ("vLLM 源码完全拆解（十六）", third walk-through:
 * s_j = <q, k_j> scaled, m = max_j s_j stabilises the softmax, the output is
 * the softmax-weighted sum of the v_j).  Produces the partial triple:
 *   m = max s_j,  l = sum exp(s_j - m),  o = sum exp(s_j - m) v_j / l.
 * An empty range gives m = -inf, l = 0, o = 0.
 */
static void attend_range(const double *qv, const float *k_ctx, const float *v_ctx,
                         int32_t key_begin, int32_t key_end, int32_t kv_head,
                         int32_t num_heads_kv, int32_t head_dim, double scale,
                         double *scores, double *m_out, double *l_out, double *o_out) {
    int64_t row = (int64_t)num_heads_kv * head_dim;
    double m = -INFINITY;
    for (int32_t j = key_begin; j < key_end; ++j) {
        const float *kj = k_ctx + (int64_t)j * row + (int64_t)kv_head * head_dim;
        double dot = 0.0;
        for (int32_t d = 0; d < head_dim; ++d) dot += qv[d] * (double)kj[d];
        double s = scale * dot;
        scores[j - key_begin] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) o_out[d] = 0.0;
    for (int32_t j = key_begin; j < key_end; ++j) {
        double w = exp(scores[j - key_begin] - m);
        const float *vj = v_ctx + (int64_t)j * row + (int64_t)kv_head * head_dim;
        l += w;
        for (int32_t d = 0; d < head_dim; ++d) o_out[d] += w * (double)vj[d];
    }
    if (l > 0.0)
        for (int32_t d = 0; d < head_dim; ++d) o_out[d] /= l;
    *m_out = m;
    *l_out = l;
}

/*
 * Step 3 -- causal GQA attention for every (or a chosen subset of) query
 * tokens ("vLLM 推理流程分析" §6.2 flash_attn_varlen_func(..., block_table,
 * causal=True); §10.1 "each token sees only itself and earlier tokens";
 * §10.2 decode reads all earlier K/V through the block table).
 *
 * key_begin_override < 0: row i of request r sees keys [0, num_computed+i].
 * key_begin_override >= 0 and key_end_override >= 0: every row instead sees
 * keys [key_begin, min(key_end, its causal end)); used by the partition pins.
 *
 * rows: optional list of n_rows token indices to compute (NULL = all T).
 * out:  [T][Hq][D] doubles, normalised output o (rows not chosen untouched).
 * out_m, out_l: optional [T][Hq] doubles receiving the partial's m and l.
 */
static int attention_core(int32_t num_reqs, int32_t num_heads_q, int32_t num_heads_kv,
                          int32_t head_dim, int32_t block_size, int32_t num_blocks,
                          int32_t max_blocks_per_req, const int32_t *query_start_loc,
                          const int32_t *seq_lens, const int32_t *num_computed,
                          const int32_t *block_table, double softmax_scale,
                          const uint16_t *q, const void *key_cache, const void *value_cache,
                          int kv_fp8, double k_scale, double v_scale,
                          const int32_t *rows, int32_t n_rows,
                          int32_t key_begin_override, int32_t key_end_override,
                          double *out, double *out_m, double *out_l) {
    if (num_heads_kv <= 0 || num_heads_q % num_heads_kv != 0) return ORACLE_BAD_METADATA;
    int st = check_metadata(num_reqs, query_start_loc, seq_lens, num_computed,
                            max_blocks_per_req, block_size);
    if (st != ORACLE_OK) return st;
    const int32_t group = num_heads_q / num_heads_kv;
    const int32_t total_tokens = query_start_loc[num_reqs];

    /* which tokens to compute */
    char *wanted = (char *)calloc((size_t)total_tokens + 1, 1);
    if (!wanted) return ORACLE_NO_MEMORY;
    if (rows == NULL) {
        memset(wanted, 1, (size_t)total_tokens);
    } else {
        for (int32_t i = 0; i < n_rows; ++i)
            if (rows[i] >= 0 && rows[i] < total_tokens) wanted[rows[i]] = 1;
    }

    int status = ORACLE_OK;
    for (int32_t r = 0; r < num_reqs && status == ORACLE_OK; ++r) {
        int32_t first = query_start_loc[r];
        int32_t q_len = query_start_loc[r + 1] - first;
        int32_t any = 0;
        for (int32_t i = 0; i < q_len; ++i) any |= wanted[first + i];
        if (!any) continue;
        int32_t length = seq_lens[r];
        int64_t row = (int64_t)num_heads_kv * head_dim;
        float *k_ctx = (float *)malloc(sizeof(float) * (size_t)length * (size_t)row + 1);
        float *v_ctx = (float *)malloc(sizeof(float) * (size_t)length * (size_t)row + 1);
        if (!k_ctx || !v_ctx) { free(k_ctx); free(v_ctx); status = ORACLE_NO_MEMORY; break; }
        status = gather_context(r, length, num_heads_kv, head_dim, block_size, num_blocks,
                                block_table, max_blocks_per_req, key_cache, value_cache,
                                kv_fp8, k_ctx, v_ctx);
        if (status == ORACLE_OK) {
            int64_t pairs = (int64_t)q_len * num_heads_q;
#pragma omp parallel
            {
                double *scores = (double *)malloc(sizeof(double) * ((size_t)length + 1));
                double *qv = (double *)malloc(sizeof(double) * (size_t)head_dim);
                double *ov = (double *)malloc(sizeof(double) * (size_t)head_dim);
#pragma omp for schedule(dynamic, 1)
                for (int64_t p = 0; p < pairs; ++p) {
                    int32_t i = (int32_t)(p / num_heads_q);
                    int32_t h = (int32_t)(p % num_heads_q);
                    int32_t t = first + i;
                    if (!wanted[t]) continue;
                    int32_t position = num_computed[r] + i;
                    int32_t kb = 0, ke = position + 1; /* keys 0..position */
                    if (key_begin_override >= 0 && key_end_override >= 0) {
                        kb = key_begin_override;
                        if (key_end_override < ke) ke = key_end_override;
                        if (kb > ke) kb = ke;
                    }
                    const uint16_t *qrow = q + ((int64_t)t * num_heads_q + h) * head_dim;
                    for (int32_t d = 0; d < head_dim; ++d) qv[d] = bf16_to_double(qrow[d]);
                    double m, l;
                    /* k = code * k_scale and v = code * v_scale (both 1 for bf16):
                     * the key scale joins the softmax scale, the value scale
                     * multiplies the normalised output */
                    attend_range(qv, k_ctx, v_ctx, kb, ke, h / group, num_heads_kv, head_dim,
                                 softmax_scale * k_scale, scores, &m, &l, ov);
                    double *orow = out + ((int64_t)t * num_heads_q + h) * head_dim;
                    for (int32_t d = 0; d < head_dim; ++d) orow[d] = ov[d] * v_scale;
                    if (out_m) out_m[(int64_t)t * num_heads_q + h] = m;
                    if (out_l) out_l[(int64_t)t * num_heads_q + h] = l;
                }
                free(scores);
                free(qv);
                free(ov);
            }
        }
        free(k_ctx);
        free(v_ctx);
    }
    free(wanted);
    return status;
}

int oracle_attention_range(int32_t num_reqs, int32_t num_heads_q, int32_t num_heads_kv,
                           int32_t head_dim, int32_t block_size, int32_t num_blocks,
                           int32_t max_blocks_per_req, const int32_t *query_start_loc,
                           const int32_t *seq_lens, const int32_t *num_computed,
                           const int32_t *block_table, double softmax_scale,
                           const uint16_t *q, const uint16_t *key_cache,
                           const uint16_t *value_cache, const int32_t *rows, int32_t n_rows,
                           int32_t key_begin_override, int32_t key_end_override,
                           double *out, double *out_m, double *out_l) {
    return attention_core(num_reqs, num_heads_q, num_heads_kv, head_dim, block_size, num_blocks,
                          max_blocks_per_req, query_start_loc, seq_lens, num_computed, block_table,
                          softmax_scale, q, key_cache, value_cache, 0, 1.0, 1.0, rows, n_rows,
                          key_begin_override, key_end_override, out, out_m, out_l);
}

/* Step 3 over FP8 caches ([num_blocks][block_size][Hkv][D] E4M3 codes):
 * every key and value is its code's value times k_scale / v_scale. */
int oracle_attention_fp8(int32_t num_reqs, int32_t num_heads_q, int32_t num_heads_kv,
                         int32_t head_dim, int32_t block_size, int32_t num_blocks,
                         int32_t max_blocks_per_req, const int32_t *query_start_loc,
                         const int32_t *seq_lens, const int32_t *num_computed,
                         const int32_t *block_table, double softmax_scale, const uint16_t *q,
                         const uint8_t *key_cache, const uint8_t *value_cache, float k_scale,
                         float v_scale, const int32_t *rows, int32_t n_rows, double *out) {
    return attention_core(num_reqs, num_heads_q, num_heads_kv, head_dim, block_size, num_blocks,
                          max_blocks_per_req, query_start_loc, seq_lens, num_computed, block_table,
                          softmax_scale, q, key_cache, value_cache, 1, (double)k_scale,
                          (double)v_scale, rows, n_rows, -1, -1, out, NULL, NULL);
}

/* The full causal attention of step 3. */
int oracle_attention(int32_t num_reqs, int32_t num_heads_q, int32_t num_heads_kv,
                     int32_t head_dim, int32_t block_size, int32_t num_blocks,
                     int32_t max_blocks_per_req, const int32_t *query_start_loc,
                     const int32_t *seq_lens, const int32_t *num_computed,
                     const int32_t *block_table, double softmax_scale, const uint16_t *q,
                     const uint16_t *key_cache, const uint16_t *value_cache,
                     const int32_t *rows, int32_t n_rows, double *out) {
    return oracle_attention_range(num_reqs, num_heads_q, num_heads_kv, head_dim, block_size,
                                  num_blocks, max_blocks_per_req, query_start_loc, seq_lens,
                                  num_computed, block_table, softmax_scale, q, key_cache,
                                  value_cache, rows, n_rows, -1, -1, out, NULL, NULL);
}

/*
 * Merge of partition partials ("vLLM 源码完全拆解（十六）", third walk-through:
 * the V2 path computes (m_r, l_r, o_r) per partition and merges them, the
 * output scaled by the same exponential factors):
 *   m = max_r m_r,  w_r = exp(m_r - m) * l_r,  o = sum_r w_r o_r / sum_r w_r.
 * Partials with l_r == 0 (empty partitions) carry no weight.
 * m_parts, l_parts: [n_parts]; o_parts: [n_parts][D]; o_out: [D].
 */
void oracle_merge_partials(int32_t n_parts, int32_t head_dim, const double *m_parts,
                           const double *l_parts, const double *o_parts, double *o_out,
                           double *m_out, double *l_out) {
    double m = -INFINITY;
    for (int32_t p = 0; p < n_parts; ++p)
        if (l_parts[p] > 0.0 && m_parts[p] > m) m = m_parts[p];
    double total = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) o_out[d] = 0.0;
    for (int32_t p = 0; p < n_parts; ++p) {
        if (!(l_parts[p] > 0.0)) continue;
        double w = exp(m_parts[p] - m) * l_parts[p];
        total += w;
        for (int32_t d = 0; d < head_dim; ++d) o_out[d] += w * o_parts[(int64_t)p * head_dim + d];
    }
    if (total > 0.0)
        for (int32_t d = 0; d < head_dim; ++d) o_out[d] /= total;
    if (m_out) *m_out = m;
    if (l_out) *l_out = total;
}

/*
 * Cascade precondition ("vLLM 推理流程分析" §4.4: num_common_prefix_blocks is
 * the number of blocks common to the batch, used by cascade attention).  Read
 * as one batch-wide count n: every request with query tokens maps its first n
 * logical blocks to the same physical blocks as every other such request, and
 * has at least n*block_size tokens already computed, so no query token of the
 * step can be masked inside the shared prefix.  Returns ORACLE_OK or
 * ORACLE_BAD_METADATA.
 * The attention result does not depend on n; only this precondition does.
 */
int oracle_check_common_prefix(int32_t num_reqs, const int32_t *query_start_loc,
                               const int32_t *num_computed, const int32_t *block_table,
                               int32_t max_blocks_per_req, int32_t block_size,
                               int32_t num_common_prefix_blocks) {
    int32_t n = num_common_prefix_blocks;
    if (n < 0 || n > max_blocks_per_req) return ORACLE_BAD_METADATA;
    if (n == 0) return ORACLE_OK;
    int32_t reference = -1;
    for (int32_t r = 0; r < num_reqs; ++r) {
        if (query_start_loc[r + 1] - query_start_loc[r] == 0) continue;
        if ((int64_t)n * block_size > num_computed[r]) return ORACLE_BAD_METADATA;
        if (reference < 0) { reference = r; continue; }
        for (int32_t b = 0; b < n; ++b)
            if (block_table[(int64_t)r * max_blocks_per_req + b] !=
                block_table[(int64_t)reference * max_blocks_per_req + b])
                return ORACLE_BAD_METADATA;
    }
    return ORACLE_OK;
}
