/*
 * Plain CPU oracle for paged decode attention, the paged KV write and the
 * block copy.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this; the product path never does.
 *
 * It shares no code, header or constant with the CUDA library.  Everything is
 * computed in double precision, one output row at a time, in the order the
 * pages state the method:
 *
 *  - decode  (MiniPaged-Qwen, section 1 formula and section 6.2 steps 1-5):
 *      for every logical position pos in [0, L):
 *          logical_block = pos / block_size, off = pos % block_size,
 *          pb = block_table[logical_block],
 *          k_pos = key_cache[pb, kvh, off, :],  v_pos = value_cache[pb, kvh, off, :]
 *      s_pos = scale * <q, k_pos>, and the output is the softmax-weighted sum
 *      over ALL L positions (section 5.2: one global normaliser).  The softmax
 *      is taken in two passes (max, then sum) rather than online, so that the
 *      oracle does not depend on the running-max recurrence it is used to check.
 *      GQA: kvh = qh / (H_q / H_kv)  (section 9.1).
 *  - write   (section 8.1/8.2): key_cache[slot / bs, h, slot % bs, :] = key[t, h, :]
 *      as a byte copy; a negative slot means "no write".
 *  - copy    (vLLM and PagedAttention page, copy-on-write section): every
 *      (src, dst) pair copies the whole physical block dst <- src, as bytes.
 *  - FP8 KV cache (the LLM-inference page's quantised KV cache, FP8 named among
 *      the remedies for a full pool; the vLLM and PagedAttention page's KV dtype and
 *      quantisation scales in the attention metadata): a cache element is an OCP
 *      FP8 E4M3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 *      infinities; S.1111.111 is NaN; largest finite 448) and every (physical
 *      block, kv head) carries a float32 scale for K and one for V.  The value
 *      the attention sees is code_value * scale.  Writing quantises
 *      x / scale (divided in float32) to the nearest code, ties to the even
 *      mantissa, magnitudes above 448 saturating to 448, NaN staying NaN.
 *  - swap    (vLLM and PagedAttention page, preemption: physical blocks move
 *      out of HBM and back; the LLM-inference page's swap of a request's KV
 *      blocks to CPU memory and back): the same byte copy, but from block src
 *      of one pool to block dst of another pool of the same block geometry.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_E4M3 = 3 };

enum {
    ORACLE_OK = 0,
    ORACLE_BAD_ARG = -1,
    ORACLE_BAD_TABLE = -2,
    ORACLE_BAD_SLOT = -3,
    ORACLE_NO_MEMORY = -4,
};

/* IEEE 754 binary16 bits -> double (exact). */
static double f16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 0x1F;
    int mantissa = h & 0x3FF;
    double v;
    if (exponent == 0) {
        v = ldexp((double)mantissa, -24); /* subnormal: m * 2^-24 */
    } else if (exponent == 31) {
        v = mantissa ? NAN : INFINITY;
    } else {
        v = ldexp((double)(mantissa + 1024), exponent - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 bits are the upper half of a binary32 (exact). */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 code -> double (exact): subnormals m * 2^-9, normals (1 + m/8) * 2^(e-7). */
static double e4m3_to_double(uint8_t c) {
    const int sign = c >> 7;
    const int e = (c >> 3) & 0xF;
    const int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* float -> E4M3 code: nearest code, ties to the even mantissa; |x| >= 448 gives 448
 * (saturation); NaN gives the NaN code.  The rounding is done in double, where
 * a / 2^k is exact. */
static uint8_t e4m3_from_float(float x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x)) return sign | 0x7F;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int e2;
    frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): floor(log2 a) = e2 - 1 */
    const int e = e2 - 1;
    if (a == 0.0 || e < -6) {
        /* subnormal range: steps of 2^-9; rounding up to 8 steps reaches 2^-6 (code 8) */
        const double n = a * 512.0;
        double r = nearbyint(n); /* round half to even (default rounding mode) */
        return sign | (uint8_t)r;
    }
    /* normal: a = n * 2^(e-3) with n in [8, 16); n rounded; n = 16 carries into the exponent */
    const double n = ldexp(a, 3 - e);
    const double r = nearbyint(n);
    return sign | (uint8_t)(((e + 7) << 3) + (int)r - 8);
}

static double element(const void* base, int dtype, int64_t index) {
    switch (dtype) {
        case ORACLE_F32: return (double)((const float*)base)[index];
        case ORACLE_F16: return f16_bits_to_double(((const uint16_t*)base)[index]);
        case ORACLE_BF16: return bf16_bits_to_double(((const uint16_t*)base)[index]);
        case ORACLE_E4M3: return e4m3_to_double(((const uint8_t*)base)[index]);
        default: return NAN;
    }
}

/* Exposed so that the tests can pin the E4M3 encoding against a library cast. */
int oracle_e4m3_encode(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_from_float(x[i]);
    return ORACLE_OK;
}

/* Exposed so that the tests can pin the element decoding against library casts. */
double oracle_element_to_double(const void* base, int dtype, int64_t index) {
    return element(base, dtype, index);
}

/*
 * One output row: attention of the query row at q_base over positions
 * 0 .. n_att - 1 of sequence b, kv head kvh (n_att <= 0 gives a zero row).
 * Address translation (position -> logical block -> table -> physical block ->
 * offset), fp64 scores, a two-pass softmax (global max, then the normaliser),
 * then the probability-weighted sum of the value rows.
 */
static int attend(double* o, const void* query, int64_t q_base, int n_att, int b, int kvh,
                  const void* key_cache, const void* value_cache, int dtype, const int32_t* block_tables,
                  int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                  double scale, int cache_dtype, const float* k_scale, const float* v_scale) {
    for (int i = 0; i < head_dim; ++i) o[i] = 0.0;
    if (n_att <= 0) return ORACLE_OK;
    double* s = (double*)malloc(sizeof(double) * (size_t)n_att);
    int64_t* row_base = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_att);
    if (!s || !row_base) {
        free(s);
        free(row_base);
        return ORACLE_NO_MEMORY;
    }
    /* Pass 1: address translation and scores. */
    for (int pos = 0; pos < n_att; ++pos) {
        const int logical_block = pos / block_size;
        const int off = pos % block_size;
        const int pb = block_tables[(int64_t)b * max_blocks_per_seq + logical_block];
        if (pb < 0 || pb >= num_blocks) {
            free(s);
            free(row_base);
            return ORACLE_BAD_TABLE;
        }
        row_base[pos] = (((int64_t)pb * num_kv_heads + kvh) * block_size + off) * head_dim;
        /* a scaled (FP8) cache: the element's value is code * the (block, kv head) scale */
        const double ks = k_scale ? (double)k_scale[(int64_t)pb * num_kv_heads + kvh] : 1.0;
        double dot = 0.0;
        for (int i = 0; i < head_dim; ++i)
            dot += element(query, dtype, q_base + i) * (element(key_cache, cache_dtype, row_base[pos] + i) * ks);
        s[pos] = scale * dot;
    }
    /* Pass 2: global max, then the normaliser over all attended positions. */
    double m = s[0];
    for (int pos = 1; pos < n_att; ++pos)
        if (s[pos] > m) m = s[pos];
    double z = 0.0;
    for (int pos = 0; pos < n_att; ++pos) {
        s[pos] = exp(s[pos] - m);
        z += s[pos];
    }
    /* Pass 3: probability-weighted sum of the value rows. */
    for (int pos = 0; pos < n_att; ++pos) {
        const double p = s[pos] / z;
        const int64_t bh = row_base[pos] / head_dim / block_size; /* pb * num_kv_heads + kvh */
        const double vs = v_scale ? (double)v_scale[bh] : 1.0;
        for (int i = 0; i < head_dim; ++i) o[i] += p * (element(value_cache, cache_dtype, row_base[pos] + i) * vs);
    }
    free(s);
    free(row_base);
    return ORACLE_OK;
}

/*
 * Decode attention for the selected output rows (b, qh).
 *   out           [n_rows, head_dim] doubles
 *   query         [num_seqs, num_heads, head_dim]
 *   caches        [num_blocks, num_kv_heads, block_size, head_dim]
 *   block_tables  [num_seqs, max_blocks_per_seq] int32
 *   context_lens  [num_seqs] int32
 * Every row attends all L = context_lens[b] positions; L == 0 gives a zero row.
 * Returns ORACLE_BAD_TABLE if a table entry that the context needs is outside
 * [0, num_blocks).
 */
int oracle_decode_rows(double* out, const int32_t* row_seq, const int32_t* row_head, int n_rows,
                       const void* query, const void* key_cache, const void* value_cache, int dtype,
                       const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                       int num_heads, int num_kv_heads, int head_dim, int block_size,
                       int max_blocks_per_seq, int num_blocks, double scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0)
        return ORACLE_BAD_ARG;
    const int group = num_heads / num_kv_heads;
    for (int r = 0; r < n_rows; ++r) {
        const int b = row_seq[r];
        const int qh = row_head[r];
        if (b < 0 || b >= num_seqs || qh < 0 || qh >= num_heads) return ORACLE_BAD_ARG;
        const int L = context_lens[b];
        if (L < 0 || L > (int64_t)max_blocks_per_seq * block_size) return ORACLE_BAD_ARG;
        const int st = attend(out + (int64_t)r * head_dim, query, ((int64_t)b * num_heads + qh) * head_dim, L, b,
                              qh / group, key_cache, value_cache, dtype, block_tables, num_kv_heads, head_dim,
                              block_size, max_blocks_per_seq, num_blocks, scale, dtype, NULL, NULL);
        if (st != ORACLE_OK) return st;
    }
    return ORACLE_OK;
}

/*
 * Multi-query decode: the verify (or chunked-prefill tail) step of the vLLM and
 * PagedAttention page, section "how the attention kernel reads paged KV": each
 * sequence has a query range and a context length, under a causal mask.
 * Sequence b has q_len query tokens, at positions L - q_len .. L - 1 of its
 * context (L = context_lens[b], their K/V already in the cache); query token t
 * attends positions 0 .. L - q_len + t, none when that bound is negative (a
 * zero row).
 *   out    [n_rows, head_dim] doubles for the rows (row_seq, row_tok, row_head)
 *   query  [num_seqs, q_len, num_heads, head_dim]
 */
int oracle_decode_multi_rows(double* out, const int32_t* row_seq, const int32_t* row_tok, const int32_t* row_head,
                             int n_rows, const void* query, const void* key_cache, const void* value_cache,
                             int dtype, const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                             int q_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                             int max_blocks_per_seq, int num_blocks, double scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 || q_len <= 0)
        return ORACLE_BAD_ARG;
    const int group = num_heads / num_kv_heads;
    for (int r = 0; r < n_rows; ++r) {
        const int b = row_seq[r], t = row_tok[r], qh = row_head[r];
        if (b < 0 || b >= num_seqs || t < 0 || t >= q_len || qh < 0 || qh >= num_heads) return ORACLE_BAD_ARG;
        const int L = context_lens[b];
        if (L < 0 || L > (int64_t)max_blocks_per_seq * block_size) return ORACLE_BAD_ARG;
        const int64_t q_base = (((int64_t)b * q_len + t) * num_heads + qh) * head_dim;
        const int st = attend(out + (int64_t)r * head_dim, query, q_base, L - q_len + t + 1, b, qh / group,
                              key_cache, value_cache, dtype, block_tables, num_kv_heads, head_dim, block_size,
                              max_blocks_per_seq, num_blocks, scale, dtype, NULL, NULL);
        if (st != ORACLE_OK) return st;
    }
    return ORACLE_OK;
}

/*
 * Decode attention over an FP8 (E4M3) cache with a float32 scale per (physical
 * block, kv head) for K (k_scale) and for V (v_scale), both [num_blocks,
 * num_kv_heads]; the query and the output rows as oracle_decode_rows (dtype is
 * the query's).  Element values are code * scale; the rest is the same attention.
 */
int oracle_decode_fp8_rows(double* out, const int32_t* row_seq, const int32_t* row_head, int n_rows,
                           const void* query, int dtype, const uint8_t* key_cache, const uint8_t* value_cache,
                           const float* k_scale, const float* v_scale, const int32_t* block_tables,
                           const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                           int block_size, int max_blocks_per_seq, int num_blocks, double scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 || !k_scale ||
        !v_scale)
        return ORACLE_BAD_ARG;
    const int group = num_heads / num_kv_heads;
    for (int r = 0; r < n_rows; ++r) {
        const int b = row_seq[r];
        const int qh = row_head[r];
        if (b < 0 || b >= num_seqs || qh < 0 || qh >= num_heads) return ORACLE_BAD_ARG;
        const int L = context_lens[b];
        if (L < 0 || L > (int64_t)max_blocks_per_seq * block_size) return ORACLE_BAD_ARG;
        const int st = attend(out + (int64_t)r * head_dim, query, ((int64_t)b * num_heads + qh) * head_dim, L, b,
                              qh / group, key_cache, value_cache, dtype, block_tables, num_kv_heads, head_dim,
                              block_size, max_blocks_per_seq, num_blocks, scale, ORACLE_E4M3, k_scale, v_scale);
        if (st != ORACLE_OK) return st;
    }
    return ORACLE_OK;
}

/*
 * Paged write into an FP8 cache: element i of token t, kv head h becomes
 * e4m3(x / scale[block, h]) with x the source element (dtype f32/f16/bf16) as a
 * float32 and the division done in float32; block = slot / block_size.  Slots as
 * oracle_write_kv.
 */
int oracle_write_kv_fp8(const void* key, const void* value, int dtype, uint8_t* key_cache, uint8_t* value_cache,
                        const float* k_scale, const float* v_scale, const int64_t* slot_mapping, int num_tokens,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks) {
    int status = ORACLE_OK;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            status = ORACLE_BAD_SLOT;
            continue;
        }
        const int64_t block = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const float ks = k_scale[block * num_kv_heads + h];
            const float vs = v_scale[block * num_kv_heads + h];
            const int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            const int64_t dst = ((block * num_kv_heads + h) * block_size + off) * head_dim;
            for (int i = 0; i < head_dim; ++i) {
                const float xk = (float)element(key, dtype, src + i);
                const float xv = (float)element(value, dtype, src + i);
                const float qk = xk / ks;
                const float qv = xv / vs;
                key_cache[dst + i] = e4m3_from_float(qk);
                value_cache[dst + i] = e4m3_from_float(qv);
            }
        }
    }
    return status;
}

/*
 * Paged KV write: token t of key/value [num_tokens, num_kv_heads, head_dim]
 * goes to slot slot_mapping[t].  Slots < 0 are skipped; a slot past the pool
 * is skipped and reported (ORACLE_BAD_SLOT) after all valid writes are done.
 */
int oracle_write_kv(const void* key, const void* value, void* key_cache, void* value_cache,
                    const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int elem_bytes) {
    const int64_t row_bytes = (int64_t)head_dim * elem_bytes;
    int status = ORACLE_OK;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            status = ORACLE_BAD_SLOT;
            continue;
        }
        const int64_t block = slot / block_size;
        const int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t src = ((int64_t)t * num_kv_heads + h) * row_bytes;
            const int64_t dst = ((block * num_kv_heads + h) * block_size + off) * row_bytes;
            memcpy((char*)key_cache + dst, (const char*)key + src, (size_t)row_bytes);
            memcpy((char*)value_cache + dst, (const char*)value + src, (size_t)row_bytes);
        }
    }
    return status;
}

/*
 * Block copy: for each pair (src, dst) in pairs [num_pairs, 2], the whole block
 * dst of both caches becomes a copy of block src.  Pairs with an id outside
 * [0, num_blocks) are skipped and reported.
 */
int oracle_copy_blocks(void* key_cache, void* value_cache, const int64_t* pairs, int num_pairs,
                       int64_t block_bytes, int num_blocks) {
    int status = ORACLE_OK;
    for (int p = 0; p < num_pairs; ++p) {
        const int64_t src = pairs[2 * p];
        const int64_t dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            status = ORACLE_BAD_TABLE;
            continue;
        }
        memcpy((char*)key_cache + dst * block_bytes, (const char*)key_cache + src * block_bytes,
               (size_t)block_bytes);
        memcpy((char*)value_cache + dst * block_bytes, (const char*)value_cache + src * block_bytes,
               (size_t)block_bytes);
    }
    return status;
}

/* Block dst of the destination pool <- block src of the source pool, both caches, as bytes.
 * A pair with an id outside its own pool is skipped and reported. */
int oracle_swap_blocks(void* dst_key, void* dst_value, const void* src_key, const void* src_value,
                       const int64_t* pairs, int num_pairs, int64_t block_bytes, int src_blocks, int dst_blocks) {
    int status = ORACLE_OK;
    for (int p = 0; p < num_pairs; ++p) {
        const int64_t src = pairs[2 * p];
        const int64_t dst = pairs[2 * p + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
            status = ORACLE_BAD_TABLE;
            continue;
        }
        memcpy((char*)dst_key + dst * block_bytes, (const char*)src_key + src * block_bytes, (size_t)block_bytes);
        memcpy((char*)dst_value + dst * block_bytes, (const char*)src_value + src * block_bytes, (size_t)block_bytes);
    }
    return status;
}
