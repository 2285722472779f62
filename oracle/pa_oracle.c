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
 *  - swap    (vLLM and PagedAttention page, preemption: physical blocks move
 *      out of HBM and back; the LLM-inference page's swap of a request's KV
 *      blocks to CPU memory and back): the same byte copy, but from block src
 *      of one pool to block dst of another pool of the same block geometry.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

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

static double element(const void* base, int dtype, int64_t index) {
    switch (dtype) {
        case ORACLE_F32: return (double)((const float*)base)[index];
        case ORACLE_F16: return f16_bits_to_double(((const uint16_t*)base)[index]);
        case ORACLE_BF16: return bf16_bits_to_double(((const uint16_t*)base)[index]);
        default: return NAN;
    }
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
                  double scale) {
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
        double dot = 0.0;
        for (int i = 0; i < head_dim; ++i)
            dot += element(query, dtype, q_base + i) * element(key_cache, dtype, row_base[pos] + i);
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
        for (int i = 0; i < head_dim; ++i) o[i] += p * element(value_cache, dtype, row_base[pos] + i);
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
                              block_size, max_blocks_per_seq, num_blocks, scale);
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
                              max_blocks_per_seq, num_blocks, scale);
        if (st != ORACLE_OK) return st;
    }
    return ORACLE_OK;
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
