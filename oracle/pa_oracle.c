/*
 * pa_oracle.c -- CPU oracle for the paged KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded
 * restatement of what the paged decode path computes, written so that a
 * reader can check every line against the pages it follows.  Only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg may
 * load it; the product path (the CUDA library) never calls it, and the two
 * share no code, header, table or helper.
 *
 * Arithmetic: every 16-bit input element is decoded exactly to double and
 * every sum, product, exponential and division is taken in double (fp64).
 * Byte-moving operations (cache writes, block copies) copy the 16-bit
 * patterns verbatim.
 *
 * Sources (web pages, cited by title and section):
 *   [GAO]  "PagedAttention & Continuous Batching" (gaoleia.github.io,
 *          2026-01-25): §1.3 physical block, §1.4 block table,
 *          §1.5 slot mapping (worked example: position 35, block_size 16,
 *          block_table[2] = 9 -> slot 147), §1.6 paged attention
 *          (gather K over the block table, softmax(q K^T / sqrt(d)),
 *          gather V, weighted sum, truncated to seq_len), §2.4 prefill vs
 *          decode (a prompt's tokens processed in parallel; a mixed batch of
 *          decode and prefill requests), §2.5 chunked prefill (a long prompt
 *          split into chunks of 512 tokens).
 *   [FEI]  "vLLM 架构详解: PagedAttention、Continuous Batching 与生产级推理优化"
 *          (feifeigd.github.io): "Block Table 实现" (append a token's K/V at
 *          its position in the last block), "共享前缀的 Block 复用"
 *          (several block tables naming the same physical blocks).
 *   [LAKE] "vLLM源码解析(二): 调度系统与PagedAttention实现"
 *          (lakecityint.com): §3.2 copy-on-write (allocate a new physical
 *          block, copy the old block's contents, remap and drop a reference).
 *
 * Readings where the pages are silent or garbled (each one is listed in the
 * design notes as well):
 *   - Pool layout is token-major [num_blocks][block_size][num_kv_heads]
 *     [head_dim], with separate K and V pools ([GAO] §1.3 gives
 *     [block_size, num_heads, head_dim] per block; the sketch in §1.6
 *     indexes a K/V axis that collides with the head axis, so K and V are
 *     read as two pools).
 *   - Grouped-query heads: query head h reads KV head h / (H / Hkv).
 *   - Attended tokens are positions [0, context_len); context_len <= 0
 *     gives an all-zero output row.
 *   - A negative slot in the slot mapping means "no write" (padding).
 *   - Split-context: partition j covers positions [j*P, min(ctx,(j+1)*P));
 *     its partial is (m_j = max score, l_j = sum exp(score - m_j),
 *     o_j = sum exp(score - m_j) v / l_j); merge by log-sum-exp weights
 *     w_j = l_j exp(m_j - max_j m_j).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* ---- 16-bit element decoding (exact) ---------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 encodes zero / subnormals (fraction * 2^-24), exponent
 * 31 encodes inf / NaN. */
static double decode_f16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -mag : mag;
}

/* bfloat16 is the upper 16 bits of an IEEE binary32 value. */
static double decode_bf16(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double decode(uint16_t bits, int dtype)
{
    return dtype == ORACLE_BF16 ? decode_bf16(bits) : decode_f16(bits);
}

/* Exposed for tests: decode n elements into doubles. */
void oracle_decode(double *out, const uint16_t *bits, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = decode(bits[i], dtype);
}

/* ---- FP8 (e4m3) KV codes ----------------------------------------------- */
/*
 * Reading (the pages name an FP8 KV cache, "--kv-cache-dtype fp8", without a
 * format): OCP e4m3 -- 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits, no infinities, S.1111.111 is NaN, largest finite 448, subnormals
 * fraction * 2^-9.  A cached value is stored as code = e4m3(x * inv_scale)
 * with one per-tensor scale; x * inv_scale is one fp32 product, rounded to
 * the nearest e4m3 value (ties to even), out-of-range finite values
 * saturate to +-448, NaN stays NaN.  Dequantised value = e4m3 value * scale.
 */
static double decode_e4m3(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int expo = (c >> 3) & 0xf;
    int frac = c & 0x7;
    double mag;
    if (expo == 15 && frac == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)frac, -9);
    else
        mag = ldexp((double)(8 + frac), expo - 10);
    return sign ? -mag : mag;
}

void oracle_decode_e4m3(double *out, const uint8_t *codes, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = decode_e4m3(codes[i]);
}

/* Nearest e4m3 code to a float (ties to even), saturating finite values:
 * the value's binade fixes the spacing of representable values (2^-9 below
 * 2^-6, else 2^(E-3) in [2^E, 2^(E+1))); the value is rounded to a multiple
 * of that spacing, an even multiple on a tie (the code's last bit), and the
 * multiple is written back as exponent and fraction. */
static uint8_t encode_e4m3(float v)
{
    if (isnan(v))
        return 0x7f;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7e; /* 448 = 1.75 * 2^8, the largest finite value */
    double spacing;
    if (a < ldexp(1.0, -6)) {
        spacing = ldexp(1.0, -9);
    } else {
        int e;
        frexp(a, &e); /* a in [2^(e-1), 2^e) */
        spacing = ldexp(1.0, (e - 1) - 3);
    }
    double q = nearbyint(a / spacing); /* ties to even in the default mode */
    double val = q * spacing;
    if (val == 0.0)
        return sign;
    if (val < ldexp(1.0, -6))
        return sign | (uint8_t)(val / ldexp(1.0, -9));
    int e;
    frexp(val, &e);
    int E = e - 1; /* val in [2^E, 2^(E+1)) */
    int mant = (int)(val / ldexp(1.0, E - 3)) - 8;
    return sign | (uint8_t)(((E + 7) << 3) | mant);
}

/* codes[i] = e4m3(float(x[i]) * inv_scale), x 16-bit (dtype). */
void oracle_quantize_e4m3(uint8_t *codes, const uint16_t *x, int64_t n, int dtype,
                          float inv_scale)
{
    for (int64_t i = 0; i < n; ++i) {
        float v = (float)decode(x[i], dtype);
        float scaled = v * inv_scale;
        codes[i] = encode_e4m3(scaled);
    }
}

/* ---- slot mapping ([GAO] §1.5) ---------------------------------------- */

/* Slot of one token: logical block = position / block_size, offset =
 * position % block_size, physical block = block_table[logical block],
 * slot = physical block * block_size + offset. */
int64_t oracle_slot_for_position(const int32_t *block_table_row,
                                 int64_t position, int block_size)
{
    int64_t logical_block = position / block_size;
    int64_t offset = position % block_size;
    int64_t physical_block = block_table_row[logical_block];
    return physical_block * block_size + offset;
}

/* Slots for num_tokens tokens; token t belongs to sequence token_seq[t] at
 * position token_pos[t].  block_tables is [num_seqs][max_blocks_per_seq]. */
void oracle_slot_mapping(int64_t *slots, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *token_seq,
                         const int32_t *token_pos, int num_tokens,
                         int block_size)
{
    for (int t = 0; t < num_tokens; ++t) {
        const int32_t *row =
            block_tables + (int64_t)token_seq[t] * max_blocks_per_seq;
        slots[t] = oracle_slot_for_position(row, token_pos[t], block_size);
    }
}

/* ---- reshape_and_cache ([GAO] §1.5, [FEI] "Block Table 实现") ----------- */

/* key/value: [num_tokens][num_kv_heads][head_dim] 16-bit elements.
 * key_cache/value_cache: [num_blocks][block_size][num_kv_heads][head_dim].
 * Token t is stored at block slot/block_size, row slot%block_size. */
void oracle_reshape_and_cache(const uint16_t *key, const uint16_t *value,
                              uint16_t *key_cache, uint16_t *value_cache,
                              const int64_t *slot_mapping, int num_tokens,
                              int num_kv_heads, int head_dim, int block_size)
{
    int64_t row_elems = (int64_t)num_kv_heads * head_dim;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        int64_t dst = (block * block_size + offset) * row_elems;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int i = 0; i < head_dim; ++i) {
                int64_t src_i = (int64_t)t * row_elems + (int64_t)h * head_dim + i;
                int64_t dst_i = dst + (int64_t)h * head_dim + i;
                key_cache[dst_i] = key[src_i];
                value_cache[dst_i] = value[src_i];
            }
        }
    }
}

/* FP8 pools: token t's K/V rows quantised with the per-tensor inverse
 * scales and stored at its slot; negative slots are skipped. */
void oracle_reshape_and_cache_fp8(const uint16_t *key, const uint16_t *value,
                                  uint8_t *key_cache, uint8_t *value_cache,
                                  const int64_t *slot_mapping, int num_tokens,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int dtype, float k_inv_scale, float v_inv_scale)
{
    int64_t row_elems = (int64_t)num_kv_heads * head_dim;
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        int64_t dst = (block * block_size + offset) * row_elems;
        oracle_quantize_e4m3(key_cache + dst, key + (int64_t)t * row_elems, row_elems,
                             dtype, k_inv_scale);
        oracle_quantize_e4m3(value_cache + dst, value + (int64_t)t * row_elems, row_elems,
                             dtype, v_inv_scale);
    }
}

/* ---- copy_blocks ([LAKE] §3.2, the "copy the contents" step) ----------- */

/* block_mapping: [num_pairs][2] = (src, dst).  Pairs are applied in order. */
void oracle_copy_blocks(uint16_t *key_cache, uint16_t *value_cache,
                        const int32_t *block_mapping, int num_pairs,
                        int block_size, int num_kv_heads, int head_dim)
{
    int64_t block_elems = (int64_t)block_size * num_kv_heads * head_dim;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t src = block_mapping[2 * p];
        int64_t dst = block_mapping[2 * p + 1];
        for (int64_t i = 0; i < block_elems; ++i) {
            key_cache[dst * block_elems + i] = key_cache[src * block_elems + i];
            value_cache[dst * block_elems + i] = value_cache[src * block_elems + i];
        }
    }
}

/* ---- paged decode attention ([GAO] §1.6) ------------------------------- */

/* Address (element index) of the K or V row for token `position` of the
 * sequence whose block table row is `row`, KV head `kv_head`. */
static int64_t cache_row(const int32_t *row, int64_t position, int kv_head,
                         int num_kv_heads, int head_dim, int block_size)
{
    int64_t physical_block = row[position / block_size];
    int64_t offset = position % block_size;
    return ((physical_block * block_size + offset) * num_kv_heads + kv_head) *
           (int64_t)head_dim;
}

/* Scores scale * q . k_p for positions p in [p0, p1) of one (seq, head). */
static void scores_for_range(double *scores, const uint16_t *q_row,
                             const uint16_t *key_cache, const int32_t *row,
                             int64_t p0, int64_t p1, int kv_head,
                             int num_kv_heads, int head_dim, int block_size,
                             double scale, int dtype)
{
    for (int64_t p = p0; p < p1; ++p) {
        int64_t k = cache_row(row, p, kv_head, num_kv_heads, head_dim, block_size);
        double dot = 0.0;
        for (int i = 0; i < head_dim; ++i)
            dot += decode(q_row[i], dtype) * decode(key_cache[k + i], dtype);
        scores[p - p0] = scale * dot;
    }
}

/* Softmax-weighted sum over positions [p0, p1): writes m = max score,
 * l = sum exp(score - m), and out[i] = sum exp(score - m) v[i] / l. */
static void attend_range(double *out, double *m_out, double *l_out,
                         const uint16_t *q_row, const uint16_t *key_cache,
                         const uint16_t *value_cache, const int32_t *row,
                         int64_t p0, int64_t p1, int kv_head, int num_kv_heads,
                         int head_dim, int block_size, double scale, int dtype)
{
    int64_t n = p1 - p0;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    scores_for_range(scores, q_row, key_cache, row, p0, p1, kv_head,
                     num_kv_heads, head_dim, block_size, scale, dtype);
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (scores[j] > m)
            m = scores[j];
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        scores[j] = exp(scores[j] - m); /* now the unnormalised weight */
        l += scores[j];
    }
    for (int i = 0; i < head_dim; ++i)
        out[i] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        int64_t v = cache_row(row, p0 + j, kv_head, num_kv_heads, head_dim,
                              block_size);
        for (int i = 0; i < head_dim; ++i)
            out[i] += scores[j] * decode(value_cache[v + i], dtype);
    }
    for (int i = 0; i < head_dim; ++i)
        out[i] /= l;
    *m_out = m;
    *l_out = l;
    free(scores);
}

/* out: [num_seqs][num_heads][head_dim] doubles.  query: [num_seqs]
 * [num_heads][head_dim].  block_tables: [num_seqs][max_blocks_per_seq].
 * If seq_subset is non-NULL only the n_subset listed sequences are
 * computed; other output rows are left untouched. */
void oracle_paged_attention(double *out, const uint16_t *query,
                            const uint16_t *key_cache,
                            const uint16_t *value_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs,
                            int num_heads, int num_kv_heads, int head_dim,
                            int block_size, double scale, int dtype,
                            const int32_t *seq_subset, int n_subset)
{
    int group = num_heads / num_kv_heads;
    int count = seq_subset ? n_subset : num_seqs;
    for (int c = 0; c < count; ++c) {
        int s = seq_subset ? seq_subset[c] : c;
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        int64_t ctx = context_lens[s];
        for (int h = 0; h < num_heads; ++h) {
            double *o = out + ((int64_t)s * num_heads + h) * head_dim;
            if (ctx <= 0) {
                for (int i = 0; i < head_dim; ++i)
                    o[i] = 0.0;
                continue;
            }
            const uint16_t *q_row = query + ((int64_t)s * num_heads + h) * head_dim;
            double m, l;
            attend_range(o, &m, &l, q_row, key_cache, value_cache, row, 0, ctx,
                         h / group, num_kv_heads, head_dim, block_size, scale,
                         dtype);
        }
    }
}

/* ---- chunked prefill over the paged pool ([GAO] §2.4, §2.5) ----------- */

/* A batch row of sequence s is one of its q_len newest tokens (a prompt
 * chunk, or q_len = 1 for a decode request in the same mixed batch), whose
 * K/V are already in the cache.  Reading (the pages show prefill processing
 * a prompt's tokens in parallel and decode seeing only earlier tokens, and
 * give no mask): row i of the chunk is the token at position
 * pos = context_len - q_len + i and attends positions [0, pos], i.e. it is
 * exactly a decode query over the first pos + 1 tokens.
 *
 * out: [num_rows][num_heads][head_dim] doubles; query: [num_rows][num_heads]
 * [head_dim] with num_rows = query_start[num_seqs]; sequence s owns rows
 * [query_start[s], query_start[s+1]).  A row whose position is negative
 * (a chunk longer than its context) attends nothing and gets zeros. */
void oracle_prefill_attention(double *out, const uint16_t *query,
                              const uint16_t *key_cache, const uint16_t *value_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *query_start, const int32_t *context_lens,
                              int num_seqs, int num_heads, int num_kv_heads,
                              int head_dim, int block_size, double scale, int dtype)
{
    int group = num_heads / num_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        int64_t q0 = query_start[s], q_len = query_start[s + 1] - query_start[s];
        int64_t ctx = context_lens[s];
        for (int64_t i = 0; i < q_len; ++i) {
            int64_t pos = ctx - q_len + i;
            for (int h = 0; h < num_heads; ++h) {
                int64_t r = (q0 + i) * num_heads + h;
                double *o = out + r * head_dim;
                if (pos < 0) {
                    for (int k = 0; k < head_dim; ++k)
                        o[k] = 0.0;
                    continue;
                }
                double m, l;
                attend_range(o, &m, &l, query + r * head_dim, key_cache, value_cache, row,
                             0, pos + 1, h / group, num_kv_heads, head_dim, block_size,
                             scale, dtype);
            }
        }
    }
}

/* Paged attention over FP8 pools: K and V are the dequantised codes
 * (code value * k_scale, * v_scale); everything else as above. */
void oracle_paged_attention_fp8(double *out, const uint16_t *query,
                                const uint8_t *key_cache, const uint8_t *value_cache,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, int num_seqs, int num_heads,
                                int num_kv_heads, int head_dim, int block_size,
                                double scale, int dtype, double k_scale, double v_scale,
                                const int32_t *seq_subset, int n_subset)
{
    int group = num_heads / num_kv_heads;
    int count = seq_subset ? n_subset : num_seqs;
    for (int c = 0; c < count; ++c) {
        int s = seq_subset ? seq_subset[c] : c;
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        int64_t ctx = context_lens[s];
        for (int h = 0; h < num_heads; ++h) {
            double *o = out + ((int64_t)s * num_heads + h) * head_dim;
            for (int i = 0; i < head_dim; ++i)
                o[i] = 0.0;
            if (ctx <= 0)
                continue;
            const uint16_t *q_row = query + ((int64_t)s * num_heads + h) * head_dim;
            int kh = h / group;
            double *scores = (double *)malloc(sizeof(double) * (size_t)ctx);
            double m = -INFINITY;
            for (int64_t p = 0; p < ctx; ++p) {
                int64_t k = cache_row(row, p, kh, num_kv_heads, head_dim, block_size);
                double dot = 0.0;
                for (int i = 0; i < head_dim; ++i)
                    dot += decode(q_row[i], dtype) * (decode_e4m3(key_cache[k + i]) * k_scale);
                scores[p] = scale * dot;
                if (scores[p] > m)
                    m = scores[p];
            }
            double l = 0.0;
            for (int64_t p = 0; p < ctx; ++p) {
                scores[p] = exp(scores[p] - m);
                l += scores[p];
            }
            for (int64_t p = 0; p < ctx; ++p) {
                int64_t v = cache_row(row, p, kh, num_kv_heads, head_dim, block_size);
                for (int i = 0; i < head_dim; ++i)
                    o[i] += scores[p] * (decode_e4m3(value_cache[v + i]) * v_scale);
            }
            for (int i = 0; i < head_dim; ++i)
                o[i] /= l;
            free(scores);
        }
    }
}

/* Chunked prefill over FP8 pools: oracle_prefill_attention with K and V the
 * dequantised codes (code value * k_scale, * v_scale).  Row i of sequence
 * s's chunk sits at pos = context_len - q_len + i and attends [0, pos]; a
 * negative position gives a zero row. */
void oracle_prefill_attention_fp8(double *out, const uint16_t *query,
                                  const uint8_t *key_cache, const uint8_t *value_cache,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *query_start, const int32_t *context_lens,
                                  int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int block_size, double scale, int dtype, double k_scale,
                                  double v_scale)
{
    int group = num_heads / num_kv_heads;
    for (int s = 0; s < num_seqs; ++s) {
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        int64_t q0 = query_start[s], q_len = query_start[s + 1] - query_start[s];
        int64_t ctx = context_lens[s];
        for (int64_t i = 0; i < q_len; ++i) {
            int64_t pos = ctx - q_len + i;
            for (int h = 0; h < num_heads; ++h) {
                int64_t r = (q0 + i) * num_heads + h;
                double *o = out + r * head_dim;
                for (int k = 0; k < head_dim; ++k)
                    o[k] = 0.0;
                if (pos < 0)
                    continue;
                const uint16_t *q_row = query + r * head_dim;
                int kh = h / group;
                int64_t n = pos + 1;
                double *scores = (double *)malloc(sizeof(double) * (size_t)n);
                double m = -INFINITY;
                for (int64_t p = 0; p < n; ++p) {
                    int64_t k = cache_row(row, p, kh, num_kv_heads, head_dim, block_size);
                    double dot = 0.0;
                    for (int c = 0; c < head_dim; ++c)
                        dot += decode(q_row[c], dtype) *
                               (decode_e4m3(key_cache[k + c]) * k_scale);
                    scores[p] = scale * dot;
                    if (scores[p] > m)
                        m = scores[p];
                }
                double l = 0.0;
                for (int64_t p = 0; p < n; ++p) {
                    scores[p] = exp(scores[p] - m);
                    l += scores[p];
                }
                for (int64_t p = 0; p < n; ++p) {
                    int64_t v = cache_row(row, p, kh, num_kv_heads, head_dim, block_size);
                    for (int c = 0; c < head_dim; ++c)
                        o[c] += scores[p] * (decode_e4m3(value_cache[v + c]) * v_scale);
                }
                for (int c = 0; c < head_dim; ++c)
                    o[c] /= l;
                free(scores);
            }
        }
    }
}

/* Block copies of 1-byte (FP8) pools, pairs applied in order. */
void oracle_copy_blocks_u8(uint8_t *key_cache, uint8_t *value_cache,
                           const int32_t *block_mapping, int num_pairs, int block_size,
                           int num_kv_heads, int head_dim)
{
    int64_t block_elems = (int64_t)block_size * num_kv_heads * head_dim;
    for (int p = 0; p < num_pairs; ++p) {
        int64_t src = block_mapping[2 * p];
        int64_t dst = block_mapping[2 * p + 1];
        memcpy(key_cache + dst * block_elems, key_cache + src * block_elems,
               (size_t)block_elems);
        memcpy(value_cache + dst * block_elems, value_cache + src * block_elems,
               (size_t)block_elems);
    }
}

/* Softmax weights of one (seq, head) over its context: weights[p] for
 * p in [0, context_lens[seq]).  Used to check that rows sum to one. */
void oracle_attention_weights(double *weights, const uint16_t *query,
                              const uint16_t *key_cache,
                              const int32_t *block_tables,
                              int max_blocks_per_seq,
                              const int32_t *context_lens, int seq, int head,
                              int num_heads, int num_kv_heads, int head_dim,
                              int block_size, double scale, int dtype)
{
    int group = num_heads / num_kv_heads;
    const int32_t *row = block_tables + (int64_t)seq * max_blocks_per_seq;
    int64_t ctx = context_lens[seq];
    if (ctx <= 0)
        return;
    const uint16_t *q_row = query + ((int64_t)seq * num_heads + head) * head_dim;
    scores_for_range(weights, q_row, key_cache, row, 0, ctx, head / group,
                     num_kv_heads, head_dim, block_size, scale, dtype);
    double m = -INFINITY;
    for (int64_t p = 0; p < ctx; ++p)
        if (weights[p] > m)
            m = weights[p];
    double l = 0.0;
    for (int64_t p = 0; p < ctx; ++p) {
        weights[p] = exp(weights[p] - m);
        l += weights[p];
    }
    for (int64_t p = 0; p < ctx; ++p)
        weights[p] /= l;
}

/* ---- split-context partition pass and merge ---------------------------- */

/* Number of partitions of partition_size tokens covering a context. */
int oracle_num_partitions(int64_t context_len, int partition_size)
{
    if (context_len <= 0)
        return 0;
    return (int)((context_len + partition_size - 1) / partition_size);
}

/* Per (seq, head, partition j): part_m, part_l [num_seqs][num_heads]
 * [max_partitions] and part_o [num_seqs][num_heads][max_partitions]
 * [head_dim].  Entries past a sequence's partition count are untouched. */
void oracle_partition_pass(double *part_m, double *part_l, double *part_o,
                           const uint16_t *query, const uint16_t *key_cache,
                           const uint16_t *value_cache,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int head_dim,
                           int block_size, double scale, int dtype,
                           int partition_size, int max_partitions,
                           const int32_t *seq_subset, int n_subset)
{
    int group = num_heads / num_kv_heads;
    int count = seq_subset ? n_subset : num_seqs;
    for (int c = 0; c < count; ++c) {
        int s = seq_subset ? seq_subset[c] : c;
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        int64_t ctx = context_lens[s];
        int nparts = oracle_num_partitions(ctx, partition_size);
        for (int h = 0; h < num_heads; ++h) {
            const uint16_t *q_row = query + ((int64_t)s * num_heads + h) * head_dim;
            for (int j = 0; j < nparts && j < max_partitions; ++j) {
                int64_t p0 = (int64_t)j * partition_size;
                int64_t p1 = p0 + partition_size;
                if (p1 > ctx)
                    p1 = ctx;
                int64_t idx = ((int64_t)s * num_heads + h) * max_partitions + j;
                attend_range(part_o + idx * head_dim, &part_m[idx], &part_l[idx],
                             q_row, key_cache, value_cache, row, p0, p1, h / group,
                             num_kv_heads, head_dim, block_size, scale, dtype);
            }
        }
    }
}

/* Merge the partials of each (seq, head): M = max_j m_j,
 * w_j = l_j exp(m_j - M), out = sum_j w_j o_j / sum_j w_j.  A sequence with
 * no partition gets a zero row. */
void oracle_partition_merge(double *out, const double *part_m,
                            const double *part_l, const double *part_o,
                            const int32_t *num_partitions, int num_seqs,
                            int num_heads, int head_dim, int max_partitions)
{
    for (int s = 0; s < num_seqs; ++s) {
        for (int h = 0; h < num_heads; ++h) {
            double *o = out + ((int64_t)s * num_heads + h) * head_dim;
            int64_t base = ((int64_t)s * num_heads + h) * max_partitions;
            int n = num_partitions[s];
            for (int i = 0; i < head_dim; ++i)
                o[i] = 0.0;
            if (n <= 0)
                continue;
            double big_m = -INFINITY;
            for (int j = 0; j < n; ++j)
                if (part_m[base + j] > big_m)
                    big_m = part_m[base + j];
            double wsum = 0.0;
            for (int j = 0; j < n; ++j) {
                double w = part_l[base + j] * exp(part_m[base + j] - big_m);
                wsum += w;
                for (int i = 0; i < head_dim; ++i)
                    o[i] += w * part_o[(base + j) * head_dim + i];
            }
            for (int i = 0; i < head_dim; ++i)
                o[i] /= wsum;
        }
    }
}
