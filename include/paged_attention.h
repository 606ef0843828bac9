/*
 * paged_attention.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode
 * library (libpaged_attention.so).
 *
 * The operations are those of a vLLM-style serving engine's decode step as
 * the following web pages describe them (cited by title and section):
 *   [GAO]  "PagedAttention & Continuous Batching" (gaoleia.github.io,
 *          2026-01-25): §1.3 physical block, §1.4 block table, §1.5 slot
 *          mapping, §1.6 paged attention, §2.4 decode is memory-bound.
 *   [FEI]  "vLLM 架构详解: PagedAttention、Continuous Batching 与生产级推理优化"
 *          (feifeigd.github.io): "Block Table 实现", "共享前缀的 Block 复用".
 *   [LAKE] "vLLM源码解析(二): 调度系统与PagedAttention实现"
 *          (lakecityint.com): §3.2 copy-on-write.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned DEVICE memory, dense, row-major (last index
 *    fastest), unless a parameter says "host".  The library allocates
 *    nothing and keeps no pointer after a call returns.
 *  - 16-bit elements (pa_dtype) are fp16 or bf16.  Tensor base addresses
 *    must be 16-byte aligned.
 *  - KV pool layout (token-major, separate K and V pools):
 *        key_cache, value_cache : [num_blocks][block_size][num_kv_heads][head_dim]
 *    Block b, row r holds the K (or V) vectors of all KV heads for the token
 *    stored in slot b * block_size + r ([GAO] §1.3, §1.5).
 *  - Block tables: int32 [num_seqs][max_blocks_per_seq]; entry i of row s is
 *    the physical block holding tokens i*block_size .. i*block_size +
 *    block_size - 1 of sequence s ([GAO] §1.4).  Entries past a sequence's
 *    last block are never read.
 *  - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  They never synchronise the device.
 *  - Host-visible argument errors return a status before anything is
 *    launched.  Device-resident indices (slots, table entries, block pairs,
 *    context lengths) are checked on the device: an out-of-range index is
 *    skipped (never dereferenced) and, when `error_word` is non-NULL, a
 *    PA_DEVERR_* bit is OR-ed into that device int32.  No kernel traps.
 *  - A launch failure returns PA_ERR_CUDA; pa_last_cuda_error() names it.
 */
#ifndef PAGED_ATTENTION_H
#define PAGED_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misalignment, ... */
    PA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head_dim, block_size, group) */
    PA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    PA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    PA_ERR_OUT_OF_BLOCKS = 5, /* block manager: not enough free physical blocks */
    PA_ERR_TABLE_FULL = 6    /* block manager: a table would pass max_blocks_per_seq */
} pa_status;

typedef enum {
    PA_F16 = 0,      /* IEEE binary16 */
    PA_BF16 = 1,     /* bfloat16 */
    PA_FP8_E4M3 = 2  /* 1-byte e4m3 KV codes (pools only; see the FP8 calls) */
} pa_dtype;

/* Bits OR-ed into the optional device error word. */
#define PA_DEVERR_SLOT_RANGE    0x01 /* slot >= num_blocks * block_size */
#define PA_DEVERR_BLOCK_RANGE   0x02 /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_PAIR_RANGE    0x04 /* copy pair block outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT_RANGE 0x08 /* context_len < 0, > max_context_len or past the table */
#define PA_DEVERR_TOKEN_RANGE   0x10 /* token's sequence or position outside its table */
#define PA_DEVERR_TIMEOUT       0x20 /* a bounded wait on staged data gave up */
#define PA_DEVERR_PREFIX_PLAN   0x40 /* prefix plan inconsistent with the tables or contexts */
#define PA_DEVERR_QUERY_RANGE   0x80 /* FP8 pools: a bf16 query element beyond the fp16 range */

/*
 * pa_slot_mapping -- [GAO] §1.5.  For every token t, writes
 *     slot_mapping[t] = block_tables[s][p / block_size] * block_size
 *                       + p % block_size,   s = token_seq[t], p = token_pos[t].
 * token_seq, token_pos: int32 [num_tokens].  slot_mapping: int32 [num_tokens]
 * (output).  A token whose sequence is outside [0, num_seqs), whose position
 * is negative or past max_blocks_per_seq * block_size, or whose table entry
 * is outside [0, num_blocks) gets slot -1 and sets PA_DEVERR_TOKEN_RANGE or
 * PA_DEVERR_BLOCK_RANGE.  num_tokens == 0 is a no-op.
 */
PA_API pa_status pa_slot_mapping(int32_t *slot_mapping, const int32_t *block_tables,
                          int max_blocks_per_seq, const int32_t *token_seq,
                          const int32_t *token_pos, int num_tokens,
                          int num_seqs, int block_size, int num_blocks,
                          int32_t *error_word, void *stream);

/*
 * pa_reshape_and_cache -- [GAO] §1.5, [FEI] "Block Table 实现".  Copies the
 * K and V vectors of num_tokens new tokens into the pools at their slots:
 *     key_cache[slot / block_size][slot % block_size][h][:] = key[t][h][:]
 * (same for value).  key, value: [num_tokens][num_kv_heads][head_dim].
 * slot_mapping: int32 [num_tokens]; slot < 0 means "skip this token";
 * slot >= num_blocks * block_size is skipped and sets PA_DEVERR_SLOT_RANGE.
 * Bytes are copied verbatim.  Two tokens with the same slot race.
 */
PA_API pa_status pa_reshape_and_cache(const void *key, const void *value,
                               void *key_cache, void *value_cache,
                               const int32_t *slot_mapping, int num_tokens,
                               int num_blocks, int block_size, int num_kv_heads,
                               int head_dim, pa_dtype dtype,
                               int32_t *error_word, void *stream);

/*
 * pa_reshape_and_cache_fp8 -- the FP8 KV cache of the deployment options in
 * [FEI] ("--kv-cache-dtype fp8"): as pa_reshape_and_cache, but the pools
 * hold 1-byte e4m3 codes (OCP e4m3: bias 7, no infinities, largest finite
 * 448) with one scale per pool.  For every element
 *     code = e4m3(float(x) * inv),   inv = 1.0f / scale (fp32),
 * the product rounded once in fp32, then to the nearest e4m3 value (ties to
 * even), finite values beyond +-448 saturating; the cached value stands for
 * e4m3(code) * scale.  key, value: [num_tokens][num_kv_heads][head_dim] of
 * src_dtype (PA_F16 or PA_BF16); key_cache, value_cache: uint8
 * [num_blocks][block_size][num_kv_heads][head_dim].  Scales must be finite
 * and > 0.  Slot rules as pa_reshape_and_cache.
 */
PA_API pa_status pa_reshape_and_cache_fp8(const void *key, const void *value,
                                          void *key_cache, void *value_cache,
                                          const int32_t *slot_mapping, int num_tokens,
                                          int num_blocks, int block_size, int num_kv_heads,
                                          int head_dim, pa_dtype src_dtype, float k_scale,
                                          float v_scale, int32_t *error_word, void *stream);

/*
 * pa_slot_mapping_and_cache, pa_slot_mapping_and_cache_fp8 -- one launch for
 * the two steps before attention: the slot of each new token as
 * pa_slot_mapping computes it ([GAO] §1.5; same checks, slot -1 and the same
 * error flags for a bad token or table entry), stored to slot_mapping, and
 * its K/V written there as pa_reshape_and_cache / pa_reshape_and_cache_fp8
 * write them (same layouts, dtypes, scales and rules).  The pools and
 * slot_mapping end bit-identical to the two calls made in turn.
 */
PA_API pa_status pa_slot_mapping_and_cache(int32_t *slot_mapping, const int32_t *block_tables,
                                           int max_blocks_per_seq, const int32_t *token_seq,
                                           const int32_t *token_pos, int num_tokens,
                                           int num_seqs, const void *key, const void *value,
                                           void *key_cache, void *value_cache, int num_blocks,
                                           int block_size, int num_kv_heads, int head_dim,
                                           pa_dtype dtype, int32_t *error_word, void *stream);

PA_API pa_status pa_slot_mapping_and_cache_fp8(int32_t *slot_mapping,
                                               const int32_t *block_tables,
                                               int max_blocks_per_seq,
                                               const int32_t *token_seq,
                                               const int32_t *token_pos, int num_tokens,
                                               int num_seqs, const void *key,
                                               const void *value, void *key_cache,
                                               void *value_cache, int num_blocks,
                                               int block_size, int num_kv_heads, int head_dim,
                                               pa_dtype src_dtype, float k_scale,
                                               float v_scale, int32_t *error_word,
                                               void *stream);

/*
 * pa_copy_blocks -- the "copy the contents" step of copy-on-write
 * ([LAKE] §3.2).  block_mapping: int32 [num_pairs][2] = (src, dst); for every
 * pair, K block dst := K block src and V block dst := V block src (whole
 * blocks of block_size * num_kv_heads * head_dim elements).  No block may be
 * both a source and a destination, and destinations must be distinct;
 * otherwise the result is unspecified.  A pair with a block outside
 * [0, num_blocks) is skipped and sets PA_DEVERR_PAIR_RANGE.  dtype gives the
 * element size: 2 bytes for PA_F16 / PA_BF16, 1 byte for PA_FP8_E4M3 pools.
 */
PA_API pa_status pa_copy_blocks(void *key_cache, void *value_cache,
                         const int32_t *block_mapping, int num_pairs,
                         int num_blocks, int block_size, int num_kv_heads,
                         int head_dim, pa_dtype dtype, int32_t *error_word,
                         void *stream);

/*
 * pa_decode_workspace_bytes -- bytes of device workspace pa_decode_attention
 * needs for these sizes (0 when partition_size == 0 or every context fits in
 * one partition).  Layout, with P = ceil(max_context_len / partition_size)
 * and every region starting on a 256-byte boundary, in this order:
 *     int32 counters[max(2^18, num_seqs * num_kv_heads)]  arrival counters
 *     float part_m[num_seqs][num_heads][P]            partition stabiliser m_j
 *     float part_l[num_seqs][num_heads][P]            sum_p exp(score_p - m_j)
 *     float part_o[num_seqs][num_heads][P][head_dim]  partition output / l_j
 * score_p = scale * q . k_p (natural-log units).  m_j is a stabiliser: the
 * partition's log-sum-exp is m_j + log(l_j).  Partials are written only for
 * sequences that span more than one partition.  The counters must hold
 * zeros before a workspace is first used (cudaMemsetAsync once after
 * allocating it); every call leaves them at zero.  The counter region has
 * the same size for every call with num_seqs * num_kv_heads <= 2^18, so one
 * workspace, zeroed once, serves calls of any such sizes; a call with more
 * needs its whole counter region zeroed first.  Returns 0 for invalid sizes.
 */
PA_API size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int max_context_len,
                                 int partition_size);

/*
 * pa_decode_attention -- paged decode attention, [GAO] §1.6 and §2.4.
 * For every sequence s and query head h (KV head kh = h / (num_heads /
 * num_kv_heads), contiguous groups):
 *     score_p = scale * q[s][h] . K[p][kh],    p in [0, context_lens[s])
 *     out[s][h][:] = sum_p softmax(score)_p * V[p][kh][:]
 * where K[p], V[p] are read from physical block block_tables[s][p /
 * block_size], row p % block_size.  Accumulation is fp32 (online softmax
 * with a running max and sum); the output is rounded to nearest even.
 *   out, query   : [num_seqs][num_heads][head_dim], dtype.
 *   context_lens : int32 [num_seqs] (device); max_context_len (host) must be
 *                  >= every context_lens[s] (larger values are clipped and
 *                  flagged PA_DEVERR_CONTEXT_RANGE).  context 0 gives a zero row.
 *   partition_size: 0 = single pass (one work unit per sequence and KV
 *                  head); otherwise a multiple of 16 tokens: contexts are
 *                  split into partitions of that many tokens.  The partition
 *                  pass writes a partial (m, l, o) per partition to the
 *                  workspace and merges a sequence's partials by
 *                  log-sum-exp weights l_j * exp(m_j - max m): in the same
 *                  kernel, as soon as the last of them is written (an
 *                  arrival counter per sequence and KV head), for sequences
 *                  of up to 8 partitions; in a reduce kernel queued behind
 *                  it by this call for longer ones.  A sequence that fits
 *                  one partition is written by the pass directly.
 *   workspace    : device, 256-byte aligned, >= pa_decode_workspace_bytes(...)
 *                  bytes, its counter region zeroed before first use (see
 *                  pa_decode_workspace_bytes); the partial regions need no
 *                  initial contents.  May be NULL when that size is 0.
 *                  Calls sharing one workspace must not overlap.
 * Supported: head_dim 64 or 128; block_size a power of two from 16 to 256;
 * num_heads / num_kv_heads in 1..16; num_blocks * block_size < 2^31.
 */
PA_API pa_status pa_decode_attention(void *out, const void *query,
                              const void *key_cache, const void *value_cache,
                              const int32_t *block_tables,
                              int max_blocks_per_seq,
                              const int32_t *context_lens, int max_context_len,
                              int num_seqs, int num_heads, int num_kv_heads,
                              int head_dim, int block_size, int num_blocks,
                              float scale, int partition_size, void *workspace,
                              size_t workspace_bytes, pa_dtype dtype,
                              int32_t *error_word, void *stream);

/*
 * pa_decode_attention_fp8 -- pa_decode_attention over FP8 pools written by
 * pa_reshape_and_cache_fp8: K and V elements are e4m3 codes standing for
 * e4m3(code) * k_scale and * v_scale.  query and out are dtype (PA_F16 or
 * PA_BF16).  Codes are widened to fp16 and the query is rounded to fp16 for
 * the tensor-core products: a bf16 query element with |q| > 65504 overflows
 * there, and is flagged PA_DEVERR_QUERY_RANGE (its rows' outputs are then
 * not finite); scores and weights
 * accumulate in fp32 as in pa_decode_attention; the V scale is applied to
 * the output.  Workspace, partitions and errors as pa_decode_attention
 * (same workspace size).  Supported: head_dim 64 or 128.
 */
PA_API pa_status pa_decode_attention_fp8(void *out, const void *query, const void *key_cache,
                                         const void *value_cache, const int32_t *block_tables,
                                         int max_blocks_per_seq, const int32_t *context_lens,
                                         int max_context_len, int num_seqs, int num_heads,
                                         int num_kv_heads, int head_dim, int block_size,
                                         int num_blocks, float scale, float k_scale,
                                         float v_scale, int partition_size, void *workspace,
                                         size_t workspace_bytes, pa_dtype dtype,
                                         int32_t *error_word, void *stream);

/*
 * pa_decode_attention_append, pa_decode_attention_append_fp8 -- one decode
 * step in one call: the slot mapping and reshape_and_cache of each running
 * sequence's new token ([GAO] §1.5 and §1.6: the token's K/V go to slot
 * block_table[pos // block_size] * block_size + pos % block_size) fused into
 * pa_decode_attention / pa_decode_attention_fp8.  The new token of sequence
 * s is at position pos = context_lens[s] - 1 (context_lens counts it):
 *   new_key, new_value : [num_seqs][num_kv_heads][head_dim], dtype (16-bit),
 *                        device, 16-byte aligned.
 *   key_cache, value_cache : written at the slot of pos -- the 16-bit rows
 *                        verbatim, or (FP8 pools) the e4m3 codes
 *                        e4m3(x * (1 / k_scale)) / e4m3(x * (1 / v_scale)),
 *                        bit for bit what pa_reshape_and_cache(_fp8) writes.
 *   slot_mapping       : int32 [num_seqs] (device) or NULL: receives each
 *                        sequence's slot (-1 for a context of 0, which
 *                        appends nothing, and for a block outside the pool).
 * Attention then covers positions [0, context_lens[s]): the cached ones
 * from the pools and pos from the new rows as the pools now hold them (for
 * FP8 pools, the codes), so out equals that of pa_slot_mapping +
 * pa_reshape_and_cache(_fp8) + pa_decode_attention(_fp8) on the same inputs
 * up to fp32 rounding order (the new token's term joins the softmax sums in
 * the pass's end-of-partition merge rather than inside a 16-token tile).
 * The block holding pos must belong to sequence s alone (copy-on-write
 * first, as the engine does before any write into a shared block); other
 * arguments, workspace and errors as pa_decode_attention(_fp8).  A table
 * entry of pos outside [0, num_blocks) flags PA_DEVERR_BLOCK_RANGE and
 * nothing is written there.
 */
PA_API pa_status pa_decode_attention_append(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    int partition_size, void *workspace, size_t workspace_bytes, pa_dtype dtype,
    int32_t *error_word, void *stream);

PA_API pa_status pa_decode_attention_append_fp8(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    float k_scale, float v_scale, int partition_size, void *workspace, size_t workspace_bytes,
    pa_dtype dtype, int32_t *error_word, void *stream);

/*
 * pa_prefill_attention -- chunked prefill and mixed batches over the paged
 * pool, [GAO] §2.4 (prefill processes a prompt's tokens in parallel; a batch
 * mixes decode requests of one token with prefill requests of many) and
 * §2.5 (a long prompt is processed in chunks, 512 tokens each).
 * Sequence s brings q_len = query_start[s+1] - query_start[s] query rows:
 * its q_len newest tokens, whose K/V have already been written to the pool
 * (pa_slot_mapping + pa_reshape_and_cache of the same tokens).  Chunk row i
 * is the token at position pos = context_lens[s] - q_len + i and attends
 * positions [0, pos] (reading, the pages give no mask: each token sees
 * itself and the tokens before it, as in decode, which is the q_len = 1
 * case):
 *     out[r][h][:] = sum_{p <= pos} softmax_p(scale * q[r][h] . K[p][kh]) V[p][kh][:]
 * with r = query_start[s] + i and K/V read through block_tables[s] as in
 * pa_decode_attention.
 *   out, query  : [num_tokens][num_heads][head_dim], dtype (PA_F16/PA_BF16).
 *   query_start : int32 [num_seqs + 1] (device), non-decreasing, query_start[0]
 *                 = 0 and query_start[num_seqs] = num_tokens (host).
 *   context_lens: int32 [num_seqs] (device), tokens in the pool for s
 *                 including its chunk; values outside [0, max_context_len] or
 *                 past the table are clipped and flagged
 *                 PA_DEVERR_CONTEXT_RANGE.  A row whose position is negative
 *                 (chunk longer than the context) gets a zero row.
 * scale must be positive (PA_ERR_INVALID_ARG otherwise).  Accumulation fp32
 * (online softmax), output rounded to nearest even.  No workspace.
 * Supported: as pa_decode_attention (FP8 pools: pa_prefill_attention_fp8).
 */
PA_API pa_status pa_prefill_attention(void *out, const void *query, const void *key_cache,
                                      const void *value_cache, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *query_start,
                                      const int32_t *context_lens, int max_context_len,
                                      int num_seqs, int num_tokens, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, float scale, pa_dtype dtype,
                                      int32_t *error_word, void *stream);

/*
 * pa_prefill_attention_fp8 -- pa_prefill_attention over FP8 pools written by
 * pa_reshape_and_cache_fp8 (K and V elements are e4m3 codes standing for
 * e4m3(code) * k_scale and * v_scale), as pa_decode_attention_fp8 is to
 * pa_decode_attention: the tensor-core tiles take the codes widened to fp16
 * (exact) and the query rounded to fp16 (a bf16 query element with |q| >
 * 65504 is flagged PA_DEVERR_QUERY_RANGE and its rows are not finite); k_scale
 * joins the softmax scale, v_scale multiplies the output.  query and out are
 * dtype (PA_F16 or PA_BF16); k_scale and v_scale must be positive and finite
 * (PA_ERR_INVALID_ARG).  Limits (head_dim 64 or 128 among them), other
 * arguments, rows and errors as pa_prefill_attention.
 */
PA_API pa_status pa_prefill_attention_fp8(void *out, const void *query, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          int max_blocks_per_seq, const int32_t *query_start,
                                          const int32_t *context_lens, int max_context_len,
                                          int num_seqs, int num_tokens, int num_heads,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float scale, float k_scale,
                                          float v_scale, pa_dtype dtype, int32_t *error_word,
                                          void *stream);

/*
 * Prefix plan -- which sequences of a decode batch share leading physical
 * blocks ([FEI] "共享前缀的 Block 复用": block tables that name the same
 * physical blocks for a common prefix, the blocks' reference counts > 1).
 * One int32 array, laid out as
 *     seq_prefix_len[num_seqs]      shared tokens of s's group, 0 if none
 *     group_start[num_groups + 1]   members of group g: [group_start[g], group_start[g+1])
 *     group_prefix_len[num_groups]  shared tokens L_g (a multiple of the block size)
 *     group_members[num_members]    sequence ids, group by group
 * (pa_prefix_plan_ints gives its length).  The first member of a group is
 * its leader; every member's first L_g / block_size table entries equal the
 * leader's, and L_g < every member's context length.
 */
PA_API size_t pa_prefix_plan_ints(int num_seqs, int num_groups, int num_members);

/*
 * pa_plan_prefix_groups -- host (CPU) planner of the prefix plan above, from
 * host copies of the block tables [num_seqs][max_blocks_per_seq] and context
 * lengths.  Sequences are ordered by their table rows; runs of sequences
 * sharing leading blocks become groups, each with the longest prefix all its
 * members share, split further where a smaller group with a longer prefix
 * saves more block reads ((members - 1) * L).  A shared prefix stops before
 * each member's last token and is at least min_shared_blocks blocks long.
 *   plan: host int32, capacity plan_capacity ints (3 * num_seqs + 1 always
 *         suffices); num_groups, num_members: out.
 * Deterministic; allocates only host memory it frees.  Returns
 * PA_ERR_INVALID_ARG on bad sizes or pointers, PA_ERR_WORKSPACE when the
 * plan does not fit plan_capacity.
 */
PA_API pa_status pa_plan_prefix_groups(const int32_t *block_tables, int max_blocks_per_seq,
                                       const int32_t *context_lens, int num_seqs,
                                       int block_size, int min_shared_blocks, int32_t *plan,
                                       size_t plan_capacity, int *num_groups,
                                       int *num_members);

/*
 * pa_cascade_workspace_bytes -- workspace of pa_decode_attention_cascade:
 * the layout of pa_decode_workspace_bytes with P = 1 + ceil(max_context_len
 * / partition_size) (1 + 1 for partition_size 0) partials per (sequence,
 * head); the first partials of a grouped sequence are its shared prefix's.
 * Counter region as for pa_decode_workspace_bytes (zero before first use).
 */
PA_API size_t pa_cascade_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                         int head_dim, int max_context_len,
                                         int partition_size);

/*
 * pa_decode_attention_cascade -- prefix-aware decode: the result of
 * pa_decode_attention, computed so that each group's shared prefix is read
 * from HBM once for all of its members instead of once per member.
 *   1. prefix pass: for every group g and KV head, the decode queries of all
 *      members (times the G query heads) attend the prefix [0, L_g), read
 *      through the leader's table, with tcgen05 tensor-core tiles of 128
 *      query rows; each (member, head) gets partials 0 .. ceil(L_g / P) - 1
 *      = (m, l, o) in the workspace, one per prefix partition of P =
 *      partition_size tokens.
 *   2. partition pass: every sequence attends its own tokens [L, ctx) (L = 0
 *      outside any group) in partitions of partition_size tokens (0: one).
 *   3. merge: log-sum-exp merge of each grouped or split sequence's
 *      partials, by whichever of the two passes stores the sequence's last
 *      partial (an arrival counter per sequence and KV head in the
 *      workspace), for sequences of up to 8 partials; by a reduce kernel
 *      queued behind the passes for longer ones.  Ungrouped single-partition
 *      sequences are written by step 2.
 * The passes are queued on `stream` by this call, the prefix pass first; the
 * partition pass reads none of the prefix pass's partials before its
 * arrival shows they are all stored, so it runs alongside it (its grid
 * finishes only after the prefix pass's).  prefix_plan is the device
 * copy of a prefix plan (num_groups, num_members as planned); an
 * inconsistent plan (a table that differs from the leader's on the prefix,
 * a prefix not below a member's context or off the 16-token grid, a
 * member's seq_prefix_len that differs from its group's) sets
 * PA_DEVERR_PREFIX_PLAN and leaves those rows undefined.  num_groups == 0
 * is plain split decode.  scale must be positive (PA_ERR_INVALID_ARG
 * otherwise).  Other arguments, limits and errors as pa_decode_attention
 * (16-bit pools; FP8 pools: pa_decode_attention_cascade_fp8).
 */
PA_API pa_status pa_decode_attention_cascade(void *out, const void *query, const void *key_cache,
                                             const void *value_cache,
                                             const int32_t *block_tables,
                                             int max_blocks_per_seq,
                                             const int32_t *context_lens, int max_context_len,
                                             int num_seqs, int num_heads, int num_kv_heads,
                                             int head_dim, int block_size, int num_blocks,
                                             float scale, const int32_t *prefix_plan,
                                             int num_groups, int num_members,
                                             int partition_size, void *workspace,
                                             size_t workspace_bytes, pa_dtype dtype,
                                             int32_t *error_word, void *stream);

/*
 * pa_decode_attention_cascade_append -- pa_decode_attention_cascade with the
 * decode step's append fused into its partition pass, as
 * pa_decode_attention_append does for pa_decode_attention: new_key /
 * new_value [num_seqs][num_kv_heads][head_dim] (dtype) are written at the
 * slot of position context_lens[s] - 1 (slot_mapping, optional, receives the
 * slots) and attended.  Every member's shared prefix must end before its new
 * token (prefix_plan's seq_start[s] < context_lens[s], as
 * pa_plan_prefix_groups plans it; otherwise PA_DEVERR_PREFIX_PLAN), so the
 * block written is the sequence's own and the prefix pass never reads it.
 * With num_groups == 0 this is pa_decode_attention_append.  Other arguments,
 * workspace (pa_cascade_workspace_bytes) and errors as
 * pa_decode_attention_cascade.
 */
PA_API pa_status pa_decode_attention_cascade_append(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    const int32_t *prefix_plan, int num_groups, int num_members, int partition_size,
    void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *error_word, void *stream);

/*
 * pa_decode_attention_cascade_fp8, pa_decode_attention_cascade_append_fp8 --
 * the prefix-aware decode (and its fused append) over FP8 pools written by
 * pa_reshape_and_cache_fp8, with the arithmetic of pa_decode_attention_fp8
 * in both passes (codes widened to fp16, query rounded to fp16 and flagged
 * PA_DEVERR_QUERY_RANGE beyond it, k_scale in the softmax scale, v_scale on
 * the output) and the append's codes as pa_decode_attention_append_fp8
 * writes them.  k_scale, v_scale positive and finite (PA_ERR_INVALID_ARG).
 * With num_groups == 0 these are pa_decode_attention_fp8 /
 * pa_decode_attention_append_fp8.  Other arguments, limits, workspace and errors as
 * pa_decode_attention_cascade(_append).
 */
PA_API pa_status pa_decode_attention_cascade_fp8(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, float k_scale, float v_scale,
    const int32_t *prefix_plan, int num_groups, int num_members, int partition_size,
    void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *error_word, void *stream);

PA_API pa_status pa_decode_attention_cascade_append_fp8(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    float k_scale, float v_scale, const int32_t *prefix_plan, int num_groups, int num_members,
    int partition_size, void *workspace, size_t workspace_bytes, pa_dtype dtype,
    int32_t *error_word, void *stream);

/*
 * pa_decode_attention_noalloc -- no counterpart on the pages: an addition
 * for callers that may not allocate device memory on their decode path (a
 * plugin whose host engine owns all device memory through its own pool, a
 * latency-critical loop that cannot take an allocation's implicit
 * synchronisation, a C interface that only passes inputs and outputs).
 * Same arguments, meaning and result as pa_decode_attention, minus the
 * workspace: the split-context partials go to a statically sized device
 * array of PA_NOALLOC_WORKSPACE_BYTES inside the library, created when the
 * library's device code is loaded on a GPU and kept by every such GPU until
 * the process exits.  The call itself allocates nothing.
 *   - Sizes whose workspace (pa_decode_workspace_bytes) exceeds
 *     PA_NOALLOC_WORKSPACE_BYTES are rejected with PA_ERR_WORKSPACE before
 *     anything is launched.
 *   - Arguments are checked first, with pa_decode_attention's statuses; a
 *     valid call whose partials need more than the array is then refused.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device, with that device current);
 *     make that first call before any stream capture.  The address is kept
 *     with the unique id of the CUDA context it belongs to: after a
 *     cudaDeviceReset (a new context), the next call looks it up again, so
 *     make that call, too, before any capture.
 *   - Every call on a device shares the one array and leaves its last
 *     contents there.  Its counter region (the workspace layout of
 *     pa_decode_workspace_bytes) starts at zero, since the array is
 *     zero-filled when the library's device code is loaded, and every call
 *     leaves it at zero; the partials need no initial contents (each call
 *     writes every partial it later reads).  Calls whose GPU work overlaps
 *     in time (for instance on two streams) race on the array.
 */
#define PA_NOALLOC_WORKSPACE_BYTES (32u * 1024u * 1024u)
PA_API pa_status pa_decode_attention_noalloc(void *out, const void *query,
                                             const void *key_cache, const void *value_cache,
                                             const int32_t *block_tables,
                                             int max_blocks_per_seq,
                                             const int32_t *context_lens, int max_context_len,
                                             int num_seqs, int num_heads, int num_kv_heads,
                                             int head_dim, int block_size, int num_blocks,
                                             float scale, int partition_size, pa_dtype dtype,
                                             int32_t *error_word, void *stream);

/*
 * Host block manager -- the bookkeeping either side of the cache write and
 * the block copy ([GAO] §1.3-§1.5, [FEI] "Block Table 实现" and
 * "共享前缀的 Block 复用", [LAKE] §3.2 and §4.2, [P1] §3.1).  Host memory
 * only; no call touches the GPU.  A manager owns the reference counts of a
 * pool of num_blocks physical blocks of block_size tokens and one block table
 * (logical block -> physical block) and token count per sequence:
 *   - a token appended at position p of a sequence goes to a new block when
 *     p % block_size == 0 (the lowest-numbered free block), otherwise into
 *     the sequence's last block;
 *   - fork gives the child the parent's table and token count, every block
 *     gaining a reference (parallel samples, shared prefixes);
 *   - appending into a last block that another table also names first copies
 *     it (copy-on-write): a new block is allocated, the (old, new) pair is
 *     returned for pa_copy_blocks -- which must run before the new tokens
 *     are written -- the sequence's table names the new block and the old
 *     one loses a reference;
 *   - freeing a sequence drops one reference from each of its blocks; a block
 *     no table names is free.
 * Calls on one manager must not overlap (no internal locking).  Every call
 * that fails leaves the manager unchanged.  Sequence ids are any values >= 0.
 */
typedef struct pa_block_manager pa_block_manager;

/* A manager with every block free.  PA_ERR_INVALID_ARG for sizes <= 0 or a
 * pool whose slots do not fit int32. */
PA_API pa_status pa_bm_create(int num_blocks, int block_size, int max_blocks_per_seq,
                              pa_block_manager **out);
PA_API void pa_bm_destroy(pa_block_manager *bm);
PA_API int pa_bm_num_free_blocks(const pa_block_manager *bm);
/* A new, empty sequence (PA_ERR_INVALID_ARG if the id exists or is < 0). */
PA_API pa_status pa_bm_add_sequence(pa_block_manager *bm, int seq_id);
/* child_id gets parent_id's table and token count (PA_ERR_INVALID_ARG if the
 * parent is unknown or the child exists). */
PA_API pa_status pa_bm_fork(pa_block_manager *bm, int parent_id, int child_id);
/* Append num_tokens tokens: slots[num_tokens] receive their cache slots
 * (block * block_size + offset, [GAO] §1.5); cow_pairs[2 * cow_capacity]
 * receive the (src, dst) copy-on-write pairs, *num_cow their count (at most
 * 1 per call).  PA_ERR_OUT_OF_BLOCKS when the free blocks do not cover the
 * new blocks and the copy, PA_ERR_TABLE_FULL past max_blocks_per_seq,
 * PA_ERR_WORKSPACE when cow_capacity is too small. */
PA_API pa_status pa_bm_append_tokens(pa_block_manager *bm, int seq_id, int num_tokens,
                                     int32_t *slots, int32_t *cow_pairs, int cow_capacity,
                                     int *num_cow);
/* One step's appends in one call: sequence seq_ids[i] gets counts[i] tokens
 * (ids distinct); the result is that of pa_bm_append_tokens called for each
 * in batch order.  slots[sum(counts)] receive the slots in batch order, and
 * cow_pairs[2 * cow_capacity] / *num_cow the copy-on-write pairs of the whole
 * batch (at most one per sequence; when every table naming a shared block
 * appends, the last one writes in place).  All or nothing, checks in this
 * order: a sequence unknown or repeated (PA_ERR_INVALID_ARG), past
 * max_blocks_per_seq (PA_ERR_TABLE_FULL), more pairs than cow_capacity
 * (PA_ERR_WORKSPACE), more blocks than are free (PA_ERR_OUT_OF_BLOCKS). */
PA_API pa_status pa_bm_append_batch(pa_block_manager *bm, const int32_t *seq_ids,
                                    const int32_t *counts, int n, int32_t *slots,
                                    int32_t *cow_pairs, int cow_capacity, int *num_cow);
/* Blocks (new ones and a copy-on-write copy) an append of num_tokens would
 * take, or -1 for an unknown sequence. */
PA_API int pa_bm_blocks_needed(const pa_block_manager *bm, int seq_id, int num_tokens);
PA_API pa_status pa_bm_free_sequence(pa_block_manager *bm, int seq_id);
/* Token and block counts of a sequence. */
PA_API pa_status pa_bm_sequence_info(const pa_block_manager *bm, int seq_id,
                                     int *num_tokens, int *num_blocks);
/* The sequence's table into row[capacity] (PA_ERR_WORKSPACE if shorter). */
PA_API pa_status pa_bm_block_table(const pa_block_manager *bm, int seq_id, int32_t *row,
                                   int capacity);
/* Number of tables naming a block (-1 out of range). */
PA_API int pa_bm_ref_count(const pa_block_manager *bm, int block);
/* Step inputs for a batch: block_tables[n][max_blocks] (rows padded with
 * pad_block) and context_lens[n] (token counts), host memory.
 * PA_ERR_WORKSPACE if a table is longer than max_blocks. */
PA_API pa_status pa_bm_build_batch(const pa_block_manager *bm, const int32_t *seq_ids, int n,
                                   int32_t *block_tables, int max_blocks,
                                   int32_t *context_lens, int32_t pad_block);

/* Human-readable name of a status code (static storage). */
PA_API const char *pa_status_string(pa_status status);

/* Name of the last CUDA error a call of this thread saw (static storage). */
PA_API const char *pa_last_cuda_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
PA_API int pa_version(void);

/*
 * Stage-wait limit -- no counterpart on the pages: the watchdog of the
 * attention kernels (pa_decode_attention*, pa_prefill_attention, the prefix
 * pass of pa_decode_attention_cascade*).  Each wait of such a kernel for
 * staged data (a K/V tile landing in shared memory, a tensor-core result)
 * gives up after limit_ns nanoseconds: the kernel then stops issuing work,
 * waits (up to the default limit) for the copies and tensor-core operations
 * it already started, releases its tensor memory, ORs PA_DEVERR_TIMEOUT into
 * the error word and returns; the outputs of that call are undefined, and
 * later calls on the stream are unaffected.  The setting is process-wide,
 * read when a call launches its kernels (calls already queued keep theirs).
 * limit_ns == 0 restores the default of one second.
 */
PA_API void pa_set_stage_wait_limit_ns(uint64_t limit_ns);
PA_API uint64_t pa_stage_wait_limit_ns(void);

/*
 * pa_debug_withhold_first_fill -- test hook of the time-out path above, no
 * counterpart on the pages.  While enabled (enable != 0; process-wide, read
 * at launch), every CTA of every attention kernel launched leaves its first
 * K/V fill unissued: nothing completes that stage, so the wait for it
 * runs out after the stage-wait limit and the kernel returns through its
 * time-out path (PA_DEVERR_TIMEOUT, undefined outputs of that call).  No
 * fault, no hang: every other copy the kernel issued is waited for.  Off by
 * default; meant only for tests of the watchdog.
 */
PA_API void pa_debug_withhold_first_fill(int enable);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTENTION_H */
