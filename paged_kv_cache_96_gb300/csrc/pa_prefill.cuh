// pa_prefill.cuh -- launch parameters of the multi-query paged attention
// kernel (chunked prefill, and the shared-prefix pass of prefix-aware
// decode) and the entry the prefix-aware decode uses to queue that pass.
#pragma once

#include "pa_decode_common.cuh"

namespace pa {

struct MqParams {
    void *out;                  // prefill: [T][H][D] in the query dtype
    const void *query;          // prefill: [T][H][D]; prefix pass: decode queries [S][H][D]
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start;     // prefill: [S + 1] chunk rows of each sequence
    const int32_t *group_start;     // prefix pass: [groups + 1] into group_members
    const int32_t *group_members;   // prefix pass: member sequences, group by group
    const int32_t *group_prefix;    // prefix pass: [groups] shared tokens
    const int32_t *seq_start;       // prefix pass: [S] each sequence's shared tokens (checked)
    float *part_m;
    float *part_l;
    float *part_o;
    // prefix pass: the partition pass's arrival counters (null: the reduce
    // kernel merges); out is then the decode output [S][H][D]
    int32_t *counters;
    int32_t *error_word;
    uint64_t wait_ns;  // limit of one stage wait (PA_DEVERR_TIMEOUT past it)
    int withhold_fill; // test hook: each CTA's key warp never issues its first fill
    int prefix_mode;   // 0: chunked prefill, 1: shared-prefix pass
    int num_segments;  // sequences (prefill) or groups (prefix pass)
    int num_seqs, num_heads, num_kv_heads, group;
    int max_blocks_per_seq, num_blocks, block_size, block_shift, max_context_len;
    int max_parts;     // partials per (sequence, head) in the workspace
    int part_tokens;   // prefix pass: tokens per prefix partition (partial j)
    float scale_log2;  // scale * log2(e) (times the K scale for FP8 pools)
    float out_scale;   // applied to the output / partials (the V scale for FP8 pools)
    int num_tokens;    // prefill: rows of query and out (T)
    int q_tma;         // 1: each unit's query tile arrives by TMA (the query map)
};

// Queue the shared-prefix pass on `stream` as a programmatic dependent of the
// kernel before it (dtype PA_FP8_E4M3: FP8 pools, query and output of
// query_dtype; else 16-bit pools of dtype).
pa_status launch_prefix_pass(const MqParams &prm, pa_dtype dtype, pa_dtype query_dtype,
                             const void *key_cache, const void *value_cache, int head_dim,
                             cudaStream_t stream, long long max_units);

}  // namespace pa
