// pa_cache_ops.cu -- the byte-moving and index kernels of the paged KV
// cache: slot mapping and reshape_and_cache ("PagedAttention & Continuous
// Batching" §1.5; "vLLM 架构详解", "Block Table 实现") and the copy-on-write
// block copy ("vLLM源码解析(二)" §3.2).  All three are bit-exact: they move
// 16-byte words or compute integers.
#include <atomic>
#include <cstdio>
#include <cstring>

#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_common.cuh"
#include "pa_ptx.cuh"

namespace pa {

namespace {
thread_local char g_last_error[256] = "no error";
// Time limit of one wait on staged data in the attention kernels, read when
// a call launches them.
std::atomic<uint64_t> g_stage_wait_ns{kDefaultStageWaitNs};
std::atomic<int> g_withhold_fill{0};
}

uint64_t stage_wait_limit_ns() { return g_stage_wait_ns.load(std::memory_order_relaxed); }
int withhold_first_fill() { return g_withhold_fill.load(std::memory_order_relaxed); }

pa_status record_cuda(cudaError_t err)
{
    if (err == cudaSuccess)
        return PA_OK;
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(err),
                  cudaGetErrorString(err));
    return PA_ERR_CUDA;
}

// ---- slot mapping ------------------------------------------------------------

// The slot of token t: table[s][p / bs] * bs + p % bs, or -1 (flagged) for a
// token outside the batch or the table, or a table entry outside the pool.
__device__ __forceinline__ int32_t token_slot(const int32_t *__restrict__ block_tables,
                                              int max_blocks_per_seq,
                                              const int32_t *__restrict__ token_seq,
                                              const int32_t *__restrict__ token_pos, int t,
                                              int num_seqs, int block_size, int num_blocks,
                                              int32_t *error_word)
{
    const int s = token_seq[t];
    const int p = token_pos[t];
    if (s < 0 || s >= num_seqs || p < 0 || p / block_size >= max_blocks_per_seq) {
        flag_error(error_word, PA_DEVERR_TOKEN_RANGE);
        return -1;
    }
    const int32_t block =
        block_tables[static_cast<int64_t>(s) * max_blocks_per_seq + p / block_size];
    if (block < 0 || block >= num_blocks) {
        flag_error(error_word, PA_DEVERR_BLOCK_RANGE);
        return -1;
    }
    return block * block_size + p % block_size;
}

// One thread per token.
__global__ void slot_mapping_kernel(int32_t *__restrict__ slot_mapping,
                                    const int32_t *__restrict__ block_tables,
                                    int max_blocks_per_seq,
                                    const int32_t *__restrict__ token_seq,
                                    const int32_t *__restrict__ token_pos, int num_tokens,
                                    int num_seqs, int block_size, int num_blocks,
                                    int32_t *error_word)
{
    pdl_wait_primary();
    pdl_launch_dependents();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= num_tokens)
        return;
    slot_mapping[t] = token_slot(block_tables, max_blocks_per_seq, token_seq, token_pos, t,
                                 num_seqs, block_size, num_blocks, error_word);
}

// Where a cache-write CTA finds its token's slot: in slot_mapping (written
// by slot_mapping_kernel), or -- fused -- computed here from the token's
// sequence and position (thread 0), stored to slot_mapping and shared.
struct SlotSource {
    int32_t *slot_mapping;
    const int32_t *block_tables;  // null: read slot_mapping
    const int32_t *token_seq;
    const int32_t *token_pos;
    int max_blocks_per_seq, num_seqs, block_size, num_blocks;
};

__device__ __forceinline__ int64_t cta_token_slot(const SlotSource &src, int t,
                                                  int32_t *error_word)
{
    if (src.block_tables == nullptr)
        return src.slot_mapping[t];
    __shared__ int32_t slot_s;
    if (threadIdx.x == 0) {
        const int32_t slot = token_slot(src.block_tables, src.max_blocks_per_seq,
                                        src.token_seq, src.token_pos, t, src.num_seqs,
                                        src.block_size, src.num_blocks, error_word);
        src.slot_mapping[t] = slot;
        slot_s = slot;
    }
    __syncthreads();
    return slot_s;
}

// ---- reshape_and_cache --------------------------------------------------------

// One CTA per token; threads stride over the token's K and V rows
// (num_kv_heads * head_dim 16-bit elements each) in 16-byte words.
__global__ void reshape_and_cache_kernel(const uint4 *__restrict__ key,
                                         const uint4 *__restrict__ value,
                                         uint4 *__restrict__ key_cache,
                                         uint4 *__restrict__ value_cache,
                                         const SlotSource slots, int64_t num_slots,
                                         int words_per_token, int32_t *error_word)
{
    pdl_wait_primary();
    pdl_launch_dependents();
    const int t = blockIdx.x;
    const int64_t slot = cta_token_slot(slots, t, error_word);
    if (slot < 0)
        return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0)
            flag_error(error_word, PA_DEVERR_SLOT_RANGE);
        return;
    }
    const uint4 *ks = key + static_cast<int64_t>(t) * words_per_token;
    const uint4 *vs = value + static_cast<int64_t>(t) * words_per_token;
    uint4 *kd = key_cache + slot * words_per_token;
    uint4 *vd = value_cache + slot * words_per_token;
    for (int i = threadIdx.x; i < words_per_token; i += blockDim.x) {
        const uint4 k = __ldg(ks + i);
        const uint4 v = __ldg(vs + i);
        kd[i] = k;
        vd[i] = v;
    }
}

// ---- reshape_and_cache into FP8 (e4m3) pools ----------------------------------

__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }

// One CTA per token; each thread converts 8 elements at a time: 16 bytes of
// 16-bit input -> 8 bytes of e4m3 codes, code = e4m3(float(x) * inv_scale).
template <typename T>
__global__ void reshape_and_cache_fp8_kernel(const uint4 *__restrict__ key,
                                             const uint4 *__restrict__ value,
                                             uint2 *__restrict__ key_cache,
                                             uint2 *__restrict__ value_cache,
                                             const SlotSource slots, int64_t num_slots,
                                             int words_per_token, float k_inv_scale,
                                             float v_inv_scale, int32_t *error_word)
{
    pdl_wait_primary();
    pdl_launch_dependents();
    const int t = blockIdx.x;
    const int64_t slot = cta_token_slot(slots, t, error_word);
    if (slot < 0)
        return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0)
            flag_error(error_word, PA_DEVERR_SLOT_RANGE);
        return;
    }
    auto quantise = [](uint4 w, float inv) {
        const T *e = reinterpret_cast<const T *>(&w);
        uint2 out;
        out.x = (uint32_t)f32x2_to_e4m3x2(to_float(e[0]) * inv, to_float(e[1]) * inv) |
                ((uint32_t)f32x2_to_e4m3x2(to_float(e[2]) * inv, to_float(e[3]) * inv) << 16);
        out.y = (uint32_t)f32x2_to_e4m3x2(to_float(e[4]) * inv, to_float(e[5]) * inv) |
                ((uint32_t)f32x2_to_e4m3x2(to_float(e[6]) * inv, to_float(e[7]) * inv) << 16);
        return out;
    };
    const uint4 *ks = key + static_cast<int64_t>(t) * words_per_token;
    const uint4 *vs = value + static_cast<int64_t>(t) * words_per_token;
    uint2 *kd = key_cache + slot * words_per_token;
    uint2 *vd = value_cache + slot * words_per_token;
    for (int i = threadIdx.x; i < words_per_token; i += blockDim.x) {
        kd[i] = quantise(__ldg(ks + i), k_inv_scale);
        vd[i] = quantise(__ldg(vs + i), v_inv_scale);
    }
}

// ---- copy_blocks ----------------------------------------------------------------

// grid.x = pair, grid.y = 0 (K) / 1 (V), grid.z = slab of 16-byte words.
constexpr int kCopyThreads = 256;
constexpr int kCopyWordsPerThread = 4;

__global__ void copy_blocks_kernel(uint4 *__restrict__ key_cache,
                                   uint4 *__restrict__ value_cache,
                                   const int32_t *__restrict__ block_mapping,
                                   int num_blocks, int64_t words_per_block,
                                   int32_t *error_word)
{
    pdl_wait_primary();
    pdl_launch_dependents();
    const int pair = blockIdx.x;
    const int src = block_mapping[2 * pair];
    const int dst = block_mapping[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            flag_error(error_word, PA_DEVERR_PAIR_RANGE);
        return;
    }
    uint4 *pool = blockIdx.y == 0 ? key_cache : value_cache;
    const uint4 *from = pool + static_cast<int64_t>(src) * words_per_block;
    uint4 *to = pool + static_cast<int64_t>(dst) * words_per_block;
    const int64_t base =
        static_cast<int64_t>(blockIdx.z) * kCopyThreads * kCopyWordsPerThread + threadIdx.x;
    uint4 w[kCopyWordsPerThread];
#pragma unroll
    for (int k = 0; k < kCopyWordsPerThread; ++k) {
        const int64_t i = base + k * kCopyThreads;
        if (i < words_per_block)
            w[k] = from[i];
    }
#pragma unroll
    for (int k = 0; k < kCopyWordsPerThread; ++k) {
        const int64_t i = base + k * kCopyThreads;
        if (i < words_per_block)
            to[i] = w[k];
    }
}

} // namespace pa

using namespace pa;

extern "C" pa_status pa_slot_mapping(int32_t *slot_mapping, const int32_t *block_tables,
                                     int max_blocks_per_seq, const int32_t *token_seq,
                                     const int32_t *token_pos, int num_tokens,
                                     int num_seqs, int block_size, int num_blocks,
                                     int32_t *error_word, void *stream)
{
    if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return PA_OK;
    if (!slot_mapping || !block_tables || !token_seq || !token_pos)
        return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    const int threads = 256;
    const int blocks = (num_tokens + threads - 1) / threads;
    return launch_pdl(slot_mapping_kernel, dim3(blocks), dim3(threads), 0, as_stream(stream),
                      slot_mapping, block_tables, max_blocks_per_seq, token_seq, token_pos,
                      num_tokens, num_seqs, block_size, num_blocks, error_word);
}

// The cache writes of both entry forms (slots given, or computed in the
// same launch).
static pa_status cache_write(const void *key, const void *value, void *key_cache,
                             void *value_cache, const SlotSource &src, int num_tokens,
                             int num_blocks, int block_size, int num_kv_heads, int head_dim,
                             pa_dtype dtype, int32_t *error_word, void *stream)
{
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || (dtype != PA_F16 && dtype != PA_BF16))
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !src.slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) ||
        !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * 2;
    if (row_bytes % 16 != 0)
        return PA_ERR_UNSUPPORTED;
    const int words = static_cast<int>(row_bytes / 16);
    const int threads = words >= 256 ? 256 : ((words + 31) / 32) * 32;
    return launch_pdl(reshape_and_cache_kernel, dim3(num_tokens), dim3(threads), 0,
                      as_stream(stream), static_cast<const uint4 *>(key),
                      static_cast<const uint4 *>(value), static_cast<uint4 *>(key_cache),
                      static_cast<uint4 *>(value_cache), src,
                      static_cast<int64_t>(num_blocks) * block_size, words, error_word);
}

static pa_status cache_write_fp8(const void *key, const void *value, void *key_cache,
                                 void *value_cache, const SlotSource &src, int num_tokens,
                                 int num_blocks, int block_size, int num_kv_heads,
                                 int head_dim, pa_dtype src_dtype, float k_scale,
                                 float v_scale, int32_t *error_word, void *stream)
{
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || (src_dtype != PA_F16 && src_dtype != PA_BF16) ||
        !std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale <= 0.f ||
        v_scale <= 0.f)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !src.slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) ||
        !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const int64_t row_elems = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (row_elems % 8 != 0)
        return PA_ERR_UNSUPPORTED;
    const int words = static_cast<int>(row_elems / 8);
    const int threads = words >= 256 ? 256 : ((words + 31) / 32) * 32;
    const float k_inv = 1.0f / k_scale;  // fp32, as the codes' contract states
    const float v_inv = 1.0f / v_scale;
    const int64_t slots = static_cast<int64_t>(num_blocks) * block_size;
    if (src_dtype == PA_BF16)
        return launch_pdl(reshape_and_cache_fp8_kernel<__nv_bfloat16>, dim3(num_tokens),
                          dim3(threads), 0, as_stream(stream), static_cast<const uint4 *>(key),
                          static_cast<const uint4 *>(value), static_cast<uint2 *>(key_cache),
                          static_cast<uint2 *>(value_cache), src, slots, words, k_inv, v_inv,
                          error_word);
    return launch_pdl(reshape_and_cache_fp8_kernel<__half>, dim3(num_tokens), dim3(threads), 0,
                      as_stream(stream), static_cast<const uint4 *>(key),
                      static_cast<const uint4 *>(value), static_cast<uint2 *>(key_cache),
                      static_cast<uint2 *>(value_cache), src, slots, words, k_inv, v_inv,
                      error_word);
}

// Slots computed in the cache-write launch: the tables and token arrays are
// checked as pa_slot_mapping checks them.
static pa_status fused_source(SlotSource *src, int32_t *slot_mapping,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *token_seq, const int32_t *token_pos,
                              int num_tokens, int num_seqs, int block_size, int num_blocks)
{
    if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!slot_mapping || !block_tables || !token_seq || !token_pos))
        return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    *src = SlotSource{slot_mapping, block_tables, token_seq, token_pos,
                      max_blocks_per_seq, num_seqs, block_size, num_blocks};
    return PA_OK;
}

extern "C" pa_status pa_reshape_and_cache(const void *key, const void *value,
                                          void *key_cache, void *value_cache,
                                          const int32_t *slot_mapping, int num_tokens,
                                          int num_blocks, int block_size,
                                          int num_kv_heads, int head_dim, pa_dtype dtype,
                                          int32_t *error_word, void *stream)
{
    const SlotSource src{const_cast<int32_t *>(slot_mapping), nullptr, nullptr, nullptr,
                         0, 0, 0, 0};
    return cache_write(key, value, key_cache, value_cache, src, num_tokens, num_blocks,
                       block_size, num_kv_heads, head_dim, dtype, error_word, stream);
}

extern "C" pa_status pa_reshape_and_cache_fp8(const void *key, const void *value,
                                              void *key_cache, void *value_cache,
                                              const int32_t *slot_mapping, int num_tokens,
                                              int num_blocks, int block_size,
                                              int num_kv_heads, int head_dim,
                                              pa_dtype src_dtype, float k_scale,
                                              float v_scale, int32_t *error_word,
                                              void *stream)
{
    const SlotSource src{const_cast<int32_t *>(slot_mapping), nullptr, nullptr, nullptr,
                         0, 0, 0, 0};
    return cache_write_fp8(key, value, key_cache, value_cache, src, num_tokens, num_blocks,
                           block_size, num_kv_heads, head_dim, src_dtype, k_scale, v_scale,
                           error_word, stream);
}

extern "C" pa_status pa_slot_mapping_and_cache(
    int32_t *slot_mapping, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *token_seq, const int32_t *token_pos, int num_tokens, int num_seqs,
    const void *key, const void *value, void *key_cache, void *value_cache, int num_blocks,
    int block_size, int num_kv_heads, int head_dim, pa_dtype dtype, int32_t *error_word,
    void *stream)
{
    SlotSource src;
    const pa_status st = fused_source(&src, slot_mapping, block_tables, max_blocks_per_seq,
                                      token_seq, token_pos, num_tokens, num_seqs, block_size,
                                      num_blocks);
    if (st != PA_OK)
        return st;
    return cache_write(key, value, key_cache, value_cache, src, num_tokens, num_blocks,
                       block_size, num_kv_heads, head_dim, dtype, error_word, stream);
}

extern "C" pa_status pa_slot_mapping_and_cache_fp8(
    int32_t *slot_mapping, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *token_seq, const int32_t *token_pos, int num_tokens, int num_seqs,
    const void *key, const void *value, void *key_cache, void *value_cache, int num_blocks,
    int block_size, int num_kv_heads, int head_dim, pa_dtype src_dtype, float k_scale,
    float v_scale, int32_t *error_word, void *stream)
{
    SlotSource src;
    const pa_status st = fused_source(&src, slot_mapping, block_tables, max_blocks_per_seq,
                                      token_seq, token_pos, num_tokens, num_seqs, block_size,
                                      num_blocks);
    if (st != PA_OK)
        return st;
    return cache_write_fp8(key, value, key_cache, value_cache, src, num_tokens, num_blocks,
                           block_size, num_kv_heads, head_dim, src_dtype, k_scale, v_scale,
                           error_word, stream);
}

extern "C" pa_status pa_copy_blocks(void *key_cache, void *value_cache,
                                    const int32_t *block_mapping, int num_pairs,
                                    int num_blocks, int block_size, int num_kv_heads,
                                    int head_dim, pa_dtype dtype, int32_t *error_word,
                                    void *stream)
{
    if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || (dtype != PA_F16 && dtype != PA_BF16 && dtype != PA_FP8_E4M3))
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0)
        return PA_OK;
    if (!key_cache || !value_cache || !block_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const int64_t elem_bytes = dtype == PA_FP8_E4M3 ? 1 : 2;
    const int64_t block_bytes =
        static_cast<int64_t>(block_size) * num_kv_heads * head_dim * elem_bytes;
    if (block_bytes % 16 != 0)
        return PA_ERR_UNSUPPORTED;
    const int64_t words = block_bytes / 16;
    const int64_t per_cta = static_cast<int64_t>(kCopyThreads) * kCopyWordsPerThread;
    const int64_t slabs = (words + per_cta - 1) / per_cta;
    if (slabs > 65535 || num_pairs > INT32_MAX / 2)
        return PA_ERR_UNSUPPORTED;
    dim3 grid(num_pairs, 2, static_cast<unsigned>(slabs));
    return launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), 0, as_stream(stream),
                      static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache),
                      block_mapping, num_blocks, words, error_word);
}

extern "C" const char *pa_status_string(pa_status status)
{
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
    case PA_ERR_TABLE_FULL: return "PA_ERR_TABLE_FULL";
    }
    return "PA_UNKNOWN_STATUS";
}

extern "C" const char *pa_last_cuda_error(void) { return g_last_error; }

extern "C" int pa_version(void) { return 100; }

extern "C" void pa_set_stage_wait_limit_ns(uint64_t limit_ns)
{
    g_stage_wait_ns.store(limit_ns == 0 ? kDefaultStageWaitNs : limit_ns,
                          std::memory_order_relaxed);
}

extern "C" uint64_t pa_stage_wait_limit_ns(void) { return stage_wait_limit_ns(); }

extern "C" void pa_debug_withhold_first_fill(int enable)
{
    g_withhold_fill.store(enable ? 1 : 0, std::memory_order_relaxed);
}
