// pa_decode_common.cuh -- pieces shared by the 16-bit and the FP8 paged
// decode passes: launch parameters, the context-length rule, the
// split-context reduce kernel and its launch, the tensor-map encoder entry
// point, per-device launch settings and the workspace layout.
#pragma once

#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pa_common.cuh"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kTileTokens = 16;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second per stage wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kSlack = 8.f;  // log2 units: softmax weights stay <= 256 before rescaling

struct DecodeParams {
    void *out;
    const void *query;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *part_m;
    float *part_l;
    float *part_o;
    int32_t *error_word;
    int num_seqs, num_heads, num_kv_heads, group;
    int max_blocks_per_seq, num_blocks, block_size, max_context_len;
    int block_shift;  // log2(block_size)
    int part_tokens;  // tokens per work unit (a multiple of 16)
    int max_parts;    // partitions per sequence the workspace holds
    float scale_log2; // scale * log2(e) (times the K scale for FP8 pools)
    float out_scale;  // applied to the attention output (the V scale for FP8 pools)
};

// Clamped context length (same rule in both kernels).
__device__ __forceinline__ int clamp_context(const DecodeParams &p, int s, bool flag)
{
    const int limit = min(p.max_context_len, p.max_blocks_per_seq * p.block_size);
    int c = p.context_lens[s];
    if (c < 0 || c > limit) {
        if (flag)
            flag_error(p.error_word, PA_DEVERR_CONTEXT_RANGE);
        c = c < 0 ? 0 : limit;
    }
    return c;
}

// ---- split-context reduce ----------------------------------------------------------
//
// One CTA per (sequence, KV head).  For the G query heads of the group it
// merges the nparts partials (m_q, l_q, o_q) of a sequence that spans more
// than one partition: M = max_q m_q, w_q = l_q exp(m_q - M),
// out = sum_q w_q o_q / sum_q w_q.  Sequences with one partition were written
// by the partition pass itself.  (1) warp w finds M and sum_q w_q for heads
// jh = w, w + 4, ...; (2) thread (item, qg) sums w_q o_q over q = qg, qg + QG,
// ...; (3) the QG group sums are added in shared memory.
constexpr int kReduceThreads = 256;
constexpr int kReduceChunk = 128;  // partitions whose weights are staged at once

template <typename T, int D>
__global__ void __launch_bounds__(kReduceThreads)
    paged_reduce_kernel(const __grid_constant__ DecodeParams p)
{
    using Op = MmaOp<T>;
    __shared__ float head_m[16], head_inv_l[16];
    __shared__ float wts[16 * kReduceChunk];
    __shared__ __align__(16) float red[kReduceThreads * 8];
    pdl_wait_primary();  // the partition pass's partials are visible past here

    const int Hkv = p.num_kv_heads;
    const int G = p.group;
    const int s = blockIdx.x / Hkv;
    const int kh = blockIdx.x - s * Hkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ctx = clamp_context(p, s, false);
    const int nparts = (ctx + p.part_tokens - 1) / p.part_tokens;
    if (nparts <= 1)
        return;

    // (1) per head: M = max_q m_q and L = sum_q l_q exp(m_q - M) (warp per head)
    const size_t hbase = ((size_t)s * p.num_heads + (size_t)kh * G) * p.max_parts;
    for (int jh = warp; jh < G; jh += kReduceThreads / 32) {
        const float *pm = p.part_m + hbase + (size_t)jh * p.max_parts;
        const float *pl = p.part_l + hbase + (size_t)jh * p.max_parts;
        float mx = -INFINITY;
        for (int q = lane; q < nparts; q += 32)
            mx = fmaxf(mx, pm[q]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
        float ls = 0.f;
        for (int q = lane; q < nparts; q += 32)
            ls += pl[q] * exp2f((pm[q] - mx) * kLog2e);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            ls += __shfl_xor_sync(kFull, ls, off);
        if (lane == 0) {
            head_m[jh] = mx;
            head_inv_l[jh] = 1.f / ls;
        }
    }
    __syncthreads();

    // (2) thread (item, qg) sums w_q o_q over q = qg, qg + QG, ... with the
    // weights w_q = l_q exp(m_q - M) / L of a chunk of partitions staged in
    // shared memory; (3) the QG group sums are added in shared memory.
    // G * D / 8 <= 16 * 128 / 8 = kReduceThreads: one (item, qg) per thread.
    static_assert(16 * D / 8 <= kReduceThreads, "one work item per thread");
    const int items = G * (D / 8);
    const int qgroups = max(1, kReduceThreads / items);
    const bool active = tid < items * qgroups;
    const int item = tid % items;
    const int qg = tid / items;
    const int jh = item / (D / 8);
    const int d0 = (item - jh * (D / 8)) * 8;
    const float *po = p.part_o + (hbase + (size_t)jh * p.max_parts) * D + d0;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < nparts; c0 += kReduceChunk) {
        const int cn = min(kReduceChunk, nparts - c0);
        for (int i = tid; i < G * cn; i += kReduceThreads) {
            const int h = i / cn, q = c0 + (i - h * cn);
            const size_t idx = hbase + (size_t)h * p.max_parts + q;
            wts[h * kReduceChunk + (q - c0)] =
                p.part_l[idx] * exp2f((p.part_m[idx] - head_m[h]) * kLog2e) * head_inv_l[h];
        }
        __syncthreads();
        if (active) {
#pragma unroll 8
            for (int q = c0 + qg; q < c0 + cn; q += qgroups) {
                const float wgt = wts[jh * kReduceChunk + (q - c0)];
                const float4 x0 = reinterpret_cast<const float4 *>(po + (size_t)q * D)[0];
                const float4 x1 = reinterpret_cast<const float4 *>(po + (size_t)q * D)[1];
                acc[0] += wgt * x0.x; acc[1] += wgt * x0.y; acc[2] += wgt * x0.z; acc[3] += wgt * x0.w;
                acc[4] += wgt * x1.x; acc[5] += wgt * x1.y; acc[6] += wgt * x1.z; acc[7] += wgt * x1.w;
            }
        }
        __syncthreads();
    }
    if (active) {
        if (qgroups == 1) {
            T vals[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                vals[e] = Op::from_float(acc[e]);
            *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) +
                                       ((size_t)s * p.num_heads + (size_t)kh * G + jh) * D +
                                       d0) = *reinterpret_cast<const uint4 *>(vals);
        } else {
            float4 *dst = reinterpret_cast<float4 *>(red + (size_t)tid * 8);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
    if (qgroups == 1)
        return;
    __syncthreads();
    for (int it = tid; it < items; it += kReduceThreads) {
        const int jh = it / (D / 8);
        const int d0 = (it - jh * (D / 8)) * 8;
        float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int g2 = 0; g2 < qgroups; ++g2) {
            const float4 *src = reinterpret_cast<const float4 *>(red + (size_t)(g2 * items + it) * 8);
            const float4 x0 = src[0], x1 = src[1];
            sum[0] += x0.x; sum[1] += x0.y; sum[2] += x0.z; sum[3] += x0.w;
            sum[4] += x1.x; sum[5] += x1.y; sum[6] += x1.z; sum[7] += x1.w;
        }
        T vals[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            vals[e] = Op::from_float(sum[e]);
        *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) +
                                   ((size_t)s * p.num_heads + (size_t)kh * G + jh) * D + d0) =
            *reinterpret_cast<const uint4 *>(vals);
    }
}

// ---- host side -------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *,
                                   const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Per-device facts and per-kernel launch settings, looked up once: the SM
// count and shared-memory limit of each device, and for each kernel the
// largest dynamic shared memory it has been enabled for and the residency
// found for the last shared-memory size.
constexpr int kMaxDevices = 64;
struct DeviceInfo {
    int sms = 0, optin = 0;
};
static pa_status device_info(int dev, DeviceInfo *out)
{
    static DeviceInfo cache[kMaxDevices];
    static std::mutex mu;
    if (dev < 0 || dev >= kMaxDevices)
        return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms == 0) {
        cudaError_t e = cudaDeviceGetAttribute(&cache[dev].optin,
                                               cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&cache[dev].sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) {
            cache[dev].sms = 0;
            return record_cuda(e);
        }
    }
    *out = cache[dev];
    return PA_OK;
}

struct KernelSetting {
    size_t smem_enabled = 0;  // dynamic shared memory the kernel may use
    size_t smem_queried = 0;  // shared-memory size of the cached residency
    int per_sm = 0;           // resident CTAs per SM at smem_queried
};

// The reduce is queued behind the partition pass with programmatic
// dependent launch: its CTAs may start while the pass drains and wait in
// griddepcontrol.wait until the pass's writes are visible.
template <typename T, int D>
static pa_status launch_reduce(const DecodeParams &prm, cudaStream_t stream)
{
    return launch_pdl(paged_reduce_kernel<T, D>, dim3((unsigned)(prm.num_seqs * prm.num_kv_heads)),
                      dim3(kReduceThreads), 0, stream, prm);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WorkspaceLayout {
    size_t m_off, l_off, o_off, total;
};

static WorkspaceLayout workspace_layout(int S, int H, int D, int parts)
{
    WorkspaceLayout w{};
    if (parts <= 1)
        return w;
    const size_t ml = align256((size_t)S * H * parts * 4);
    w.m_off = 0;
    w.l_off = ml;
    w.o_off = 2 * ml;
    w.total = w.o_off + align256((size_t)S * H * parts * D * 4);
    return w;
}

static int num_parts(int max_context_len, int partition_size)
{
    if (partition_size <= 0 || max_context_len <= 0)
        return 1;
    return (int)(((long long)max_context_len + partition_size - 1) / partition_size);
}

// Host-side checks shared by the decode entry points, then the launch
// parameters and the workspace carve-up.  Returns PA_OK with nothing filled
// in when num_seqs == 0.
static pa_status prepare_decode(DecodeParams *prm, void *out, const void *query,
                                const void *key_cache, const void *value_cache,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, int max_context_len,
                                int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, float scale,
                                int partition_size, void *workspace, size_t workspace_bytes,
                                int32_t *error_word)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        max_context_len < 0 || partition_size < 0 || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) ||
        !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || block_size < kTileTokens ||
        block_size > 256 || (block_size & (block_size - 1)) != 0 || group > 16 ||
        (long long)num_blocks * block_size >= (1ll << 31) ||
        (long long)max_blocks_per_seq * block_size >= (1ll << 31))
        return PA_ERR_UNSUPPORTED;
    if (partition_size != 0 && partition_size % kTileTokens != 0)
        return PA_ERR_UNSUPPORTED;

    const int parts = num_parts(max_context_len, partition_size);
    const WorkspaceLayout wl = workspace_layout(num_seqs, num_heads, head_dim, parts);
    if (wl.total > 0 && (workspace == nullptr || workspace_bytes < wl.total ||
                         (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return PA_ERR_WORKSPACE;

    prm->out = out;
    prm->query = query;
    prm->block_tables = block_tables;
    prm->context_lens = context_lens;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    prm->part_m = wl.total ? reinterpret_cast<float *>(ws + wl.m_off) : nullptr;
    prm->part_l = wl.total ? reinterpret_cast<float *>(ws + wl.l_off) : nullptr;
    prm->part_o = wl.total ? reinterpret_cast<float *>(ws + wl.o_off) : nullptr;
    prm->error_word = error_word;
    prm->num_seqs = num_seqs;
    prm->num_heads = num_heads;
    prm->num_kv_heads = num_kv_heads;
    prm->group = group;
    prm->max_blocks_per_seq = max_blocks_per_seq;
    prm->num_blocks = num_blocks;
    prm->block_size = block_size;
    prm->max_context_len = max_context_len;
    prm->block_shift = __builtin_ctz((unsigned)block_size);
    // Single pass: one unit covers the longest possible context.
    const long long ctx_cap = (long long)max_blocks_per_seq * block_size;
    const long long whole = ((std::max<long long>(1, std::min<long long>(
                                  max_context_len, ctx_cap)) + kTileTokens - 1) /
                             kTileTokens) * kTileTokens;
    prm->part_tokens = parts > 1 ? partition_size : (int)whole;
    prm->max_parts = parts;
    prm->scale_log2 = scale * kLog2e;
    prm->out_scale = 1.f;
    return PA_OK;
}

} // namespace pa
