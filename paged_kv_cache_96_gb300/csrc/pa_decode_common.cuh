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
// Partials of a sequence the partition pass merges itself, at most.
constexpr int kMergeMax = 8;
// Arrival counters a workspace holds at least (1 MB; one per sequence and
// KV head).
constexpr size_t kCounterWords = size_t(1) << 18;
constexpr uint64_t kDrainWaitNs = kDefaultStageWaitNs;  // waits for copies in flight at exit
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kSlack = 8.f;  // log2 units: softmax weights stay <= 256 before rescaling

struct DecodeParams {
    void *out;
    const void *query;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *seq_start;  // prefix-aware decode: first private token per sequence (or null)
    float *part_m;
    float *part_l;
    float *part_o;
    // Arrival counters of the merge fused into the pass, one per (sequence,
    // KV head) (null: the reduce kernel merges every split sequence).
    int32_t *counters;
    int32_t *error_word;
    uint64_t wait_ns;  // limit of one stage wait (PA_DEVERR_TIMEOUT past it)
    int withhold_fill; // test hook: warp 0 of each CTA never issues its first fill
    int num_seqs, num_heads, num_kv_heads, group;
    int max_blocks_per_seq, num_blocks, block_size, max_context_len;
    int block_shift;  // log2(block_size)
    int part_tokens;  // tokens per work unit (a multiple of 16)
    int reduce_heads; // reduce kernel: query heads per CTA (1 or the group)
    int max_parts;    // partitions per sequence the workspace holds
    float scale_log2; // scale * log2(e) (times the K scale for FP8 pools)
    float out_scale;  // applied to the attention output (the V scale for FP8 pools)
    // Deal: the first early_rounds rounds go to CTAs [0, early_ctas) alone (the
    // others start late, behind the shared-prefix pass's CTAs), then every
    // CTA takes one unit per round.
    int early_ctas, early_rounds;
    int prefix_sms;   // SMs the shared-prefix pass is expected to hold (0: none)
    int concurrent;   // 1: the kernel before it on the stream (the shared-prefix
                      // pass) writes nothing this pass reads -- run alongside it
                      // and wait for it only before finishing
    // Decode step with the append fused in (null new_key: attention only).
    // Sequence s's new token sits at position context_lens[s] - 1; its rows
    // new_key/new_value [num_seqs][num_kv_heads][head_dim] (16-bit, type T)
    // are written to the pools at that position's slot (as e4m3 codes times
    // k_inv_scale / v_inv_scale for FP8 pools) and attended from the copy in
    // shared memory; slot_out (optional) receives each sequence's slot.
    void *key_cache;
    void *value_cache;
    const void *new_key;
    const void *new_value;
    int32_t *slot_out;
    float k_inv_scale, v_inv_scale;
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

// First token a sequence's own units attend: 0, or (prefix-aware decode) the
// length of the shared prefix that the prefix pass covers.  A start outside
// [0, ctx] or off the 16-token tile grid is ignored here (the prefix pass
// flags the plan); both the partition pass and the reduce use this rule, so
// they agree on where a sequence's partials go.
__device__ __forceinline__ int seq_start_of(const DecodeParams &p, int s, int ctx)
{
    if (p.seq_start == nullptr)
        return 0;
    const int st = p.seq_start[s];
    return (st < 0 || st > ctx || (st & (kTileTokens - 1)) != 0) ? 0 : st;
}

// Partials a sequence leaves in the workspace: its own partitions of
// [start, ctx), after the prefix pass's partitions of [0, start).
__device__ __forceinline__ int own_partitions(int ctx, int start, int part_tokens)
{
    return ctx > start ? (ctx - start + part_tokens - 1) / part_tokens : 0;
}

// Partials of the shared prefix [0, start): partitions of part_tokens tokens
// (partial indices 0 .. n-1, ahead of the sequence's own partitions).
__device__ __forceinline__ int prefix_partitions(int start, int part_tokens)
{
    return start > 0 ? (start + part_tokens - 1) / part_tokens : 0;
}

// ---- split-context reduce ----------------------------------------------------------
//
// One CTA per (sequence, KV head).  For the G query heads of the group it
// merges the nparts partials (m_q, l_q, o_q) of a sequence that spans more
// than one partition: M = max_q m_q, w_q = l_q exp(m_q - M),
// out = sum_q w_q o_q / sum_q w_q.  Sequences with one partition were written
// by the partition pass itself.  With a shared prefix (start > 0) the first
// partials are the prefix pass's and the sequence's own partitions follow.
//
// One CTA per (sequence, run of R = reduce_heads query heads): R = 1 when
// the batch is small enough that a CTA per head keeps the grid below
// kReduceCtas (more threads per head, fewer trips to memory), else the G
// heads of a KV head (a grid of one CTA per head would cost more to
// schedule than it saves).  Thread (item, qg) -- item = (head, 8 consecutive
// d), QG = 256 / (R * D / 8) threads per item -- takes partitions q = qg,
// qg + QG, ... in chunks of kReduceUnroll whose loads are all issued before
// any is used, and keeps its own (M_t, L_t, A_t) with the same log-sum-exp
// rescaling; the QG threads of an item then combine theirs in shared
// memory.  After the context length, every global load of a chunk is
// independent, so a sequence with up to QG * kReduceUnroll partitions costs
// two dependent trips to memory (64 partitions at R = 1, d 128).
constexpr int kReduceThreads = 256;
constexpr int kReduceCtas = 1024;
#ifndef PA_REDUCE_UNROLL
#define PA_REDUCE_UNROLL 4
#endif
#ifndef PA_REDUCE_MINB
#define PA_REDUCE_MINB 3
#endif
// partitions whose loads are issued together per thread; CTAs per SM the
// register budget is sized for (3 x 256 threads, 85 registers; measured
// against 2 to 8 CTAs and unrolls of 2 to 8)
constexpr int kReduceUnroll = PA_REDUCE_UNROLL;

template <typename T, int D>
__global__ void __launch_bounds__(kReduceThreads, PA_REDUCE_MINB)
    paged_reduce_kernel(const __grid_constant__ DecodeParams p)
{
    using Op = MmaOp<T>;
    __shared__ __align__(16) float red_o[kReduceThreads * 8];
    __shared__ float red_m[kReduceThreads], red_l[kReduceThreads];
    pdl_wait_primary();  // the partition pass's partials are visible past here

    const int H = p.num_heads;
    const int R = p.reduce_heads;
    const int runs = H / R;
    const int s = blockIdx.x / runs;
    const int h0 = (blockIdx.x - s * runs) * R;  // first head of this CTA
    const int tid = threadIdx.x;
    const int ctx = clamp_context(p, s, false);
    const int start = seq_start_of(p, s, ctx);
    const int nparts = own_partitions(ctx, start, p.part_tokens) +
                       prefix_partitions(start, p.part_tokens);
    if (nparts == 0 || (nparts == 1 && start == 0))
        return;  // nothing to merge: the partition pass wrote the row
    if (p.counters != nullptr && nparts <= kMergeMax)
        return;  // merged by the partition pass

    // R * D / 8 <= 16 * 128 / 8 = kReduceThreads: one (item, qg) per thread.
    static_assert(16 * D / 8 <= kReduceThreads, "one work item per thread");
    const int items = R * (D / 8);
    const int qgroups = kReduceThreads / items;
    const bool active = tid < items * qgroups;
    const int item = tid % items;
    const int qg = tid / items;
    const int jh = item / (D / 8);
    const int d0 = (item - jh * (D / 8)) * 8;
    const size_t hrow = ((size_t)s * H + h0 + jh) * p.max_parts;

    float mt = -INFINITY, lt = 0.f;  // natural-log units, like the stored m_q
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (active) {
        for (int c0 = qg; c0 < nparts; c0 += qgroups * kReduceUnroll) {
            float cm[kReduceUnroll], cl[kReduceUnroll];
            float4 c_lo[kReduceUnroll], c_hi[kReduceUnroll];
#pragma unroll
            for (int u = 0; u < kReduceUnroll; ++u) {
                const int q = c0 + u * qgroups;
                if (q < nparts) {
                    cm[u] = p.part_m[hrow + q];
                    cl[u] = p.part_l[hrow + q];
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.part_o + (hrow + q) * D + d0);
                    c_lo[u] = src[0];
                    c_hi[u] = src[1];
                } else {
                    cm[u] = -INFINITY;
                    cl[u] = 0.f;
                    c_lo[u] = c_hi[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            // q = c0 < nparts, so the chunk's maximum is finite
            float mn = mt;
#pragma unroll
            for (int u = 0; u < kReduceUnroll; ++u)
                mn = fmaxf(mn, cm[u]);
            const float alpha = exp2f((mt - mn) * kLog2e);  // 0 while mt is -inf
            lt *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[e] *= alpha;
#pragma unroll
            for (int u = 0; u < kReduceUnroll; ++u) {
                const float w = cl[u] * exp2f((cm[u] - mn) * kLog2e);
                lt += w;
                acc[0] += w * c_lo[u].x; acc[1] += w * c_lo[u].y;
                acc[2] += w * c_lo[u].z; acc[3] += w * c_lo[u].w;
                acc[4] += w * c_hi[u].x; acc[5] += w * c_hi[u].y;
                acc[6] += w * c_hi[u].z; acc[7] += w * c_hi[u].w;
            }
            mt = mn;
        }
    }

    const size_t out_off = ((size_t)s * H + h0 + jh) * D + d0;
    if (qgroups == 1) {
        if (active) {
            const float inv = 1.f / lt;
            T vals[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                vals[e] = Op::from_float(acc[e] * inv);
            *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + out_off) =
                *reinterpret_cast<const uint4 *>(vals);
        }
        return;
    }
    if (active) {
        red_m[tid] = mt;
        red_l[tid] = lt;
        float4 *dst = reinterpret_cast<float4 *>(red_o + (size_t)tid * 8);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();
    if (tid >= items)
        return;
    // group 0 holds q = 0 < nparts: the maximum over groups is finite
    float mx = -INFINITY;
    for (int g2 = 0; g2 < qgroups; ++g2)
        mx = fmaxf(mx, red_m[g2 * items + tid]);
    float lsum = 0.f;
    float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int g2 = 0; g2 < qgroups; ++g2) {
        const int r = g2 * items + tid;
        const float w = exp2f((red_m[r] - mx) * kLog2e);  // 0 for a group with no partition
        lsum += w * red_l[r];
        const float4 *src = reinterpret_cast<const float4 *>(red_o + (size_t)r * 8);
        const float4 x0 = src[0], x1 = src[1];
        sum[0] += w * x0.x; sum[1] += w * x0.y; sum[2] += w * x0.z; sum[3] += w * x0.w;
        sum[4] += w * x1.x; sum[5] += w * x1.y; sum[6] += w * x1.z; sum[7] += w * x1.w;
    }
    const float inv = 1.f / lsum;
    T vals[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        vals[e] = Op::from_float(sum[e] * inv);
    *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + out_off) =
        *reinterpret_cast<const uint4 *>(vals);
}

// ---- the split-context merge fused into the pass ------------------------------------
//
// A partition unit of a sequence that spans several partitions leaves its
// partial (m, l, o) in the workspace and then arrives on the (sequence, KV
// head) counter; the warp whose arrival completes the count merges the
// partials -- by log-sum-exp weights, as paged_reduce_kernel does -- and
// writes the output row, so no reduce kernel runs after the pass.  The
// arrival is one acquire-release atomic by lane 0 after a warp barrier (the
// warp's partial stores come before it; the last arrival sees everyone's),
// the partials are read through L2, and the counter goes back to zero once
// its last arrival is in.  Merges are kept to at most kMergeMax partials:
// each costs the merging warp a round trip to L2 per batch of partials, and
// the pass's tile warps wait for the merge warp at their next unit's end;
// sequences with more partials are left to paged_reduce_kernel.

// The n (<= kMergeMax) partials of (s, kh) merged in index order by one warp
// into the output row.  Lane l takes items l, l + 32, ... (item = a query
// head's 8 consecutive elements of d), in blocks of up to 4 per lane; up to
// REC partial records per lane (at least one per item) are loaded before any
// is used.  NH: query heads per KV head the caller's kernel serves, at most.
// PT: the caller's parameters (part_m/l/o, out, num_heads, group,
// max_parts).
template <typename T, int D, int NH, int REC, typename PT>
__device__ __forceinline__ void warp_merge(const PT &p, int s, int kh, int n, int lane)
{
    constexpr int IPL = NH * (D / 8) / 32;          // items per lane, at most
    constexpr int IB = IPL < 4 ? IPL : 4;           // items per lane and block
    constexpr int QB = IB >= REC ? 1 : REC / IB;    // partials per item and batch
    static_assert(IPL >= 1 && NH * (D / 8) % 32 == 0 && IPL % IB == 0, "whole items per lane");
    const int G = p.group;
    const int items = G * (D / 8);
#pragma unroll 1
    for (int kb = 0; kb < IPL; kb += IB) {
        if (lane + 32 * kb >= items)
            break;
        float mt[IB], lt[IB], acc[IB][8];
        size_t hrow[IB];
        int d0[IB];
#pragma unroll
        for (int k = 0; k < IB; ++k) {
            const int it = lane + 32 * (kb + k);
            const int jh = it / (D / 8);
            d0[k] = (it - jh * (D / 8)) * 8;
            hrow[k] = ((size_t)s * p.num_heads + (size_t)kh * G + jh) * p.max_parts;
            mt[k] = -INFINITY;
            lt[k] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[k][e] = 0.f;
        }
        for (int qb = 0; qb < n; qb += QB) {
            float cm[IB][QB], cl[IB][QB];
            float4 lo[IB][QB], hi[IB][QB];
#pragma unroll
            for (int k = 0; k < IB; ++k)
#pragma unroll
                for (int b = 0; b < QB; ++b) {
                    const int q = qb + b;
                    if (lane + 32 * (kb + k) < items && q < n) {
                        const size_t idx = hrow[k] + q;
                        cm[k][b] = __ldcg(p.part_m + idx);
                        cl[k][b] = __ldcg(p.part_l + idx);
                        const float4 *src =
                            reinterpret_cast<const float4 *>(p.part_o + idx * D + d0[k]);
                        lo[k][b] = __ldcg(src);
                        hi[k][b] = __ldcg(src + 1);
                    } else {
                        cm[k][b] = -INFINITY;
                        cl[k][b] = 0.f;
                        lo[k][b] = hi[k][b] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
            for (int k = 0; k < IB; ++k) {
                float mn = mt[k];
#pragma unroll
                for (int b = 0; b < QB; ++b)
                    mn = fmaxf(mn, cm[k][b]);
                if (mn == -INFINITY)
                    continue;  // no partial of this item in the batch
                const float alpha = exp2f((mt[k] - mn) * kLog2e);  // 0 while mt is -inf
                lt[k] *= alpha;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[k][e] *= alpha;
#pragma unroll
                for (int b = 0; b < QB; ++b) {
                    const float w = cl[k][b] * exp2f((cm[k][b] - mn) * kLog2e);
                    lt[k] += w;
                    acc[k][0] += w * lo[k][b].x; acc[k][1] += w * lo[k][b].y;
                    acc[k][2] += w * lo[k][b].z; acc[k][3] += w * lo[k][b].w;
                    acc[k][4] += w * hi[k][b].x; acc[k][5] += w * hi[k][b].y;
                    acc[k][6] += w * hi[k][b].z; acc[k][7] += w * hi[k][b].w;
                }
                mt[k] = mn;
            }
        }
#pragma unroll
        for (int k = 0; k < IB; ++k) {
            const int it = lane + 32 * (kb + k);
            if (it >= items)
                continue;
            const int jh = it / (D / 8);
            const float inv = 1.f / lt[k];
            T vals[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                vals[e] = MmaOp<T>::from_float(acc[k][e] * inv);
            *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) +
                                       ((size_t)s * p.num_heads + (size_t)kh * G + jh) * D +
                                       d0[k]) = *reinterpret_cast<const uint4 *>(vals);
        }
    }
}

// Partials of sequence s in all: the prefix pass's partitions of its shared
// prefix [0, start) and its own partitions of [start, ctx) (the rule of the
// partition pass, with the same clamped context and checked start).
__device__ __forceinline__ int total_partitions(int ctx, int start, int part_tokens)
{
    return prefix_partitions(start, part_tokens) + own_partitions(ctx, start, part_tokens);
}

// One arrival of `add` head-rows of partials of (s, kh) (the counter of a
// sequence with n partials completes at n * G), made with an acquire-release
// atomic by the calling lane after its rows' stores are ordered before it
// (its own stores, or its warp's behind a __syncwarp).  Returns whether this
// arrival completed the count; the counter is then zero again.
__device__ __forceinline__ bool arrive_rows(int32_t *cnt, int add, int total)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(cnt), "r"(add)
                 : "memory");
    const bool last = old + add == total;
    if (last)
        *cnt = 0;  // every arrival is in: zero for the next call
    return last;
}

// The partition pass's arrival of one partial of (s, kh), all G heads, made
// by the merge warp right after it stored them; the warp completing the
// count writes the output row.
template <typename T, int D, int NH, int REC>
__device__ __forceinline__ void arrive_and_merge(const DecodeParams &p, int s, int kh, int ntot,
                                                 int lane)
{
    __syncwarp();  // the warp's partial stores come before lane 0's release
    int last = 0;
    if (lane == 0)
        last = arrive_rows(p.counters + (size_t)s * p.num_kv_heads + kh, p.group,
                           ntot * p.group);
    last = __shfl_sync(kFull, last, 0);  // the lanes' loads come after lane 0's acquire
    if (last)
        warp_merge<T, D, NH, REC>(p, s, kh, ntot, lane);
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

// Tensor map over a pool [num_blocks][block_size][num_kv_heads][head_dim]
// (dims d, head, token, block).  16-bit pools: a box of 64 elements x 1 head
// x 16 tokens x 1 block lands as 16 rows of 128 bytes with the 128-byte
// swizzle; a 16-token tile of one KV head takes head_dim / 64 boxes.  FP8
// pools: a box of head_dim one-byte elements (one row of 128 bytes, 128-byte
// swizzle; or of 64 bytes, 64-byte swizzle) x 1 head x 16 tokens x 1 block.
static bool encode_pool_map(CUtensorMap *map, const void *pool, pa_dtype dtype,
                            int num_blocks, int block_size, int num_kv_heads,
                            int head_dim)
{
    EncodeTiledFn fn = get_encode_fn();
    if (!fn)
        return false;
    const bool fp8 = dtype == PA_FP8_E4M3;
    const cuuint64_t e = fp8 ? 1 : 2;
    const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads,
                                (cuuint64_t)block_size, (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)head_dim * e,
                                   (cuuint64_t)num_kv_heads * head_dim * e,
                                   (cuuint64_t)block_size * num_kv_heads * head_dim * e};
    const cuuint32_t box[4] = {fp8 ? (cuuint32_t)head_dim : 64u, 1, (cuuint32_t)kTileTokens, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle swz =
        fp8 && head_dim == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    return fn(map, ty, 4, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    DecodeParams r = prm;
    const long long per_head = (long long)prm.num_seqs * prm.num_heads;
    r.reduce_heads = per_head <= kReduceCtas ? 1 : prm.group;
    return launch_pdl(paged_reduce_kernel<T, D>,
                      dim3((unsigned)(per_head / r.reduce_heads)), dim3(kReduceThreads), 0,
                      stream, r);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the split path: the arrival counters first (a region of at
// least kCounterWords words, so that calls of different sizes reusing one
// workspace find theirs at the same place, zero), then the partials.
struct WorkspaceLayout {
    size_t cnt_off, m_off, l_off, o_off, total;
};

static WorkspaceLayout workspace_layout(int S, int H, int Hkv, int D, int parts)
{
    WorkspaceLayout w{};
    if (parts <= 1)
        return w;
    const size_t words = std::max<size_t>(kCounterWords, (size_t)S * Hkv);
    const size_t ml = align256((size_t)S * H * parts * 4);
    w.cnt_off = 0;
    w.m_off = align256(words * 4);
    w.l_off = w.m_off + ml;
    w.o_off = w.l_off + ml;
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
    const WorkspaceLayout wl = workspace_layout(num_seqs, num_heads, num_kv_heads, head_dim,
                                                parts);
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
    prm->counters = wl.total ? reinterpret_cast<int32_t *>(ws + wl.cnt_off) : nullptr;
    prm->error_word = error_word;
    prm->wait_ns = stage_wait_limit_ns();
    prm->withhold_fill = withhold_first_fill();
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
