// pa_prefill.cu -- multi-query paged attention for sm_103a on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Two uses of one kernel:
//  * Chunked prefill and mixed batches ("PagedAttention & Continuous
//    Batching", §2.4 prefill vs decode, §2.5 chunked prefill): sequence s
//    brings its q_len newest tokens as query rows; chunk row i sits at
//    position pos = context_len - q_len + i and attends positions [0, pos]
//    of the paged pool (its own chunk's K/V were written by
//    reshape_and_cache before the call).  A decode request is q_len = 1.
//  * The shared-prefix pass of prefix-aware decode ("vLLM 架构详解",
//    "共享前缀的 Block 复用": several block tables naming the same physical
//    blocks): the decode queries of every member of a group attend each
//    partition of the group's shared prefix [0, L) once, read through the
//    first member's table, and leave a partial (m, l, o) per (sequence,
//    head, partition) to be merged with the members' own partitions -- by
//    whichever pass stores a sequence's last partial (the row warps here
//    arrive on the sequence's counter after their stores), or by the reduce
//    kernel for sequences of more than 8 partials.
//
// Design (GB300): a CTA takes 128 query rows of one KV head -- a chunk's
// tokens times the G query heads of the group, or the members' decode
// queries times G -- as the M = 128 dimension of tcgen05.mma tiles, and its
// seven warps split the work.  Warps 0-3 (one thread per row) write the rows
// into shared memory as the K-major A operand (128-byte swizzle) -- unless
// the tensor-core warp brings them by TMA in batches of more than one round
// (whole-token row tiles; over FP8 pools the row warps then round a bf16
// tile to fp16 in place) -- read each S row from tensor memory, apply the causal / range mask and the online
// softmax (fp32, log2 units, a reference maximum that moves only when a
// score exceeds it by 2^8, rescaling O in tensor memory then), and write P as
// bf16/fp16 pairs back over S, where it is the A operand of the value
// product.  Warps 4 and 5 look up the physical blocks and stream the keys,
// resp. the values, through a 2-stage ring of 64-token tiles by 4-D TMA loads
// (2 KB boxes, 128-byte swizzle) whose layout is directly the K-major B
// operand of S = Q K^T and the MN-major B operand of O += P V.  Warp 6 issues
// the MMAs from one elected lane: S of tile g into S buffer g % 2 as soon as
// its keys have landed and the buffer's previous P has been consumed, then
// the value product of tile g - 1, and commits each to an mbarrier that frees
// the ring stage or the S buffer it used.  S (128 x 64, fp32,
// double-buffered) and O (128 x d, fp32) live in tensor memory (256 columns,
// so two CTAs share an SM).  The roles meet only at mbarriers whose phase is
// the tile's index over the CTA's units / 2; every wait is bounded in time,
// the first to run out stops all roles, and tensor memory is released on
// every exit path.  Value rows past the key range are zeroed in shared
// memory before the value product, so a poisoned (NaN) slot never reaches
// the output.  FP8 (e4m3) pools: each tile lands as codes in the upper half
// of its 16-bit stage and is widened there to fp16 before the tensor-core
// warp may read it (keys by the row warps, values by the value warp); the
// products run in fp16 with the query rounded to fp16.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pa_decode_common.cuh"
#include "pa_prefill.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

// ---- fp32 helpers for the softmax ---------------------------------------------

// Maximum of three (max.f32 with three sources; a NaN source is ignored as
// in fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Two fp32 values in one 64-bit register, and packed fp32 FMA / add on them
// (fma.rn.f32x2 / add.rn.f32x2: each lane rounds as its scalar form).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t ffma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint64_t fadd_f32x2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

constexpr int kTcRows = 128;     // query rows per CTA (M of the MMAs)
constexpr int kRowWarps = 4;     // warps 0-3: one thread per row (softmax, epilogue)
constexpr int kKeyWarp = 4;      // table lookups and key fetches
constexpr int kValueWarp = 5;    // table lookups and value fetches
constexpr int kMmaWarp = 6;      // tensor-core issue
constexpr int kTcThreads = 32 * (kRowWarps + 3);
constexpr int kTcTokens = 64;    // key/value tokens per stage (N of S = Q K^T)
constexpr int kTcSubs = kTcTokens / kTileTokens;
constexpr int kTcStages = 2;
constexpr uint32_t kTmemCols = 256;  // S/P buffers at columns 0 and 64, O at column 128
constexpr uint32_t kTmemO = 128;
// Prefill batches whose units may take more than one round of the grid:
// segments (up to kMqOrderSegs of them) are numbered by their longest unit's
// key tiles, most first (a counting sort over kMqOrderBuckets buckets, stable
// by index), each segment's row tiles last-first, and the ranks are dealt
// boustrophedon (round r: CTA b takes rank r * grid + b, or r * grid + grid -
// 1 - b for odd r), so that a CTA that drew a long unit in one round draws a
// short one in the next.  The shared-prefix pass keeps the natural order and
// the round-robin deal.
constexpr int kMqOrderBuckets = 64;
constexpr int kMqOrderSegs = 512;

template <int D, bool kFp8> struct TcLayout {
    static constexpr int kHalves = D / 64;                    // 128-byte rows of 64 elements
    static constexpr int kQHalf = kTcRows * 128;              // 16 KB: 128 rows of one d-half
    static constexpr int kKVHalf = kTcTokens * 128;           // 8 KB: 64 tokens of one d-half
    static constexpr int kKVBytes = kHalves * kKVHalf;        // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kKVBytes;          // K then V
    static constexpr int kQ = kTcStages * kStageBytes;
    // FP8 pools: a tile's e4m3 codes (kTcTokens rows of D bytes) land in the
    // upper d-half of its 16-bit stage at d 128, in a region of their own
    // (stage-major, K then V) at d 64
    static constexpr int kCodeTile = kTcTokens * D;
    static constexpr int kCodes = kQ + kHalves * kQHalf;
    static constexpr int kCodesBytes = (kFp8 && D == 64) ? kTcStages * 2 * kCodeTile : 0;
    static constexpr int kBars = kCodes + kCodesBytes;        // 17 mbarriers
    static constexpr int kTmemSlot = kBars + 17 * 8;
    static constexpr int kAbort = kTmemSlot + 8;
    // int unit prefix[n + 1], then (ordered) order[n], units[n], key[n] and
    // the sort's buckets
    static constexpr int kSeg = kTmemSlot + 16;
    static size_t bytes(int segments, bool ordered)
    {
        return 1024 + kSeg + 4 * ((size_t)segments + 1) +
               (ordered ? 4 * (3 * (size_t)segments + kMqOrderBuckets) : 0);
    }
    static_assert(kStageBytes % 1024 == 0 && kQ % 1024 == 0, "1024-byte aligned operands");
};

// 3-D tiled bulk tensor load global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, uint32_t bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Context length of a chunked-prefill sequence, clamped like the decode pass.
__device__ __forceinline__ int clamp_context_mq(const MqParams &p, int s)
{
    const int limit = min(p.max_context_len, p.max_blocks_per_seq * p.block_size);
    int c = p.context_lens[s];
    if (c < 0 || c > limit) {
        flag_error(p.error_word, PA_DEVERR_CONTEXT_RANGE);
        c = c < 0 ? 0 : limit;
    }
    return c;
}

// Rows of one segment (a sequence's chunk, or a prefix group's members).
__device__ __forceinline__ int mq_segment_count(const MqParams &p, int seg)
{
    if (p.prefix_mode)
        return max(0, p.group_start[seg + 1] - p.group_start[seg]);
    return max(0, p.query_start[seg + 1] - p.query_start[seg]);
}

// Shared prefix length of a group, kept inside the table.
__device__ __forceinline__ int mq_group_prefix(const MqParams &p, int seg)
{
    return min(max(p.group_prefix[seg], 0), p.max_blocks_per_seq * p.block_size);
}

// Work units of a segment per KV head: row tiles (x prefix partitions).
__device__ __forceinline__ int mq_segment_units(const MqParams &p, int seg)
{
    const int tiles = (mq_segment_count(p, seg) * p.group + kTcRows - 1) / kTcRows;
    if (!p.prefix_mode)
        return tiles;
    return tiles * ((mq_group_prefix(p, seg) + p.part_tokens - 1) / p.part_tokens);
}

// kFp8: the pools hold e4m3 codes (head_dim 64 or 128).  The fetch warps land each 64-token FP8
// tile in the upper half of its 16-bit stage and widen it there to fp16 (the
// stage's K-major / MN-major operand layout, as a 16-bit fill leaves it),
// then release the stage; the products run in fp16 with the query rounded to
// fp16, the K scale folded into the exponent's scale and the V scale into
// the output.
template <typename T, int D, bool kFp8, bool kOrdered>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_mq_kernel(const __grid_constant__ MqParams p,
                    const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_q)
{
    using L = TcLayout<D, kFp8>;
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    using OT = typename std::conditional<kFp8, __half, T>::type;  // operand type
    constexpr bool kBf16 = std::is_same<OT, __nv_bfloat16>::value;
    constexpr uint32_t kIdescS = idesc_f16(kBf16, kTcRows, kTcTokens, false, false);
    constexpr uint32_t kIdescO = idesc_f16(kBf16, kTcRows, D, false, true);
    constexpr int KT = D / 16;  // MMAs of S = Q K^T (16 elements of d each)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);
    const uint32_t qbase = sbase + L::kQ;
    int *pref = reinterpret_cast<int *>(smem + L::kSeg);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbort);
    // mbarriers: K / V of stage st landed (fetch warp, transaction bytes);
    // S of buffer b computed (its commit also frees K stage b); value product
    // of stage st done (frees V stage st and S buffer st, makes O current);
    // P of buffer b stored by the 4 row warps; query tile in shared memory
    // (4 row warps, or one TMA transaction); every tensor-core operation of
    // the CTA done (drain)
    auto bar = [&](int i) { return sbase + L::kBars + 8 * i; };
    auto kfull = [&](int st) { return bar(st); };
    auto vfull = [&](int st) { return bar(2 + st); };
    auto sfull = [&](int b) { return bar(4 + b); };
    auto vfree = [&](int st) { return bar(6 + st); };
    auto pfull = [&](int b) { return bar(8 + b); };
    const uint32_t qfull = bar(10), mma_drain = bar(11);
    // FP8 pools: the codes of K / V stage st landed (before widening)
    auto kland = [&](int st) { return bar(12 + st); };
    auto vland = [&](int st) { return bar(14 + st); };
    // FP8 pools, bf16 queries, query tiles by TMA: the bf16 tile landed (the
    // row warps then round it to fp16 in place and arrive on qfull)
    constexpr bool kConvQ = kFp8 && std::is_same<T, __nv_bfloat16>::value;
    const uint32_t qland = bar(16);
    const uint32_t qtma_bar = kConvQ ? qland : qfull;
    auto kbase = [&](int st) { return sbase + st * L::kStageBytes; };
    // FP8 pools: where the codes of stage st's keys (values) land, and the
    // shared address of 16-byte chunk cc of code row r there (the TMA's
    // 128-byte swizzle for 128-byte rows, 64-byte swizzle for 64-byte rows)
    auto code_base = [&](int st, bool vals) -> uint32_t {
        if constexpr (D == 128)
            return kbase(st) + (vals ? L::kKVBytes : 0) + L::kKVHalf;
        else
            return sbase + L::kCodes + (st * 2 + (vals ? 1 : 0)) * L::kCodeTile;
    };
    auto code_chunk = [&](uint32_t cb, int r, int cc) -> uint32_t {
        if constexpr (D == 128)
            return cb + r * 128 + ((cc ^ (r & 7)) << 4);
        else
            return cb + r * 64 + ((cc ^ ((r >> 1) & 3)) << 4);
    };
    // fp16 chunk f (elements 8f .. 8f + 7) of row r of a 16-bit operand tile
    auto f16_chunk = [&](uint32_t tb, int r, int f) -> uint32_t {
        return tb + (f >> 3) * L::kKVHalf + r * 128 + (((f & 7) ^ (r & 7)) << 4);
    };
    // operand descriptors of stage 0 and of the query tile; other stages and
    // k-steps add their byte offset / 16 to the start-address field
    const uint64_t desc_q0 = smem_desc_sw128(qbase, 16, 1024);
    const uint64_t desc_k0 = smem_desc_sw128(sbase, 16, 1024);
    const uint64_t desc_v0 = smem_desc_sw128(sbase + L::kKVBytes, L::kKVHalf, 1024);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group, Hkv = p.num_kv_heads, H = p.num_heads;
    const int nseg = p.num_segments;

    if (tid == 0) {
        for (int st = 0; st < kTcStages; ++st) {
            // FP8 pools: the 4 row warps widen the keys, the value warp the values
            mbar_init(kfull(st), kFp8 ? kRowWarps : 1);
            mbar_init(vfull(st), 1);
            mbar_init(sfull(st), 1);
            mbar_init(vfree(st), 1);
            mbar_init(pfull(st), kRowWarps);
            mbar_init(kland(st), 1);
            mbar_init(vland(st), 1);
        }
        // the query tile: written by the 4 row warps, or one TMA transaction
        // (rounded to fp16 by the row warps after it lands, for kConvQ)
        mbar_init(qfull, (p.q_tma && !kConvQ) ? 1 : kRowWarps);
        mbar_init(qland, 1);
        mbar_init(mma_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
        if (p.q_tma)
            prefetch_tensormap(&tmap_q);
    }
    // Everything from here on comes after the kernel before this one on the
    // stream has finished -- including an earlier launch of this kernel, so
    // the tensor memory below is never contended by one.
    pdl_wait_primary();
    // the shared-prefix pass lets the partition pass after it start at once
    // (that pass reads nothing this one writes, and waits for this grid
    // before it finishes)
    if (p.prefix_mode)
        pdl_launch_dependents();
    // tensor memory: one warp allocates, every thread reads the address
    if (warp == 0) {
        tmem_alloc(sbase + L::kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);

    // ---- work units per segment and their prefix sums -------------------------------
    int *order = pref + nseg + 1;  // k-th segment of the unit order (kOrdered)
    int *seg_units = order + nseg;
    if (warp == 0) {
        if constexpr (kOrdered) {
            // counting sort by the key tiles of the segment's last row tile
            // (its context), most first, by index within a count; every CTA
            // computes the same order.  Each segment's loads are issued once.
            int *seg_key = seg_units + nseg;
            int *hist = seg_key + nseg;
            hist[lane] = 0;
            hist[lane + 32] = 0;
            __syncwarp();
            for (int sg = lane; sg < nseg; sg += 32) {
                const int tiles = (clamp_context_mq(p, sg) + kTcTokens - 1) / kTcTokens;
                const int key = kMqOrderBuckets - 1 - min(tiles, kMqOrderBuckets - 1);
                seg_units[sg] = mq_segment_units(p, sg);
                seg_key[sg] = key;
                atomicAdd(&hist[key], 1);
            }
            __syncwarp();
            const int c0 = hist[2 * lane], c1 = hist[2 * lane + 1];
            int x = c0 + c1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, x, o);
                if (lane >= o)
                    x += y;
            }
            __syncwarp();
            hist[2 * lane] = x - c0 - c1;  // first place of each count
            hist[2 * lane + 1] = x - c1;
            __syncwarp();
            for (int base = 0; base < nseg; base += 32) {
                const int sg = base + lane;
                const int key = sg < nseg ? seg_key[sg] : -1;
                const unsigned same = __match_any_sync(kFull, key);
                const int rank = __popc(same & ((1u << lane) - 1u));
                const int off = key >= 0 ? hist[key] : 0;
                __syncwarp();
                if (key >= 0) {
                    order[off + rank] = sg;
                    if (rank == 0)
                        hist[key] = off + __popc(same);
                }
                __syncwarp();
            }
        }
        int carry = 0;
        for (int base = 0; base < nseg; base += 32) {
            const int k = base + lane;
            int n = 0;
            if (k < nseg) {
                if constexpr (kOrdered)
                    n = seg_units[order[k]];
                else
                    n = mq_segment_units(p, k);
            }
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, x, o);
                if (lane >= o)
                    x += y;
            }
            if (k < nseg)
                pref[k] = carry + x - n;
            carry += __shfl_sync(kFull, x, 31);
        }
        if (lane == 0)
            pref[nseg] = carry;
    }
    __syncthreads();
    const int total_units = pref[nseg] * Hkv;
    // this CTA's unit after unit u in the deal (its first unit is blockIdx.x)
    auto next_unit = [&](int u) -> int {
        const int grid = gridDim.x;
        if constexpr (kOrdered) {
            const int r = u / grid + 1;  // the next round
            return r * grid + ((r & 1) ? grid - 1 - (int)blockIdx.x : (int)blockIdx.x);
        } else {
            return u + grid;
        }
    };

    // ---- unit -> (segment, KV head, row tile, prefix partition, key range) -------------
    // Every role walks the same units in the same order and counts the same
    // 64-token tiles, so a tile's global index g (across this CTA's units)
    // names its ring stage g % 2, its S buffer g % 2 and the phase g / 2 of
    // every barrier of that stage.
    struct Unit {
        int seg, kh, rt, part, count, nrows, kbeg, kend, n;
        const int32_t *table;
    };
    auto decode = [&](int u, Unit &w) {
        const int q = u / Hkv;
        w.kh = u - q * Hkv;
        int lo = 0, hi = nseg - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pref[mid] <= q)
                lo = mid;
            else
                hi = mid - 1;
        }
        w.seg = kOrdered ? order[lo] : lo;
        w.count = mq_segment_count(p, w.seg);
        const int tiles = (w.count * G + kTcRows - 1) / kTcRows;
        // ordered: the segment's row tiles last-first
        const int idx = kOrdered ? pref[lo + 1] - 1 - q : q - pref[lo];
        w.rt = idx % tiles;    // row tile
        w.part = idx / tiles;  // prefix partition (0 for prefill)
        w.nrows = min(kTcRows, w.count * G - w.rt * kTcRows);
        int table_seq;
        if (p.prefix_mode) {
            // a bad leader id is flagged by the plan check of the row warps
            table_seq = min(max(p.group_members[p.group_start[w.seg]], 0), p.num_seqs - 1);
            w.kbeg = w.part * p.part_tokens;
            w.kend = min(mq_group_prefix(p, w.seg), w.kbeg + p.part_tokens);
        } else {
            table_seq = w.seg;
            const int ctx = clamp_context_mq(p, w.seg);
            const int last = (w.rt * kTcRows + w.nrows - 1) / G;  // chunk row of the last row
            w.kbeg = 0;
            w.kend = max(0, ctx - w.count + last + 1);
        }
        w.table = p.block_tables + (size_t)table_seq * p.max_blocks_per_seq;
        w.n = w.kend > w.kbeg ? (w.kend - w.kbeg + kTcTokens - 1) / kTcTokens : 0;
    };
    // a bounded wait, warp-uniform; the first one to run out stops every role
    // (the abort flag is read only when the phase is not already complete)
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        if (__all_sync(kFull, mbar_try_wait(b, parity)))
            return true;
        bool ok = *abort_flag == 0 && mbar_wait_bounded(b, parity, p.wait_ns);
        ok = __all_sync(kFull, ok);
        if (!ok)
            *abort_flag = 1;
        return ok;
    };

    if (warp < kRowWarps) {
        // ===== row warps: query rows in, online softmax, P out, epilogue ===============
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;  // this warp's TMEM lanes
        uint32_t g = 0;
        bool ok = true;
        // this thread's row of a unit: query row, output location, key limit
        struct Row {
            long long qoff, ooff;
            int lim, seq;
        };
        auto row_of = [&](const Unit &w, Row &r, bool check) {
            // prefix pass, first KV head and partition: check the plan for this
            // tile's members -- the prefix is on the tile grid and within every
            // member's context, each member records it as its start, and each
            // member's table names the leader's blocks for the whole prefix
            if (check && p.prefix_mode && w.kh == 0 && w.part == 0 && tid < w.nrows &&
                (w.rt * kTcRows + tid) % G == 0) {
                const int s = p.group_members[p.group_start[w.seg] + (w.rt * kTcRows + tid) / G];
                const int Lg = p.group_prefix[w.seg];
                const int leader = p.group_members[p.group_start[w.seg]];
                bool bad = s < 0 || s >= p.num_seqs || Lg <= 0 ||
                           (Lg & (kTileTokens - 1)) != 0 ||
                           Lg > p.max_blocks_per_seq * p.block_size || leader < 0 ||
                           leader >= p.num_seqs;
                if (!bad) {
                    const int c = p.context_lens[s];
                    bad = c < Lg || c > p.max_context_len || p.seq_start[s] != Lg;
                    const int32_t *mine = p.block_tables + (size_t)s * p.max_blocks_per_seq;
                    for (int bk = 0; !bad && bk < (Lg >> p.block_shift); ++bk)
                        bad = __ldg(mine + bk) != __ldg(w.table + bk);
                }
                if (bad)
                    flag_error(p.error_word, PA_DEVERR_PREFIX_PLAN);
            }
            r.qoff = -1;
            r.ooff = -1;
            r.lim = 0;
            r.seq = -1;
            if (tid < w.nrows) {
                const int rr = w.rt * kTcRows + tid;
                const int i = rr / G, hg = rr - (rr / G) * G;
                const int h = w.kh * G + hg;
                if (p.prefix_mode) {
                    int sq = p.group_members[p.group_start[w.seg] + i];
                    sq = min(max(sq, 0), p.num_seqs - 1);  // a bad member id is flagged above
                    r.seq = sq;
                    r.qoff = ((long long)sq * H + h) * D;
                    r.ooff = ((long long)sq * H + h) * p.max_parts + w.part;
                    r.lim = w.kend;
                } else {
                    const long long row = (long long)p.query_start[w.seg] + i;
                    r.qoff = (row * H + h) * D;
                    r.ooff = r.qoff;
                    const int last = (w.rt * kTcRows + w.nrows - 1) / G;
                    r.lim = max(0, w.kend - (last - i));
                }
            }
        };
        // the next unit's query row is pulled into L2 while the current unit's
        // last value product runs and its output is written
        auto prefetch_q = [&](const Unit &w, const Row &r) {
            if (w.n > 0 && r.qoff >= 0) {
                const char *src = reinterpret_cast<const char *>(static_cast<const T *>(p.query) +
                                                                 r.qoff);
#pragma unroll
                for (int c = 0; c < D * (int)sizeof(T); c += 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(src + c));
            }
        };
        // a unit's query rows -> shared memory (K-major, 128-byte swizzle;
        // zeros past the tile), announced to the MMA warp.  Called once every
        // S of the unit before has finished (they read the query tile).
        bool q_over = false;  // FP8 pools: a bf16 query element past the fp16 range
        auto write_q = [&](const Unit &w, const Row &r) {
            if (w.n <= 0)
                return;
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.query) +
                                                               (r.qoff < 0 ? 0 : r.qoff));
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                uint4 v = r.qoff >= 0 ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                if constexpr (kFp8 && std::is_same<T, __nv_bfloat16>::value) {
                    // the fp16 operand: a bf16 element past the fp16 range is flagged
                    uint32_t *wv = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float lo = __uint_as_float(wv[k] << 16);
                        const float hi = __uint_as_float(wv[k] & 0xffff0000u);
                        q_over |= fmaxf(fabsf(lo), fabsf(hi)) > 65504.f;
                        wv[k] = pack_f16x2(lo, hi);
                    }
                }
                const uint32_t a = qbase + (c >> 3) * L::kQHalf + tid * 128 +
                                   (((c & 7) ^ (tid & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x),
                             "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(qfull);
        };
        // kConvQ with q_tma: a unit's bf16 query tile has landed by TMA; each
        // thread rounds its own row to fp16 in place (same swizzled chunks),
        // flags a bf16 element past the fp16 range, and the row warps
        // announce the tile on qfull.
        uint32_t nql = 0;  // bf16 query tiles waited for
        auto convert_q = [&](const Unit &w) -> bool {
            if (w.n <= 0)
                return true;
            if (!wait(qland, nql & 1))
                return false;
            ++nql;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint32_t a = qbase + (c >> 3) * L::kQHalf + tid * 128 +
                                   (((c & 7) ^ (tid & 7)) << 4);
                uint32_t wv[4];
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(wv[0]), "=r"(wv[1]), "=r"(wv[2]), "=r"(wv[3])
                             : "r"(a)
                             : "memory");
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = __uint_as_float(wv[k] << 16);
                    const float hi = __uint_as_float(wv[k] & 0xffff0000u);
                    q_over |= fmaxf(fabsf(lo), fabsf(hi)) > 65504.f;
                    wv[k] = pack_f16x2(lo, hi);
                }
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(wv[0]),
                             "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(qfull);
            return true;
        };
        // FP8 pools: the row warps widen each key tile in place once its codes
        // have landed (see the fetch warps), two threads per 128-code row, and
        // announce it on the stage's "keys full" barrier.  Tile gg + 1 is widened
        // before the row warps wait for S of tile gg, so it is ready when the
        // tensor-core warp moves on.
        int ntiles_cta = 0;  // tiles of this CTA, over all its units
        if constexpr (kFp8) {
            for (int u = blockIdx.x; u < total_units; u = next_unit(u)) {
                Unit x;
                decode(u, x);
                ntiles_cta += x.n;
            }
        }
        auto widen_k = [&](uint32_t gg) -> bool {
            const uint32_t st = gg & 1;
            if (!wait(kland(st), (gg >> 1) & 1))
                return false;
            const uint32_t base = kbase(st), cb = code_base(st, false);
            // row r; this thread's half of its code chunks (16 codes each)
            constexpr int kCh = D / 32;
            const int r = tid >> 1, h = tid & 1;
            uint4 src[kCh];
#pragma unroll
            for (int j = 0; j < kCh; ++j) {
                const uint32_t a = code_chunk(cb, r, h * kCh + j);
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(src[j].x), "=r"(src[j].y), "=r"(src[j].z), "=r"(src[j].w)
                             : "r"(a)
                             : "memory");
            }
            __syncwarp();  // (d 128) the row is read before d-half 1 overwrites its codes
#pragma unroll
            for (int c = 0; c < 2 * kCh; ++c) {
                // fp16 chunk f = codes 8f .. 8f + 7
                const int f = 2 * h * kCh + c;
                const uint4 sc = src[c >> 1];
                const uint32_t lo = (c & 1) ? sc.z : sc.x;
                const uint32_t hi = (c & 1) ? sc.w : sc.y;
                const uint32_t a = f16_chunk(base, r, f);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                             "r"(e4m3x2_to_f16x2((uint16_t)(lo & 0xffffu))),
                             "r"(e4m3x2_to_f16x2((uint16_t)(lo >> 16))),
                             "r"(e4m3x2_to_f16x2((uint16_t)(hi & 0xffffu))),
                             "r"(e4m3x2_to_f16x2((uint16_t)(hi >> 16)))
                             : "memory");
            }
            fence_proxy_async_smem();  // the widened tile, for the tensor cores
            __syncwarp();
            if (lane == 0)
                mbar_arrive(kfull(st));
            return true;
        };
        Unit w;
        Row rw;
        if ((int)blockIdx.x < total_units) {
            decode(blockIdx.x, w);
            row_of(w, rw, true);
            if (!p.q_tma)  // (else the tensor-core warp brings it by TMA)
                write_q(w, rw);
            else if constexpr (kConvQ)
                ok = convert_q(w);
        }
        if constexpr (kFp8) {
            if (ok && ntiles_cta > 0)
                ok = widen_k(0);
        }
        for (int u = blockIdx.x; u < total_units && ok; u = next_unit(u)) {
            const long long ooff = rw.ooff;
            const int lim = rw.lim;
            const int u_next = next_unit(u);
            const bool has_next = u_next < total_units;
            if (has_next) {
                // the next unit's query rows, pulled into L2 while this unit runs
                Unit wn;
                Row rn;
                decode(u_next, wn);
                row_of(wn, rn, false);
                prefetch_q(wn, rn);
            }
            float m_ref = -INFINITY, l_run = 0.f;
            if (w.n > 0) {
                for (int si = 0; si < w.n; ++si) {
                    const uint32_t gg = g + si, b = gg & 1;
                    const int t0 = w.kbeg + si * kTcTokens;
                    if constexpr (kFp8) {
                        if ((int)gg + 1 < ntiles_cta) {
                            ok = widen_k(gg + 1);
                            if (!ok)
                                break;
                        }
                    }
                    // 1. S of this tile
                    ok = wait(sfull(b), (gg >> 1) & 1);
                    if (!ok)
                        break;
                    tc_fence_after();

                    // 2. softmax of this thread's row: raw scores (q . k); the
                    //    scale is applied inside the exponent
                    float sv[kTcTokens];
                    {
                        uint32_t r[kTcTokens];
                        tmem_ld_32x32b_x64(tmem + lane_base + b * kTcTokens, r);
#pragma unroll
                        for (int i = 0; i < kTcTokens; ++i)
                            sv[i] = __uint_as_float(r[i]);
                    }
                    if (lim < t0 + kTcTokens) {  // causal / range mask (diagonal, last tiles)
#pragma unroll
                        for (int i = 0; i < kTcTokens; ++i)
                            sv[i] = t0 + i < lim ? sv[i] : -INFINITY;
                    }
                    // maximum raw score (the scale is positive): a tree of
                    // three-input maxima, 64 -> 22 -> 8 -> 3 -> 1
                    static_assert(kTcTokens == 64, "max tree sized for 64 keys");
                    float m22[22], m8[8];
#pragma unroll
                    for (int k = 0; k < 21; ++k)
                        m22[k] = fmax3(sv[3 * k], sv[3 * k + 1], sv[3 * k + 2]);
                    m22[21] = sv[63];
#pragma unroll
                    for (int k = 0; k < 7; ++k)
                        m8[k] = fmax3(m22[3 * k], m22[3 * k + 1], m22[3 * k + 2]);
                    m8[7] = m22[21];
                    const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                                           fmaxf(m8[6], m8[7])) *
                                     p.scale_log2;  // -inf for a fully masked row
                    // the reference maximum moves only when a score passes it by 2^kSlack
                    const bool moved = mx > m_ref + kSlack;
                    float alpha = 1.f;
                    if (moved) {
                        alpha = exp2f(m_ref - mx);  // 0 while m_ref is -inf
                        m_ref = mx;
                        l_run *= alpha;
                    }
                    const float neg_mu = m_ref == -INFINITY ? 0.f : -m_ref;
                    // exponents two at a time (packed fp32 FMA), weights
                    // summed in two packed accumulators
                    uint32_t pw[kTcTokens / 2];
                    const uint64_t sl2 = pack_f32x2(p.scale_log2, p.scale_log2);
                    const uint64_t nm2 = pack_f32x2(neg_mu, neg_mu);
                    uint64_t acc[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
#pragma unroll
                    for (int i = 0; i < kTcTokens / 2; ++i) {
                        float e0, e1;
                        unpack_f32x2(ffma_f32x2(pack_f32x2(sv[2 * i], sv[2 * i + 1]), sl2, nm2),
                                     e0, e1);
                        const float p0 = exp2f(e0), p1 = exp2f(e1);
                        acc[i & 1] = fadd_f32x2(acc[i & 1], pack_f32x2(p0, p1));
                        pw[i] = MmaOp<OT>::pack(p0, p1);
                    }
                    {
                        float a0, a1, b0, b1;
                        unpack_f32x2(acc[0], a0, a1);
                        unpack_f32x2(acc[1], b0, b1);
                        l_run += (a0 + a1) + (b0 + b1);
                    }

                    // 3. a row's reference maximum moved: rescale O in tensor
                    //    memory once the previous tile's value product is done
                    //    (the next one waits for this tile's P, below)
                    if (si > 0 && __any_sync(kFull, moved)) {
                        const uint32_t gp = gg - 1;
                        ok = wait(vfree(gp & 1), (gp >> 1) & 1);
                        if (!ok)
                            break;
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t r[32];
                            tmem_ld_32x32b_x32(tmem + lane_base + kTmemO + c * 32, r);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                            tmem_st_32x32b_x32(tmem + lane_base + kTmemO + c * 32, r);
                        }
                    }
                    // 4. P over this tile's S (A operand of the value product)
                    tmem_st_32x32b_x32(tmem + lane_base + b * kTcTokens, pw);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(pfull(b));
                }
                if (!ok)
                    break;
            }
            // every S of this unit has finished: the next unit's query rows go
            // into shared memory now (unless the tensor-core warp brings them
            // by TMA), so its first S can run during this unit's last value
            // product and epilogue
            Unit wn;
            Row rn;
            if (has_next) {
                decode(u_next, wn);
                row_of(wn, rn, true);
                if (!p.q_tma)
                    write_q(wn, rn);
                else if constexpr (kConvQ) {
                    ok = convert_q(wn);
                    if (!ok)
                        break;
                }
            } else {
                wn.n = 0;
                rn.qoff = rn.ooff = -1;
                rn.lim = 0;
                rn.seq = -1;
            }
            // this unit's last value product
            if (w.n > 0) {
                const uint32_t gl = g + w.n - 1;
                ok = wait(vfree(gl & 1), (gl >> 1) & 1);
                tc_fence_after();
                if (!ok)
                    break;
            }

            // epilogue: this thread's row of O / l (TMEM loads are warp-wide)
            const float inv = (w.n > 0 && l_run > 0.f) ? p.out_scale / l_run : 0.f;
            const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
            if (p.prefix_mode && ooff >= 0) {
                p.part_m[ooff] = m_ref * kLn2;
                p.part_l[ooff] = l_run;
            }
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t r[64];
                if (w.n > 0) {
                    tmem_ld_32x32b_x64(tmem + lane_base + kTmemO + c * 64, r);
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        r[i] = 0u;
                }
                if (ooff < 0)
                    continue;
                if (p.prefix_mode) {
                    float4 *dst = reinterpret_cast<float4 *>(p.part_o + ooff * D) + c * 16;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv,
                                             __uint_as_float(r[4 * i + 1]) * inv,
                                             __uint_as_float(r[4 * i + 2]) * inv,
                                             __uint_as_float(r[4 * i + 3]) * inv);
                } else if (out32) {
                    // 32-byte stores: half the store instructions of 16-byte ones
                    // for the row's 256-byte run (rows sit 256 bytes apart)
                    T *dst = static_cast<T *>(p.out) + ooff + c * 64;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t v[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            v[k] = MmaOp<T>::pack(__uint_as_float(r[16 * i + 2 * k]) * inv,
                                                  __uint_as_float(r[16 * i + 2 * k + 1]) * inv);
                        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                                         dst + 16 * i),
                                     "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]),
                                     "r"(v[5]), "r"(v[6]), "r"(v[7])
                                     : "memory");
                    }
                } else {
                    uint4 *dst =
                        reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + ooff) + c * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        uint4 v;
                        v.x = MmaOp<T>::pack(__uint_as_float(r[8 * i]) * inv,
                                             __uint_as_float(r[8 * i + 1]) * inv);
                        v.y = MmaOp<T>::pack(__uint_as_float(r[8 * i + 2]) * inv,
                                             __uint_as_float(r[8 * i + 3]) * inv);
                        v.z = MmaOp<T>::pack(__uint_as_float(r[8 * i + 4]) * inv,
                                             __uint_as_float(r[8 * i + 5]) * inv);
                        v.w = MmaOp<T>::pack(__uint_as_float(r[8 * i + 6]) * inv,
                                             __uint_as_float(r[8 * i + 7]) * inv);
                        dst[i] = v;
                    }
                }
            }
            // prefix pass: this row's partial is stored; arrive on the
            // sequence's counter (one head-row), and a warp whose lane
            // completed a count merges that sequence's partials into its
            // output row
            if (p.prefix_mode && p.counters != nullptr) {
                const int sq = rw.seq;
                int ntot = 0;
                bool last = false;
                if (ooff >= 0) {
                    const int limit = min(p.max_context_len, p.max_blocks_per_seq * p.block_size);
                    const int c = min(max(p.context_lens[sq], 0), limit);
                    int st = p.seq_start[sq];
                    st = (st < 0 || st > c || (st & (kTileTokens - 1)) != 0) ? 0 : st;
                    ntot = total_partitions(c, st, p.part_tokens);
                    if (ntot <= kMergeMax)
                        last = arrive_rows(p.counters + (size_t)sq * Hkv + w.kh, 1, ntot * G);
                }
                unsigned todo = __ballot_sync(kFull, last);
                while (todo != 0) {
                    const int src = __ffs(todo) - 1;
                    todo &= todo - 1;
                    const int ms = __shfl_sync(kFull, sq, src);
                    const int mn = __shfl_sync(kFull, ntot, src);
                    warp_merge<T, D, 16, 4>(p, ms, w.kh, mn, lane);
                }
            }
            g += w.n;
            w = wn;
            rw = rn;
        }
        if (kFp8 && __any_sync(kFull, q_over) && lane == 0)
            flag_error(p.error_word, PA_DEVERR_QUERY_RANGE);
    } else if (warp == kKeyWarp || warp == kValueWarp) {
        // ===== fetch warps: keys (warp 4) and values (warp 5) into the 2-stage ring ====
        // Lane j < 2 * kTcSubs (j < kTcSubs for d = 64) owns the 16-token
        // sub-tile j / halves and d-half j % halves of every tile: it looks up
        // that sub-tile's physical block one tile ahead of its use and issues
        // its own 2 KB box.  K of tile g goes out once S of tile g - 2 is done,
        // V of tile g once the value product of tile g - 2 is.
        const bool values = warp == kValueWarp;
        // FP8: one box of 16 whole 128-byte rows per sub-tile
        const int my_sb = kFp8 ? lane : lane / L::kHalves;
        const int my_hf = kFp8 ? 0 : lane % L::kHalves;
        uint32_t g = 0;
        int last0 = -1, last1 = -1;  // last fill per stage
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u = next_unit(u)) {
            Unit w;
            decode(u, w);
            auto lookup = [&](int si) {
                const int tok = w.kbeg + si * kTcTokens + my_sb * kTileTokens;
                int e = (my_sb < kTcSubs && tok < w.kend)
                            ? __ldg(w.table + (tok >> p.block_shift))
                            : 0;
                return e;
            };
            auto checked = [&](int e) {
                if (e < 0 || e >= p.num_blocks) {
                    flag_error(p.error_word, PA_DEVERR_BLOCK_RANGE);
                    e = 0;  // stays inside the pool; the row's output is undefined
                }
                return e;
            };
            auto issue = [&](int si, uint32_t st, int ent) {
                const int t0 = w.kbeg + si * kTcTokens;
                const int nsub = min(kTcSubs, (w.kend - t0 + kTileTokens - 1) / kTileTokens);
                if constexpr (kFp8) {
                    // the codes land where code_base says: one box of 16 rows
                    // of D codes per sub-tile
                    const uint32_t fb = values ? vland(st) : kland(st);
                    if (lane == 0)
                        mbar_arrive_expect_tx(fb, (uint32_t)(nsub * kTileTokens * D));
                    __syncwarp();
                    if (my_sb < nsub) {
                        const int row = (t0 + my_sb * kTileTokens) & (p.block_size - 1);
                        tma_load_4d(code_base(st, values) + my_sb * kTileTokens * D,
                                    values ? &tmap_v : &tmap_k, fb, 0, w.kh, row, ent);
                    }
                } else {
                    const uint32_t fb = values ? vfull(st) : kfull(st);
                    if (lane == 0)
                        mbar_arrive_expect_tx(fb, (uint32_t)(nsub * L::kHalves * 2048));
                    __syncwarp();
                    if (my_sb < nsub) {
                        const int row = (t0 + my_sb * kTileTokens) & (p.block_size - 1);
                        tma_load_4d(kbase(st) + (values ? L::kKVBytes : 0) + my_hf * L::kKVHalf +
                                        my_sb * 2048,
                                    values ? &tmap_v : &tmap_k, fb, my_hf * 64, w.kh, row, ent);
                    }
                }
                return nsub;
            };
            // FP8: widen the tile's landed codes in place -- row r's 128 codes
            // (128-byte swizzled row r of the upper half) become fp16 row r of
            // d-half 0 (d 0..63) and of d-half 1 (d 64..127, over the codes'
            // own row: each lane reads its whole row before writing it) --
            // then hand the stage to the tensor-core warp.
            auto widen = [&](uint32_t gg, int nsub) -> bool {
                const uint32_t st = gg & 1;
                if (!wait(values ? vland(st) : kland(st), (gg >> 1) & 1))
                    return false;
                const uint32_t base = kbase(st) + (values ? L::kKVBytes : 0);
                const uint32_t cb = code_base(st, values);
                for (int r = lane; r < nsub * kTileTokens; r += 32) {
                    uint4 src[D / 16];
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) {
                        const uint32_t a = code_chunk(cb, r, c);
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(src[c].x), "=r"(src[c].y), "=r"(src[c].z),
                                       "=r"(src[c].w)
                                     : "r"(a)
                                     : "memory");
                    }
#pragma unroll
                    for (int f = 0; f < D / 8; ++f) {
                        // fp16 chunk f = codes 8f .. 8f + 7
                        const uint4 sc = src[f >> 1];
                        const uint32_t lo = (f & 1) ? sc.z : sc.x;
                        const uint32_t hi = (f & 1) ? sc.w : sc.y;
                        const uint32_t a = f16_chunk(base, r, f);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                                     "r"(e4m3x2_to_f16x2((uint16_t)(lo & 0xffffu))),
                                     "r"(e4m3x2_to_f16x2((uint16_t)(lo >> 16))),
                                     "r"(e4m3x2_to_f16x2((uint16_t)(hi & 0xffffu))),
                                     "r"(e4m3x2_to_f16x2((uint16_t)(hi >> 16)))
                                     : "memory");
                    }
                }
                fence_proxy_async_smem();  // the widened tile, for the tensor cores
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(values ? vfull(st) : kfull(st));
                return true;
            };
            // FP8: a tile is widened after the next one has been issued, so
            // that one's fill is in flight meanwhile
            int pend = -1, pend_nsub = 0;
            int ent_next = w.n > 0 ? lookup(0) : 0;
            for (int si = 0; si < w.n; ++si) {
                const uint32_t gg = g + si, st = gg & 1;
                const int ent = checked(ent_next);
                if (si + 1 < w.n)
                    ent_next = lookup(si + 1);
                // the stage's tile gg - 2 is consumed: its S (keys), its
                // value product (values)
                if (gg >= kTcStages) {
                    ok = wait(values ? vfree(st) : sfull(st), ((gg - 2) >> 1) & 1);
                    if (!ok)
                        break;
                }
                // test hook of the time-out path: a CTA's first key fill is
                // never issued, so the wait for it runs out
                if (p.withhold_fill != 0 && !values && gg == 0)
                    continue;
                const int nsub = issue(si, st, ent);
                (st ? last1 : last0) = (int)gg;
                if constexpr (kFp8) {
                    if (values) {  // (the row warps widen the keys)
                        if (pend >= 0) {
                            ok = widen(g + pend, pend_nsub);
                            if (!ok)
                                break;
                        }
                        pend = si;
                        pend_nsub = nsub;
                    }
                }
            }
            if constexpr (kFp8) {
                if (values && ok && pend >= 0)
                    ok = widen(g + pend, pend_nsub);
            }
            g += w.n;
        }
        // fills still landing (only after an abort: the MMA warp -- or, for
        // FP8 pools, the widening -- waited the rest)
        const uint32_t landed0 = kFp8 ? (values ? vland(0) : kland(0)) : (values ? vfull(0) : kfull(0));
        const uint32_t landed1 = kFp8 ? (values ? vland(1) : kland(1)) : (values ? vfull(1) : kfull(1));
        if (last0 >= 0)
            mbar_wait_bounded(landed0, (last0 >> 1) & 1, kDrainWaitNs);
        if (last1 >= 0)
            mbar_wait_bounded(landed1, (last1 >> 1) & 1, kDrainWaitNs);
    } else if (warp == kMmaWarp) {
        // ===== tensor-core warp: S = Q K^T and O += P V, one elected lane issues ========
        uint32_t g = 0, nq = 0;
        bool ok = true;
        // O += P V of tile gg (tile si of unit w): P stored, V landed; value rows
        // past the key range are zeroed first (never fetched, or past the context)
        auto issue_pv = [&](const Unit &w, int si, uint32_t gg) -> bool {
            const uint32_t st = gg & 1;
            if (!wait(pfull(st), (gg >> 1) & 1) || !wait(vfull(st), (gg >> 1) & 1))
                return false;
            const int nvalid = w.kend - (w.kbeg + si * kTcTokens);
            if (nvalid < kTcTokens) {
                const int rows = kTcTokens - nvalid;
                for (int c = lane; c < L::kHalves * rows * 8; c += 32) {
                    const int hf = c / (rows * 8), rem = c - hf * rows * 8;
                    const uint32_t a = kbase(st) + L::kKVBytes + hf * L::kKVHalf +
                                       (nvalid + rem / 8) * 128 + (rem % 8) * 16;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0)
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc_fence_after();
            const uint64_t dv = desc_v0 + (uint64_t)((st * L::kStageBytes) >> 4);
            if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < kTcTokens / 16; ++ks)
                    tc_mma_ts(tmem + kTmemO, tmem + st * kTcTokens + ks * 8,
                              dv + (uint64_t)((ks * 2048) >> 4), kIdescO,
                              (si > 0 || ks > 0) ? 1u : 0u);
                tc_commit(vfree(st));
            }
            return true;
        };
        for (int u = blockIdx.x; u < total_units && ok; u = next_unit(u)) {
            Unit w;
            decode(u, w);
            if (w.n == 0)
                continue;
            // q_tma: this unit's query tile by TMA -- per d-half one box of 64
            // elements x G heads x 128 / G tokens, rows in (token, head) order
            // as the row tile numbers them, landing in the 128-byte swizzled
            // K-major layout; rows past the segment read the next rows (or
            // zero past T), whose keys are all masked.  Every S of the unit
            // before has finished: its last value product, issued above,
            // waited for the P of its last S.
            if (p.q_tma && lane == 0) {
                const int tok0 = p.query_start[w.seg] + w.rt * (kTcRows / G);
                mbar_arrive_expect_tx(qtma_bar, L::kHalves * L::kQHalf);
#pragma unroll
                for (int h = 0; h < L::kHalves; ++h)
                    tma_load_3d(qbase + h * L::kQHalf, &tmap_q, qtma_bar, 64 * h, w.kh * G,
                                tok0);
            }
            ok = wait(qfull, nq & 1);  // this unit's queries; O read out by the last unit
            ++nq;
            if (!ok)
                break;
            tc_fence_after();
            for (int si = 0; si < w.n && ok; ++si) {
                const uint32_t gg = g + si, st = gg & 1;
                // S of tile gg into buffer st: its keys landed, and the value
                // product of tile gg - 2 (the buffer's P) is done
                ok = wait(kfull(st), (gg >> 1) & 1);
                if (ok && gg >= kTcStages)
                    ok = wait(vfree(st), ((gg - 2) >> 1) & 1);
                if (!ok)
                    break;
                tc_fence_after();
                const uint64_t dk = desc_k0 + (uint64_t)((st * L::kStageBytes) >> 4);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < KT; ++kk) {
                        const uint32_t qo = ((kk >> 2) * L::kQHalf + (kk & 3) * 32) >> 4;
                        const uint32_t ko = ((kk >> 2) * L::kKVHalf + (kk & 3) * 32) >> 4;
                        tc_mma_ss(tmem + st * kTcTokens, desc_q0 + qo, dk + ko, kIdescS,
                                  kk > 0 ? 1u : 0u);
                    }
                    tc_commit(sfull(st));
                }
                // the previous tile's value product, queued behind this S
                if (si > 0)
                    ok = issue_pv(w, si - 1, gg - 1);
            }
            if (ok)
                ok = issue_pv(w, w.n - 1, g + w.n - 1);
            g += w.n;
        }
        // every tensor-core operation this warp issued has finished
        if (elect_one())
            tc_commit(mma_drain);
        __syncwarp();
        mbar_wait_bounded(mma_drain, 0, kDrainWaitNs);
    }
    pdl_launch_dependents();

    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag)
        flag_error(p.error_word, PA_DEVERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side -------------------------------------------------------------------

template <typename T, int D, bool kFp8, bool kOrdered>
static pa_status launch_mq_as(const MqParams &prm, const CUtensorMap &mk, const CUtensorMap &mv,
                              const CUtensorMap &mq, cudaStream_t stream, long long max_units)
{
    using L = TcLayout<D, kFp8>;
    auto kernel = paged_mq_kernel<T, D, kFp8, kOrdered>;
    static KernelSetting setting[kMaxDevices];
    static std::mutex mu;
    const size_t smem = L::bytes(prm.num_segments, kOrdered);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return record_cuda(e);
    DeviceInfo info;
    const pa_status st = device_info(dev, &info);
    if (st != PA_OK)
        return st;
    if (smem > (size_t)info.optin)
        return PA_ERR_UNSUPPORTED;
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        KernelSetting &ks = setting[dev];
        if (smem > ks.smem_enabled) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
            // the whole unified L1/shared array as shared memory, so that the
            // residency below is the one shared memory allows
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess)
                return record_cuda(e);
            ks.smem_enabled = smem;
        }
        if (smem != ks.smem_queried) {
            // Residency from the kernel's own needs -- shared memory (plus the
            // 1 KB the system reserves per CTA), registers, and tensor memory
            // (kTmemCols of the SM's 512 columns per CTA).  (The runtime's
            // occupancy query answers 1 for this kernel at any shared-memory
            // size, while the launch itself fits two CTAs per SM.)
            cudaFuncAttributes fa;
            int smem_sm = 0, regs_sm = 0;
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e == cudaSuccess)
                e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                           dev);
            if (e == cudaSuccess)
                e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor,
                                           dev);
            if (e != cudaSuccess)
                return record_cuda(e);
            const int by_smem = smem_sm / (int)(smem + 1024);
            const int by_regs = regs_sm / (((fa.numRegs + 7) & ~7) * kTcThreads);
            ks.per_sm = std::min(std::min(by_smem, by_regs), (int)(512 / kTmemCols));
            ks.smem_queried = smem;
        }
        per_sm = ks.per_sm;
    }
    if (per_sm < 1)
        return PA_ERR_UNSUPPORTED;
    long long grid = std::min<long long>((long long)info.sms * per_sm, max_units);
    if (grid < 1)
        grid = 1;
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kTcThreads), smem, stream, prm, mk,
                      mv, mq);
}

// Prefill batches whose units may take more than one round of the grid (two
// CTAs per SM) take the query tiles by TMA (when the query map applies), and
// those of up to kMqOrderSegs sequences the ordered deal.  In a single round
// the order cannot matter and the sort would only add latency, and each
// CTA's one query tile comes sooner from the row warps' own loads than
// through the table lookup and round trip of a TMA issued by the
// tensor-core warp.
template <typename T, int D, bool kFp8>
static pa_status launch_mq(const MqParams &prm_in, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mq, cudaStream_t stream, long long max_units)
{
    MqParams prm = prm_in;
    if (!prm.prefix_mode) {
        int dev = 0;
        const cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return record_cuda(e);
        DeviceInfo info;
        const pa_status st = device_info(dev, &info);
        if (st != PA_OK)
            return st;
        const bool rounds = max_units > 2LL * info.sms;
        if (!rounds)
            prm.q_tma = 0;
        if (rounds && prm.num_segments <= kMqOrderSegs)
            return launch_mq_as<T, D, kFp8, true>(prm, mk, mv, mq, stream, max_units);
    }
    return launch_mq_as<T, D, kFp8, false>(prm, mk, mv, mq, stream, max_units);
}

// Tensor map of a prefill query [T][H][D] (16-bit): boxes of 64 elements x
// group heads x 128 / group tokens, 128-byte swizzle, zero fill past T.
static bool encode_query_map(CUtensorMap *map, const void *query, pa_dtype dtype, int tokens,
                             int heads, int head_dim, int group)
{
    EncodeTiledFn fn = get_encode_fn();
    if (!fn)
        return false;
    const CUtensorMapDataType ty = dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2};
    const cuuint32_t box[3] = {64u, (cuuint32_t)group, (cuuint32_t)(kTcRows / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, ty, 3, const_cast<void *>(query), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// pool_dtype PA_FP8_E4M3: e4m3 pools, query and output of
// query_dtype; otherwise 16-bit pools and query of pool_dtype.
static pa_status dispatch_mq(const MqParams &prm_in, pa_dtype pool_dtype, pa_dtype query_dtype,
                             const void *key_cache, const void *value_cache, int head_dim,
                             cudaStream_t stream, long long max_units)
{
    CUtensorMap mk, mv, mq;
    if (!encode_pool_map(&mk, key_cache, pool_dtype, prm_in.num_blocks, prm_in.block_size,
                         prm_in.num_kv_heads, head_dim) ||
        !encode_pool_map(&mv, value_cache, pool_dtype, prm_in.num_blocks, prm_in.block_size,
                         prm_in.num_kv_heads, head_dim))
        return PA_ERR_CUDA;
    // Prefill with row tiles of whole tokens (the group divides 128) and a
    // 16-byte aligned query: the query tiles may arrive by TMA (launch_mq
    // keeps that for batches of more than one round; over FP8 pools a bf16
    // tile is rounded to fp16 by the row warps once it lands).
    MqParams prm = prm_in;
    std::memset(&mq, 0, sizeof(mq));
    prm.q_tma = 0;
    if (!prm.prefix_mode && prm.group > 0 && kTcRows % prm.group == 0 && prm.num_tokens > 0 &&
        (reinterpret_cast<uintptr_t>(prm.query) & 15) == 0) {
        const pa_dtype qdt = pool_dtype == PA_FP8_E4M3 ? query_dtype : pool_dtype;
        if (!encode_query_map(&mq, prm.query, qdt, prm.num_tokens, prm.num_heads, head_dim,
                              prm.group))
            return PA_ERR_CUDA;
        prm.q_tma = 1;
    }
    using B16 = __nv_bfloat16;
    if (pool_dtype == PA_FP8_E4M3) {
        const bool qbf = query_dtype == PA_BF16;
        if (head_dim == 128)
            return qbf ? launch_mq<B16, 128, true>(prm, mk, mv, mq, stream, max_units)
                       : launch_mq<__half, 128, true>(prm, mk, mv, mq, stream, max_units);
        return qbf ? launch_mq<B16, 64, true>(prm, mk, mv, mq, stream, max_units)
                   : launch_mq<__half, 64, true>(prm, mk, mv, mq, stream, max_units);
    }
    if (head_dim == 128)
        return pool_dtype == PA_BF16
                   ? launch_mq<B16, 128, false>(prm, mk, mv, mq, stream, max_units)
                   : launch_mq<__half, 128, false>(prm, mk, mv, mq, stream, max_units);
    return pool_dtype == PA_BF16 ? launch_mq<B16, 64, false>(prm, mk, mv, mq, stream, max_units)
                                 : launch_mq<__half, 64, false>(prm, mk, mv, mq, stream, max_units);
}

pa_status launch_prefix_pass(const MqParams &prm, pa_dtype dtype, pa_dtype query_dtype,
                             const void *key_cache, const void *value_cache, int head_dim,
                             cudaStream_t stream, long long max_units)
{
    return dispatch_mq(prm, dtype, query_dtype, key_cache, value_cache, head_dim, stream,
                       max_units);
}

}  // namespace pa

using namespace pa;

static pa_status run_prefill(void *out, const void *query, const void *key_cache,
                             const void *value_cache, const int32_t *block_tables,
                             int max_blocks_per_seq, const int32_t *query_start,
                             const int32_t *context_lens, int max_context_len, int num_seqs,
                             int num_tokens, int num_heads, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, float scale, bool fp8,
                             float k_scale, float v_scale, pa_dtype dtype,
                             int32_t *error_word, void *stream)
{
    if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        max_context_len < 0 || !std::isfinite(scale) || !(scale > 0.f) ||
        num_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F16 && dtype != PA_BF16)
        return dtype == PA_FP8_E4M3 && !fp8 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (fp8 && !(std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f &&
                 v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_tokens == 0)
        return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !query_start ||
        !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) ||
        !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) ||
        block_size < kTileTokens || block_size > 256 || (block_size & (block_size - 1)) != 0 ||
        group > 16 || (long long)num_blocks * block_size >= (1ll << 31) ||
        (long long)max_blocks_per_seq * block_size >= (1ll << 31))
        return PA_ERR_UNSUPPORTED;

    MqParams prm{};
    prm.out = out;
    prm.query = query;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.query_start = query_start;
    prm.error_word = error_word;
    prm.wait_ns = stage_wait_limit_ns();
    prm.withhold_fill = withhold_first_fill();
    prm.prefix_mode = 0;
    prm.num_segments = num_seqs;
    prm.num_seqs = num_seqs;
    prm.num_heads = num_heads;
    prm.num_kv_heads = num_kv_heads;
    prm.group = group;
    prm.max_blocks_per_seq = max_blocks_per_seq;
    prm.num_blocks = num_blocks;
    prm.block_size = block_size;
    prm.block_shift = __builtin_ctz((unsigned)block_size);
    prm.max_context_len = max_context_len;
    prm.max_parts = 0;
    prm.part_tokens = 0;
    prm.scale_log2 = scale * (fp8 ? k_scale : 1.f) * kLog2e;
    prm.out_scale = fp8 ? v_scale : 1.f;
    prm.num_tokens = num_tokens;
    // row tiles: at most one partial tile per sequence beyond the full ones
    const long long max_units =
        ((long long)num_tokens * group / kTcRows + num_seqs) * num_kv_heads;
    return dispatch_mq(prm, fp8 ? PA_FP8_E4M3 : dtype, dtype, key_cache, value_cache, head_dim,
                       as_stream(stream), max_units);
}

extern "C" pa_status pa_prefill_attention(void *out, const void *query, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          int max_blocks_per_seq, const int32_t *query_start,
                                          const int32_t *context_lens, int max_context_len,
                                          int num_seqs, int num_tokens, int num_heads,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float scale, pa_dtype dtype,
                                          int32_t *error_word, void *stream)
{
    return run_prefill(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                       query_start, context_lens, max_context_len, num_seqs, num_tokens,
                       num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, false,
                       1.f, 1.f, dtype, error_word, stream);
}

extern "C" pa_status pa_prefill_attention_fp8(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *query_start,
    const int32_t *context_lens, int max_context_len, int num_seqs, int num_tokens,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    float k_scale, float v_scale, pa_dtype dtype, int32_t *error_word, void *stream)
{
    return run_prefill(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                       query_start, context_lens, max_context_len, num_seqs, num_tokens,
                       num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, true,
                       k_scale, v_scale, dtype, error_word, stream);
}
