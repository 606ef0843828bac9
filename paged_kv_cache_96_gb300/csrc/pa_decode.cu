// pa_decode.cu -- paged decode attention for sm_103a.
//
// What it computes ("PagedAttention & Continuous Batching", §1.6 and §2.4):
// for every running sequence s and query head h, the softmax-weighted sum of
// the value vectors of the sequence's cached tokens, where token p's K and V
// live in physical block block_tables[s][p / block_size], row
// p % block_size of the token-major pools [num_blocks][block_size]
// [num_kv_heads][head_dim].  Query heads are grouped over KV heads
// (kh = h / G), so one KV head serves G query heads.
//
// How (GB300 design):
//  * Work unit = (sequence, KV head, partition of `part_tokens` tokens).  A
//    persistent grid (as many CTAs as fit on every SM) walks the units
//    round-robin; units are numbered KV-head-fastest so the CTAs working on
//    the Hkv heads of one partition run side by side and together stream
//    whole token rows of the pool.
//  * Each warp owns a ring of NST shared-memory stages.  A stage holds one
//    16-token tile of K and of V for one KV head, fetched from the pool by
//    4-D tiled TMA loads (128-byte swizzle) that complete on the stage's
//    mbarrier.  The warp consumes tile i and immediately refills the stage
//    with its tile i + NST, crossing into the next unit when the current
//    one runs out, so the loads in flight never drain at unit boundaries.
//  * The G query heads of a KV head form the N dimension of tensor-core
//    tiles: S^T-tile [16 tokens x 8 heads] = K[16 x d] . Q^T[d x 8] and
//    O^T[d x 8] += V^T[d x 16] . P^T[16 x 8] with mma.sync m16n8k16 (fp32
//    accumulate); P goes from the S accumulator layout to the B-operand
//    layout with movmatrix.  Every K/V byte is read from HBM once per step.
//  * Softmax is online in fp32 (a reference max, running sum, exp2 with the
//    scale folded into log2 units).  At the end of a unit the tile warps
//    hand their (m, l, O) to the CTA's merge warp through shared memory (two
//    named barriers, no CTA-wide sync), which combines them and writes the
//    output row or the unit's partial.
//  * Split context: a unit that is one of several partitions of its
//    sequence writes a partial (m, l, o) to the workspace and arrives on the
//    sequence's counter; the arrival that completes a sequence of up to 8
//    partials merges them by log-sum-exp weights in the same pass, and the
//    reduce kernel queued behind this one merges longer sequences.
//  * Bounds: table entries outside [0, num_blocks) are never fetched (the
//    tile is skipped, an error bit is set); tokens past the context are
//    masked in the scores and their value rows are zeroed before the
//    contraction, so poisoned (NaN) slots never reach the output.  Every
//    wait on a stage is bounded in time.
#include <cuda.h>

#include <type_traits>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "pa_decode_common.cuh"
#include "pa_prefill.cuh"

namespace pa {

// FP8 pools: units are numbered sequence by sequence, the sequences with
// the most partitions first (by index within a count; counts from
// kOrderBuckets - 1 up share the first place), so that the static deal's
// last round -- run while most CTAs have finished -- holds the short
// sequences' units (the FP8 pass is bound by its instructions per tile, so
// the CTAs left at the end cannot take up the bandwidth the others free).
// 16-bit pools, and batches of more than kOrderSeqs sequences, keep the
// sequences' own order.
constexpr int kOrderBuckets = 64;
constexpr int kOrderSeqs = 512;

// Shared-memory layout (offsets from a 1024-byte aligned base): NW warps,
// each with a private ring of NST stages.  EB = bytes per cached element
// (2 for fp16/bf16 pools, 1 for FP8 pools).
template <int D, int NT, int NW, int NST, int EB> struct Layout {
    static constexpr int kHalfBytes = kTileTokens * 128;      // 16 rows x 64 elements (EB 2)
    static constexpr int kTileBytes = kTileTokens * D * EB;   // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;        // K tile + V tile
    static constexpr int kHeads = 8 * NT;
    static constexpr int kPitch = D + 4;  // floats per merge row (bank spread)
    static constexpr int kStages = 0;
    static constexpr int kMergeO = kStages + NW * NST * kStageBytes;
    static constexpr int kMergeM = kMergeO + NW * kHeads * kPitch * 4;
    static constexpr int kMergeL = kMergeM + NW * kHeads * 4;
    // fused append: the new token's value row (fp32) and per-head scores,
    // one buffer per parity of the CTA's unit count
    static constexpr int kAppV = kMergeL + NW * kHeads * 4;
    static constexpr int kAppM = kAppV + 2 * D * 4;
    static constexpr int kBars = kAppM + 2 * kHeads * 4;  // NW * NST stage barriers
    static constexpr int kFlags = kBars + NW * NST * 8;
    static constexpr bool kOrdered = EB == 1;  // FP8 pools: the unit order below
    static constexpr int kHist = kFlags + NW * NST * 4;  // the unit order's buckets
    // int ctx[S], prefix[S + 1], start[S], then (ordered) order[S]
    static constexpr int kSeq = kHist + (kOrdered ? kOrderBuckets * 4 : 0);
    static size_t bytes(int num_seqs)
    {
        const size_t per_seq = kOrdered && num_seqs <= kOrderSeqs ? 4 : 3;
        return 1024 + kSeq + 4 * (per_seq * (size_t)num_seqs + 1);
    }
    static_assert(kBars % 8 == 0, "mbarriers need 8-byte alignment");
    static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

// T: query/output type.  KV: cached element type -- T itself, or uint8_t
// for FP8 (e4m3) pools, whose tiles are widened to fp16 in registers (the
// tensor-core products then run in fp16).
// Fused append, one warp, once per (sequence s, KV head kh) at the start of
// the sequence's last unit: the new token at position pos goes to its pool
// slot (the 16-bit row verbatim, or its e4m3 codes computed as
// reshape_and_cache_fp8 computes them) and its merge record is staged --
// app_v = the value row as attention sees it (the codes, widened, for FP8
// pools: the V scale is applied with the output), app_m[jh] = the score of
// query head kh * G + jh in log2 units.  The tiles of the unit stop before
// pos, so the record enters the softmax exactly once, in the end-of-unit
// merge.  Each lane holds D / 32 consecutive elements; every load is issued
// before the first use (one round trip).  NH: query heads the kernel
// instance serves per KV head (>= the group).
template <typename T, bool kFp8, int D, int NH>
__device__ __noinline__ void append_token(const DecodeParams &p, int s, int kh, int pos,
                                          float *app_v, float *app_m, int lane)
{
    constexpr int E = D / 32;
    using Raw = typename std::conditional<E == 4, uint2, uint32_t>::type;
    auto f = [](T x) -> float {
        if constexpr (std::is_same<T, __half>::value)
            return __half2float(x);
        else
            return __bfloat162float(x);
    };
    const int G = p.group;
    const size_t row = ((size_t)s * p.num_kv_heads + kh) * D + (size_t)lane * E;
    const Raw kr = __ldg(reinterpret_cast<const Raw *>(static_cast<const T *>(p.new_key) + row));
    const Raw vr = __ldg(reinterpret_cast<const Raw *>(static_cast<const T *>(p.new_value) + row));
    const int32_t ent =
        __ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + (pos >> p.block_shift));
    Raw qr[NH];
    const T *q0 = static_cast<const T *>(p.query) +
                  ((size_t)s * p.num_heads + (size_t)kh * G) * D + (size_t)lane * E;
#pragma unroll
    for (int jh = 0; jh < NH; ++jh)
        qr[jh] = jh < G ? __ldg(reinterpret_cast<const Raw *>(q0 + (size_t)jh * D)) : Raw{};
    const T *ke = reinterpret_cast<const T *>(&kr);
    const T *ve = reinterpret_cast<const T *>(&vr);
    float kf[E], vf[E];
    const bool ok = ent >= 0 && ent < p.num_blocks;
    const int64_t slot = ok ? (int64_t)ent * p.block_size + (pos & (p.block_size - 1)) : -1;
    const size_t elem = ((size_t)slot * p.num_kv_heads + kh) * D + (size_t)lane * E;
    if constexpr (kFp8) {
        // the e4m3 codes of this lane's E elements, as reshape_and_cache_fp8
        // computes them, stored E bytes at a time
        uint32_t kc = 0, vc = 0;
#pragma unroll
        for (int h = 0; h < E / 2; ++h) {
            kc |= (uint32_t)f32x2_to_e4m3x2(f(ke[2 * h]) * p.k_inv_scale,
                                            f(ke[2 * h + 1]) * p.k_inv_scale) << (16 * h);
            vc |= (uint32_t)f32x2_to_e4m3x2(f(ve[2 * h]) * p.v_inv_scale,
                                            f(ve[2 * h + 1]) * p.v_inv_scale) << (16 * h);
        }
        if (ok) {
            uint8_t *kd = static_cast<uint8_t *>(p.key_cache) + elem;
            uint8_t *vd = static_cast<uint8_t *>(p.value_cache) + elem;
            if constexpr (E == 4) {
                *reinterpret_cast<uint32_t *>(kd) = kc;
                *reinterpret_cast<uint32_t *>(vd) = vc;
            } else {
                *reinterpret_cast<uint16_t *>(kd) = (uint16_t)kc;
                *reinterpret_cast<uint16_t *>(vd) = (uint16_t)vc;
            }
        }
#pragma unroll
        for (int h = 0; h < E / 2; ++h) {
            const uint32_t kw = e4m3x2_to_f16x2((uint16_t)(kc >> (16 * h)));
            const uint32_t vw = e4m3x2_to_f16x2((uint16_t)(vc >> (16 * h)));
            kf[2 * h] = __half2float(__ushort_as_half((unsigned short)(kw & 0xffffu)));
            kf[2 * h + 1] = __half2float(__ushort_as_half((unsigned short)(kw >> 16)));
            vf[2 * h] = __half2float(__ushort_as_half((unsigned short)(vw & 0xffffu)));
            vf[2 * h + 1] = __half2float(__ushort_as_half((unsigned short)(vw >> 16)));
        }
    } else {
        if (ok) {
            *reinterpret_cast<Raw *>(static_cast<T *>(p.key_cache) + elem) = kr;
            *reinterpret_cast<Raw *>(static_cast<T *>(p.value_cache) + elem) = vr;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            kf[e] = f(ke[e]);
            vf[e] = f(ve[e]);
        }
    }
    if (lane == 0) {
        if (!ok)
            flag_error(p.error_word, PA_DEVERR_BLOCK_RANGE);
        if (kh == 0 && p.slot_out != nullptr)
            p.slot_out[s] = (int32_t)slot;
    }
#pragma unroll
    for (int e = 0; e < E; ++e)
        app_v[lane * E + e] = vf[e];
#pragma unroll
    for (int jh = 0; jh < NH; ++jh) {
        if (jh >= G)
            break;
        const T *qe = reinterpret_cast<const T *>(&qr[jh]);
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            // FP8 pools take the query in fp16, as the tiles' products do
            const float q = kFp8 ? __half2float(__float2half_rn(f(qe[e]))) : f(qe[e]);
            dot = fmaf(q, kf[e], dot);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            dot += __shfl_xor_sync(kFull, dot, off);
        if (lane == 0)
            app_m[jh] = dot * p.scale_log2;
    }
}

// Register budget for MINB resident CTAs of NW warps: an SM's 64K registers
// sit in four 16K sub-partition files and each warp lives in one of them, so
// the binding limit is the fullest file (ceil(NW * MINB / 4) warps).  The
// thread count given to __launch_bounds__ is the one whose even split over
// MINB CTAs yields that per-warp budget, in whole warps (the compiler rounds
// a partial warp up, which would shrink the budget); the block itself is NW
// warps.
constexpr int bound_threads(int NW, int MINB)
{
    return 128 * ((NW * MINB + 3) / 4) / MINB / 32 * 32;
}

template <typename T, typename KV, int D, int NT, int NW, int NST, int MINB>
__global__ void __launch_bounds__(bound_threads(NW + 1, MINB), MINB)
    paged_decode_kernel(const __grid_constant__ DecodeParams p,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v)
{
    constexpr bool kFp8 = sizeof(KV) == 1;
    using L = Layout<D, NT, NW, NST, sizeof(KV)>;
    using MT = typename std::conditional<kFp8, __half, T>::type;  // tensor-core input type
    using Op = MmaOp<MT>;
    constexpr int KT = D / 16;  // k-steps of the score product, m-tiles of the output
    constexpr int kHeads = L::kHeads;
    constexpr int kThreads = (NW + 1) * 32;  // NW tile warps, then the merge warp
    static_assert(bound_threads(NW + 1, MINB) >= kThreads, "launch bound below the block size");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int g = lane >> 2;  // mma group (row of the accumulator fragment)
    const int t4 = lane & 3;  // thread in group (column pair)

    const int S = p.num_seqs;
    const int Hkv = p.num_kv_heads;
    const int G = p.group;
    const int P = p.part_tokens;
    // Fused append: each sequence's last position holds the new token, whose
    // K/V come from new_key/new_value; the tiles cover the positions before it.
    const int napp = p.new_key != nullptr ? 1 : 0;

    int *ctx_s = reinterpret_cast<int *>(smem + L::kSeq);
    int *pref = ctx_s + S;  // over the unit order: pref[k] = partitions of order[0 .. k)
    int *start_s = pref + S + 1;
    const bool ordered = L::kOrdered && S <= kOrderSeqs;
    int *order = start_s + S;  // k-th sequence of the unit order (when ordered)
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L::kFlags);
    float *merge_o = reinterpret_cast<float *>(smem + L::kMergeO);
    float *merge_m = reinterpret_cast<float *>(smem + L::kMergeM);
    float *merge_l = reinterpret_cast<float *>(smem + L::kMergeL);
    float *app_v = reinterpret_cast<float *>(smem + L::kAppV);
    float *app_m = reinterpret_cast<float *>(smem + L::kAppM);
    auto bar_of = [&](int stage) { return sbase + L::kBars + (warp * NST + stage) * 8; };
    auto stage_of = [&](int stage) {
        return sbase + L::kStages + (warp * NST + stage) * L::kStageBytes;
    };
    if (lane == 0 && warp < NW) {
        for (int k = 0; k < NST; ++k)
            mbar_init(bar_of(k), 1);
        fence_barrier_init();
    }
    if (tid == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    // Launched as a programmatic dependent of the kernel before it on the
    // stream: every global read below comes after the predecessor's writes
    // are visible.  Alongside the shared-prefix pass (which starts this one
    // only once everything before it has finished, and writes only partial
    // slots this pass leaves alone) the wait moves to the end, so that this
    // grid -- and the reduce after it -- finishes after that pass.
    if (!p.concurrent)
        pdl_wait_primary();

    // ---- context lengths and partition prefix sums -----------------------
    for (int s = tid; s < S; s += kThreads) {
        const int c = clamp_context(p, s, blockIdx.x == 0);
        ctx_s[s] = c;
        start_s[s] = seq_start_of(p, s, c);
        // with the append fused in, a shared prefix must end before the new
        // token (which is then in a block of the sequence's own)
        if (napp != 0 && c > 0 && start_s[s] >= c && blockIdx.x == 0)
            flag_error(p.error_word, PA_DEVERR_PREFIX_PLAN);
    }
    __syncthreads();
    if (warp == 0) {
        if (ordered) {
            // counting sort by partitions, most first, by index within a count;
            // every CTA computes the same order
            int *hist = reinterpret_cast<int *>(smem + L::kHist);
            auto key_of = [&](int sq) {
                return kOrderBuckets - 1 -
                       min(own_partitions(ctx_s[sq], start_s[sq], P), kOrderBuckets - 1);
            };
            hist[lane] = 0;
            hist[lane + 32] = 0;
            __syncwarp();
            for (int sq = lane; sq < S; sq += 32)
                atomicAdd(&hist[key_of(sq)], 1);
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
            for (int base = 0; base < S; base += 32) {
                const int sq = base + lane;
                const int key = sq < S ? key_of(sq) : -1;
                const unsigned same = __match_any_sync(kFull, key);
                const int rank = __popc(same & ((1u << lane) - 1u));
                const int off = key >= 0 ? hist[key] : 0;
                __syncwarp();
                if (key >= 0) {
                    order[off + rank] = sq;
                    if (rank == 0)
                        hist[key] = off + __popc(same);
                }
                __syncwarp();
            }
        }
        int carry = 0;
        for (int base = 0; base < S; base += 32) {
            const int k = base + lane;
            const int sq = k < S ? (ordered ? order[k] : k) : 0;
            const int n = k < S ? own_partitions(ctx_s[sq], start_s[sq], P) : 0;
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, x, o);
                if (lane >= o)
                    x += y;
            }
            if (k < S)
                pref[k] = carry + x - n;
            carry += __shfl_sync(kFull, x, 31);
        }
        if (lane == 0)
            pref[S] = carry;
    }
    __syncthreads();
    const int total_units = pref[S] * Hkv;

    // ---- sequences with no context get zero rows ----------------------------
    for (int s = blockIdx.x; s < S; s += gridDim.x) {
        if (ctx_s[s] != 0)
            continue;
        if (tid == 0 && p.new_key != nullptr && p.slot_out != nullptr)
            p.slot_out[s] = -1;  // nothing to append
        uint4 *row = reinterpret_cast<uint4 *>(static_cast<T *>(p.out) +
                                               (size_t)s * p.num_heads * D);
        for (int i = tid; i < p.num_heads * D / 8; i += kThreads)
            row[i] = make_uint4(0, 0, 0, 0);
    }

    // unit u -> partition q = u / Hkv, kv head u % Hkv; sequence s is the
    // k-th of the unit order, k the one with pref[k] <= q < pref[k + 1].
    auto decode_unit = [&](int u, int &s, int &kh, int &j, int &tok0, int &ntiles) {
        const int q = u / Hkv;
        kh = u - q * Hkv;
        int lo = 0, hi = S - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pref[mid] <= q)
                lo = mid;
            else
                hi = mid - 1;
        }
        j = q - pref[lo];
        s = ordered ? order[lo] : lo;
        tok0 = start_s[s] + j * P;
        const int tok_end = min(ctx_s[s] - napp, tok0 + P);
        ntiles = (tok_end - tok0 + kTileTokens - 1) / kTileTokens;
    };

    // this CTA's units: the first, and the one after unit u
    const int early_units = p.early_rounds * p.early_ctas;
    const int u_first = (int)blockIdx.x < p.early_ctas ? (int)blockIdx.x
                                                        : early_units + (int)blockIdx.x;
    auto next_u = [&](int u) -> int {
        return u < early_units ? u + p.early_ctas : u + (int)gridDim.x;
    };
    // ---- this warp's fetch cursor: its next tile, possibly in a later unit ----
    int pu = u_first, ps = 0, pkh = 0, pj = 0, ptok0 = 0, pnt = 0, ptile = warp;
    bool pdone = pu >= total_units || warp >= NW;  // the merge warp fetches nothing
    if (!pdone)
        decode_unit(pu, ps, pkh, pj, ptok0, pnt);
    auto skip_empty = [&]() {
        while (!pdone && ptile >= pnt) {
            pu = next_u(pu);
            if (pu >= total_units) {
                pdone = true;
                break;
            }
            decode_unit(pu, ps, pkh, pj, ptok0, pnt);
            ptile = warp;
        }
    };
    skip_empty();
    // Lane 0 loads the table entry of the tile at the cursor one tile ahead
    // of issuing its fetch, so the load's latency overlaps a tile of compute.
    int pphys = 0, prow = 0;
    auto prefetch_entry = [&]() {
        if (!pdone && lane == 0) {
            const int tok = ptok0 + ptile * kTileTokens;
            prow = tok & (p.block_size - 1);
            pphys = __ldg(p.block_tables + (size_t)ps * p.max_blocks_per_seq +
                          (tok >> p.block_shift));
        }
    };
    prefetch_entry();

    uint32_t issued = 0, consumed = 0;
    uint32_t inflight = 0;  // stages with a fetch not yet waited for
    bool aborted = false;
    auto produce = [&]() {
        if (pdone || aborted)
            return;
        const int stage = issued % NST;
        // test hook of the time-out path: a fill that is never issued, so
        // nothing completes the stage's phase and its wait runs out
        const bool withheld = p.withhold_fill != 0 && warp == 0 && issued == 0;
        if (lane == 0 && !withheld) {
            const bool ok = pphys >= 0 && pphys < p.num_blocks;
            flags[warp * NST + stage] = ok;
            if (ok) {
                const uint32_t dst = stage_of(stage);
                mbar_arrive_expect_tx(bar_of(stage), L::kStageBytes);
                if constexpr (kFp8) {
                    // one 128-byte row per token: a 2 KB box per tile and tensor
                    tma_load_4d(dst, &tmap_k, bar_of(stage), 0, pkh, prow, pphys);
                    tma_load_4d(dst + L::kTileBytes, &tmap_v, bar_of(stage), 0, pkh, prow,
                                pphys);
                } else {
#pragma unroll
                    for (int hf = 0; hf < D / 64; ++hf) {
                        tma_load_4d(dst + hf * L::kHalfBytes, &tmap_k, bar_of(stage), hf * 64,
                                    pkh, prow, pphys);
                        tma_load_4d(dst + L::kTileBytes + hf * L::kHalfBytes, &tmap_v,
                                    bar_of(stage), hf * 64, pkh, prow, pphys);
                    }
                }
            } else {
                flag_error(p.error_word, PA_DEVERR_BLOCK_RANGE);
                mbar_arrive(bar_of(stage));
            }
        }
        if (!withheld)
            inflight |= 1u << stage;
        ++issued;
        ptile += NW;
        skip_empty();
        prefetch_entry();
    };
    for (int k = 0; k < NST; ++k)
        produce();

    // Per-lane ldmatrix row/chunk selectors.
    const int li = lane & 7, lj = lane >> 3;
    const int k_row = li + ((lj & 1) << 3), k_cj = lj >> 1;  // K: A operand
    const int v_row = li + ((lj >> 1) << 3), v_cj = lj & 1;  // V^T: A operand (trans)
    // Shared-memory address of 16-byte chunk `chunk` of (token, d-half) in a
    // tile at `base`: rows of 128 bytes; chunk c of row r sits at chunk
    // c ^ (r & 7) (the TMA's 128-byte swizzle).
    auto tile_addr = [&](uint32_t base, int token, int half, int chunk) -> uint32_t {
        if constexpr (kFp8) {
            const int r = token;
            if constexpr (D == 64)  // one 64-byte row per token, chunk 0..3, 64-byte swizzle
                return base + r * 64 + ((chunk ^ ((r >> 1) & 3)) << 4);
            // one 128-byte row per token, chunk 0..7
            return base + r * 128 + (((chunk + 4 * half) ^ (r & 7)) << 4);
        }
        const int r = half * kTileTokens + token;
        return base + r * 128 + ((chunk ^ (r & 7)) << 4);
    };

    // Query fragments (B operand of the score product): head 8nt+g of the
    // group.  16-bit pools: elements d = 16kk + 2t4 (+1) and +8 (+9).  FP8
    // pools: the score's sum over d is taken in a permuted order matching the
    // FP8 tile fragments -- k-steps 2t4, 2t4+1 <- d = 16kk + 4t4 (+1) and
    // k-steps 2t4+8, 2t4+9 <- d = 16kk + 4t4 + 2 (+3) -- in fp16.
    uint32_t qf[NT][KT][2];
    bool q_over = false;  // FP8 pools: a bf16 query element past the fp16 range
    auto load_query = [&](int s, int kh) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hg = nt * 8 + g;
            const T *qrow = static_cast<const T *>(p.query) +
                            ((size_t)s * p.num_heads + (size_t)kh * G + (hg < G ? hg : 0)) * D;
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                if constexpr (kFp8) {
                    uint2 w = make_uint2(0u, 0u);
                    if (hg < G)
                        w = __ldg(reinterpret_cast<const uint2 *>(qrow + kk * 16 + 4 * t4));
                    if constexpr (std::is_same<T, __half>::value) {
                        qf[nt][kk][0] = w.x;
                        qf[nt][kk][1] = w.y;
                    } else {
                        const T *e = reinterpret_cast<const T *>(&w);
                        const float x0 = __bfloat162float(e[0]), x1 = __bfloat162float(e[1]);
                        const float x2 = __bfloat162float(e[2]), x3 = __bfloat162float(e[3]);
                        // the fp16 products need |q| within the fp16 range
                        q_over |= fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))) >
                                  65504.f;
                        qf[nt][kk][0] = pack_f16x2(x0, x1);
                        qf[nt][kk][1] = pack_f16x2(x2, x3);
                    }
                } else {
                    const uint32_t *qw = reinterpret_cast<const uint32_t *>(qrow);
                    qf[nt][kk][0] = hg < G ? __ldg(qw + kk * 8 + t4) : 0u;
                    qf[nt][kk][1] = hg < G ? __ldg(qw + kk * 8 + 4 + t4) : 0u;
                }
            }
        }
    };
    if (u_first < total_units && warp < NW) {
        int s, kh, j, tok0, ntiles;
        decode_unit(u_first, s, kh, j, tok0, ntiles);
        load_query(s, kh);
    }

    // ---- units --------------------------------------------------------------------
    // The tile warps stream a unit's tiles and hand their (m, l, O) to the
    // merge warp through shared memory; the merge warp combines them (and the
    // appended token's record), writes the output row or the partition's
    // partial, and -- for split sequences -- arrives on the sequence's counter
    // and merges the partials when its arrival completes them.  The two sides
    // meet only at two named barriers per unit ("records written": the tile
    // warps arrive, the merge warp waits; "records read": the other way
    // round, skipped after the CTA's last unit), so tile warps never wait for
    // each other at a unit's end and the merge warp sleeps in hardware.
    constexpr int kRecFull = 1, kRecFree = 2;  // named barrier ids (0 is __syncthreads)
    if (warp < NW) {
        int k_unit = 0;          // units of this CTA so far
        bool rec_aborted = false;
        for (int u = u_first; u < total_units; u = next_u(u), ++k_unit) {
            int s, kh, j, tok0, ntiles;
            decode_unit(u, s, kh, j, tok0, ntiles);
            const int tok_end = min(ctx_s[s] - napp, tok0 + P);
            // fused append: the sequence's last unit also takes the new token
            const bool app = napp != 0 && tok0 + P >= ctx_s[s];

            float o[KT][NT][4];
            float mrun[NT][2], lrun[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mrun[nt][0] = mrun[nt][1] = -INFINITY;
                lrun[nt][0] = lrun[nt][1] = 0.f;
#pragma unroll
                for (int mt = 0; mt < KT; ++mt)
                    o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
            }
            // the new token counts as tile ntiles of the round-robin deal: its
            // warp is one with a tile fewer than the others (or the first)
            if (app && warp == ntiles % NW)
                append_token<T, kFp8, D, kHeads>(p, s, kh, ctx_s[s] - 1, app_v + (k_unit & 1) * D,
                                                 app_m + (k_unit & 1) * kHeads, lane);

            for (int tile = warp; tile < ntiles; tile += NW) {
                const int stage = consumed % NST;
                const uint32_t parity = (consumed / NST) & 1u;
                bool ready = false;
                if (!aborted) {
                    ready = __all_sync(kFull, mbar_wait_bounded(bar_of(stage), parity, p.wait_ns));
                    if (ready) {
                        inflight &= ~(1u << stage);
                    } else {
                        aborted = true;
                        if (lane == 0)
                            flag_error(p.error_word, PA_DEVERR_TIMEOUT);
                    }
                }
                if (ready && flags[warp * NST + stage] != 0) {
                    const uint32_t kbase = stage_of(stage);
                    const uint32_t vbase = kbase + L::kTileBytes;
                    const int nv = tok_end - (tok0 + tile * kTileTokens);  // valid rows
                    const bool partial = nv < kTileTokens;

                    // scores S[token][head] = K . Q^T in independent accumulator
                    // chains (k-step kk feeds chain kk % kChains), summed at the end
                    constexpr int kChains = KT >= 4 ? 4 : KT;
                    float part[kChains][NT][4];
#pragma unroll
                    for (int c = 0; c < kChains; ++c)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            part[c][nt][0] = part[c][nt][1] = part[c][nt][2] = part[c][nt][3] = 0.f;
                    if constexpr (kFp8) {
                        // one ldmatrix brings two 16-d chunks of 16 tokens as byte
                        // pairs: thread (g, t4) gets d = 16c + 4t4 .. +3 of tokens g
                        // and g + 8; widening gives the (permuted-k) A fragment
#pragma unroll
                        for (int kp = 0; kp < KT / 2; ++kp) {
                            uint32_t r[4];
                            ldmatrix_x4(tile_addr(kbase, k_row, 0, 2 * kp + k_cj), r);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int kk = 2 * kp + h;
                                const uint32_t w0 = r[2 * h], w1 = r[2 * h + 1];
                                uint32_t a[4];
                                a[0] = e4m3x2_to_f16x2((uint16_t)(w0 & 0xffffu));
                                a[1] = e4m3x2_to_f16x2((uint16_t)(w1 & 0xffffu));
                                a[2] = e4m3x2_to_f16x2((uint16_t)(w0 >> 16));
                                a[3] = e4m3x2_to_f16x2((uint16_t)(w1 >> 16));
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    Op::run(part[kk % kChains][nt], a, qf[nt][kk][0], qf[nt][kk][1]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < KT; ++kk) {
                            uint32_t a[4];
                            ldmatrix_x4(tile_addr(kbase, k_row, kk >> 2, (kk & 3) * 2 + k_cj), a);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                Op::run(part[kk % kChains][nt], a, qf[nt][kk][0], qf[nt][kk][1]);
                        }
                    }
                    float sc[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float x = part[0][nt][e];
#pragma unroll
                            for (int c = 1; c < kChains; ++c)
                                x += part[c][nt][e];
                            sc[nt][e] = x;
                        }

                    // V^T fragments (their latency overlaps the softmax); rows past
                    // the context are zeroed so NaN padding never meets a zero weight
                    uint32_t va[KT][4];
                    if constexpr (kFp8) {
                        // transposed byte-pair loads: thread (g, t4) gets tokens 2t4,
                        // 2t4+1 (and +8, +9) at d = 16c + 2g, 2g+1; fragment row g is
                        // d = 16c + 2g and row g + 8 is d = 16c + 2g + 1
#pragma unroll
                        for (int mp = 0; mp < KT / 2; ++mp) {
                            uint32_t r[4];
                            ldmatrix_x4_trans(tile_addr(vbase, k_row, 0, 2 * mp + k_cj), r);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint32_t p0 = byte_perm(r[2 * h], 0u, 0x3120u);
                                const uint32_t p1 = byte_perm(r[2 * h + 1], 0u, 0x3120u);
                                va[2 * mp + h][0] = e4m3x2_to_f16x2((uint16_t)(p0 & 0xffffu));
                                va[2 * mp + h][1] = e4m3x2_to_f16x2((uint16_t)(p0 >> 16));
                                va[2 * mp + h][2] = e4m3x2_to_f16x2((uint16_t)(p1 & 0xffffu));
                                va[2 * mp + h][3] = e4m3x2_to_f16x2((uint16_t)(p1 >> 16));
                            }
                        }
                    } else {
#pragma unroll
                        for (int mt = 0; mt < KT; ++mt)
                            ldmatrix_x4_trans(tile_addr(vbase, v_row, mt >> 2, (mt & 3) * 2 + v_cj),
                                              va[mt]);
                    }
                    if (partial) {
                        const uint32_t m01 = (2 * t4 < nv ? 0x0000ffffu : 0u) |
                                             (2 * t4 + 1 < nv ? 0xffff0000u : 0u);
                        const uint32_t m89 = (2 * t4 + 8 < nv ? 0x0000ffffu : 0u) |
                                             (2 * t4 + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
                        for (int mt = 0; mt < KT; ++mt) {
                            va[mt][0] &= m01;
                            va[mt][1] &= m01;
                            va[mt][2] &= m89;
                            va[mt][3] &= m89;
                        }
                    }

                    // online softmax; P^T fragments for the value product
                    uint32_t pb[NT][2];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float s0 = sc[nt][0] * p.scale_log2, s1 = sc[nt][1] * p.scale_log2;
                        float s2 = sc[nt][2] * p.scale_log2, s3 = sc[nt][3] * p.scale_log2;
                        if (partial) {
                            if (g >= nv)
                                s0 = s1 = -INFINITY;
                            if (g + 8 >= nv)
                                s2 = s3 = -INFINITY;
                        }
                        // mrun is a reference point, not necessarily the running max:
                        // while every score of the tile stays within kSlack of it
                        // (weights <= 2^kSlack) it is kept, which skips the
                        // cross-lane max and the rescale; otherwise it moves up to
                        // the running max and l and O are rescaled.
                        const bool fits = s0 <= mrun[nt][0] + kSlack && s2 <= mrun[nt][0] + kSlack &&
                                          s1 <= mrun[nt][1] + kSlack && s3 <= mrun[nt][1] + kSlack;
                        if (!__all_sync(kFull, fits)) {
                            float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
                            for (int off = 4; off < 32; off <<= 1) {
                                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
                                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
                            }
                            const float mn0 = fmaxf(mrun[nt][0], mx0);
                            const float mn1 = fmaxf(mrun[nt][1], mx1);
                            const float al0 = mn0 == -INFINITY ? 1.f : exp2f(mrun[nt][0] - mn0);
                            const float al1 = mn1 == -INFINITY ? 1.f : exp2f(mrun[nt][1] - mn1);
                            lrun[nt][0] *= al0;
                            lrun[nt][1] *= al1;
#pragma unroll
                            for (int mt = 0; mt < KT; ++mt) {
                                o[mt][nt][0] *= al0;
                                o[mt][nt][1] *= al1;
                                o[mt][nt][2] *= al0;
                                o[mt][nt][3] *= al1;
                            }
                            mrun[nt][0] = mn0;
                            mrun[nt][1] = mn1;
                        }
                        const float mu0 = mrun[nt][0] == -INFINITY ? 0.f : mrun[nt][0];
                        const float mu1 = mrun[nt][1] == -INFINITY ? 0.f : mrun[nt][1];
                        const float p0 = exp2f(s0 - mu0), p2 = exp2f(s2 - mu0);
                        const float p1 = exp2f(s1 - mu1), p3 = exp2f(s3 - mu1);
                        lrun[nt][0] += p0 + p2;
                        lrun[nt][1] += p1 + p3;
                        pb[nt][0] = movmatrix_trans(Op::pack(p0, p1));
                        pb[nt][1] = movmatrix_trans(Op::pack(p2, p3));
                    }

                    // O^T[d][head] += V^T . P^T
#pragma unroll
                    for (int mt = 0; mt < KT; ++mt)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            Op::run(o[mt][nt], va[mt], pb[nt][0], pb[nt][1]);
                }
                __syncwarp();
                ++consumed;
                produce();  // refill the stage just consumed
            }

            // Next unit's query: its loads land while this unit's records go out.
            if (next_u(u) < total_units) {
                int sn, khn, jn, tn, ntn;
                decode_unit(next_u(u), sn, khn, jn, tn, ntn);
                load_query(sn, khn);
            }

            // ---- end of unit: this warp's (m, l, O) to the merge warp -------------------
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int k = 0; k < 2; ++k)
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1)
                        lrun[nt][k] += __shfl_xor_sync(kFull, lrun[nt][k], off);
            // the merge warp has read the previous unit's records
            if (k_unit > 0)
                named_barrier_sync(kRecFree, kThreads);
            {
                float *mo = merge_o + warp * kHeads * L::kPitch;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int h0 = nt * 8 + 2 * t4;
#pragma unroll
                    for (int mt = 0; mt < KT; ++mt) {
                        // fragment rows g, g + 8 are d = 16mt + g, + 8 (16-bit pools)
                        // or d = 16mt + 2g, + 1 (FP8 pools)
                        const int d0 = kFp8 ? mt * 16 + 2 * g : mt * 16 + g;
                        const int d1 = kFp8 ? d0 + 1 : d0 + 8;
                        mo[h0 * L::kPitch + d0] = o[mt][nt][0];
                        mo[(h0 + 1) * L::kPitch + d0] = o[mt][nt][1];
                        mo[h0 * L::kPitch + d1] = o[mt][nt][2];
                        mo[(h0 + 1) * L::kPitch + d1] = o[mt][nt][3];
                    }
                    if (g == 0) {
                        merge_m[warp * kHeads + h0] = mrun[nt][0];
                        merge_m[warp * kHeads + h0 + 1] = mrun[nt][1];
                        merge_l[warp * kHeads + h0] = lrun[nt][0];
                        merge_l[warp * kHeads + h0 + 1] = lrun[nt][1];
                    }
                }
            }
            named_barrier_arrive(kRecFull, kThreads);  // this unit's records are written
        }
    } else {
        // ===== the merge warp ======================================================
        int k_unit = 0;
        for (int u = u_first; u < total_units; u = next_u(u), ++k_unit) {
            int s, kh, j, tok0, ntiles;
            decode_unit(u, s, kh, j, tok0, ntiles);
            const bool app = napp != 0 && tok0 + P >= ctx_s[s];
            const int nparts = own_partitions(ctx_s[s], start_s[s], P);
            // the first partials belong to the prefix pass
            const int pbase = prefix_partitions(start_s[s], P);
            const bool split = nparts > 1 || pbase > 0;
            named_barrier_sync(kRecFull, kThreads);  // every tile warp's records are in
            const float *av = app_v + (k_unit & 1) * D;
            const float *am = app_m + (k_unit & 1) * kHeads;
            const int items = G * (D / 8);
            for (int it = lane; it < items; it += 32) {
                const int jh = it / (D / 8);
                const int d0 = (it - jh * (D / 8)) * 8;
                float mmax = -INFINITY;
#pragma unroll
                for (int w = 0; w < NW; ++w)
                    mmax = fmaxf(mmax, merge_m[w * kHeads + jh]);
                if (app)
                    mmax = fmaxf(mmax, am[jh]);
                const float mu = mmax == -INFINITY ? 0.f : mmax;
                float lsum = 0.f;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float wgt = exp2f(merge_m[w * kHeads + jh] - mu);
                    lsum += wgt * merge_l[w * kHeads + jh];
                    const float4 *src = reinterpret_cast<const float4 *>(
                        merge_o + (w * kHeads + jh) * L::kPitch + d0);
                    const float4 x0 = src[0], x1 = src[1];
                    acc[0] += wgt * x0.x; acc[1] += wgt * x0.y; acc[2] += wgt * x0.z; acc[3] += wgt * x0.w;
                    acc[4] += wgt * x1.x; acc[5] += wgt * x1.y; acc[6] += wgt * x1.z; acc[7] += wgt * x1.w;
                }
                if (app) {
                    // the new token: m = its score, l = 1, o = its value row
                    const float wgt = exp2f(am[jh] - mu);
                    lsum += wgt;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        acc[e] += wgt * av[d0 + e];
                }
                const float inv = p.out_scale / lsum;
                const size_t h = (size_t)kh * G + jh;
                if (!split) {
                    T vals[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        vals[e] = MmaOp<T>::from_float(acc[e] * inv);
                    *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) +
                                               ((size_t)s * p.num_heads + h) * D + d0) =
                        *reinterpret_cast<const uint4 *>(vals);
                } else {
                    // partial of partition j, merged below (or by the reduce kernel)
                    const size_t idx = ((size_t)s * p.num_heads + h) * p.max_parts + pbase + j;
                    float4 *dst = reinterpret_cast<float4 *>(p.part_o + idx * D + d0);
                    dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
                    dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
                    if (d0 == 0) {
                        p.part_m[idx] = mmax * kLn2;
                        p.part_l[idx] = lsum;
                    }
                }
            }
            // the records (and the append buffer) may be rewritten; the tile
            // warps wait for this only from their next unit on
            if (next_u(u) < total_units)
                named_barrier_arrive(kRecFree, kThreads);
            if (split && p.counters != nullptr && pbase + nparts <= kMergeMax)
                // records loaded per lane at once: fewer under the FP8 register cap
                arrive_and_merge<T, D, kHeads, kFp8 ? 2 : 8>(p, s, kh, pbase + nparts, lane);
        }
    }
    if (kFp8 && __any_sync(kFull, q_over) && lane == 0)
        flag_error(p.error_word, PA_DEVERR_QUERY_RANGE);
    pdl_launch_dependents();

    // ---- drain: wait (bounded) for any fetch still landing in this warp's ring ----
    if (inflight != 0) {
        for (int k = 0; k < NST; ++k) {
            if (!(inflight & (1u << k)))
                continue;
            // the most recent fetch into stage k was issue number
            // issued - 1 - ((issued - 1 - k) % NST)
            const uint32_t last = issued - 1 - ((issued - 1 - k) % NST);
            mbar_wait_bounded(bar_of(k), (last / NST) & 1u, kDrainWaitNs);
        }
    }
    if (p.concurrent)
        pdl_wait_primary();  // the shared-prefix pass has finished
}

// ---- host side -------------------------------------------------------------------

#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 5
#endif
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 2
#endif
#ifndef PA_DECODE_MINB
#define PA_DECODE_MINB 2
#endif
#ifndef PA_DECODE_WARPS_FP8
#define PA_DECODE_WARPS_FP8 4
#endif
#ifndef PA_DECODE_STAGES_FP8
#define PA_DECODE_STAGES_FP8 3
#endif
#ifndef PA_DECODE_MINB_FP8
#define PA_DECODE_MINB_FP8 3
#endif
// 16-bit pools: tile warps per CTA (the merge warp comes on top), ring
// stages per warp, CTAs per SM the register budget is sized for.
constexpr int kWarps = PA_DECODE_WARPS;
constexpr int kStagesPerWarp = PA_DECODE_STAGES;
constexpr int kMinBlocks = PA_DECODE_MINB;
// FP8 pools: stages are half the size and the widening adds arithmetic per
// byte, so the kernel wants more warps per SM than the 16-bit one.
constexpr int kWarpsFp8 = PA_DECODE_WARPS_FP8;
constexpr int kStagesPerWarpFp8 = PA_DECODE_STAGES_FP8;
constexpr int kMinBlocksFp8 = PA_DECODE_MINB_FP8;
// Fewer stages for batches whose per-sequence shared arrays (8 B each) do
// not fit next to the default rings.
constexpr int kStagesManySeqs = 1;

template <typename T, typename KV, int D, int NT, int NST>
static pa_status launch_pass(const DecodeParams &prm, const CUtensorMap &mk,
                             const CUtensorMap &mv, cudaStream_t stream, long long max_units)
{
    constexpr bool kFp8 = sizeof(KV) == 1;
    constexpr int NW = kFp8 ? kWarpsFp8 : kWarps;
    // the 16-head variant keeps twice the accumulators: no register cap
    constexpr int MINB = NT > 1 ? 1 : kFp8 ? kMinBlocksFp8 : kMinBlocks;
    using L = Layout<D, NT, NW, NST, sizeof(KV)>;
    auto kernel = paged_decode_kernel<T, KV, D, NT, NW, NST, MINB>;
    constexpr int kThreads = (NW + 1) * 32;
    static KernelSetting setting[kMaxDevices];
    static std::mutex mu;
    const size_t smem = L::bytes(prm.num_seqs);
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
    const int sms = info.sms;
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
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ks.per_sm, kernel, kThreads, smem);
            if (e != cudaSuccess)
                return record_cuda(e);
            ks.smem_queried = smem;
        }
        per_sm = ks.per_sm;
    }
    if (per_sm < 1)
        return PA_ERR_UNSUPPORTED;
    long long grid = (long long)sms * per_sm;
    if (grid > max_units)
        grid = max_units;
    if (grid < 1)
        grid = 1;
    // Beside the shared-prefix pass, the partition CTAs that do not fit on
    // the SMs its CTAs hold (per_sm per such SM, the last ones dispatched)
    // start only when those CTAs end: they skip the first round of units.
    DecodeParams dp = prm;
    dp.early_ctas = (int)grid;
    dp.early_rounds = 0;
    if (prm.concurrent && prm.prefix_sms > 0 && prm.prefix_sms < sms) {
        const long long late = std::min<long long>(grid, (long long)per_sm * prm.prefix_sms);
        dp.early_ctas = (int)(grid - late);
        dp.early_rounds = dp.early_ctas > 0 ? 1 : 0;
    }
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kThreads), smem, stream, dp, mk, mv);
}

// The partition pass, then (prefix-aware decode) the shared-prefix pass, then
// the reduce when any partial exists; all on one stream, each a programmatic
// dependent of the one before.
struct PrefixPass {
    const MqParams *prm;
    pa_dtype dtype;        // the pools' (PA_FP8_E4M3 for e4m3 pools)
    pa_dtype query_dtype;  // the query's and the output's
    const void *key_cache, *value_cache;
    long long max_units;
};

template <typename T, typename KV, int D, int NT>
static pa_status launch_decode(const DecodeParams &prm, const CUtensorMap &mk,
                               const CUtensorMap &mv, cudaStream_t stream,
                               long long max_units, const PrefixPass *prefix = nullptr)
{
    constexpr int kStages = sizeof(KV) == 1 ? kStagesPerWarpFp8 : kStagesPerWarp;
    // prefix-aware decode: the shared-prefix pass (tensor cores) goes first
    // and the partition pass (memory-bound) runs alongside it
    DecodeParams pass = prm;
    pass.concurrent = 0;
    if (prefix != nullptr) {
        const pa_status ps = launch_prefix_pass(*prefix->prm, prefix->dtype,
                                                prefix->query_dtype, prefix->key_cache,
                                                prefix->value_cache, D, stream,
                                                prefix->max_units);
        if (ps != PA_OK)
            return ps;
        pass.concurrent = 1;
    }
    pa_status st = launch_pass<T, KV, D, NT, kStages>(pass, mk, mv, stream, max_units);
    if (st == PA_ERR_UNSUPPORTED)
        st = launch_pass<T, KV, D, NT, kStagesManySeqs>(pass, mk, mv, stream, max_units);
    // the pass merges split sequences of up to kMergeMax partials itself when
    // it has arrival counters; the reduce kernel merges the rest
    if (st != PA_OK || prm.max_parts <= 1 ||
        (prm.counters != nullptr && prm.max_parts <= kMergeMax))
        return st;
    return launch_reduce<T, D>(prm, stream);
}

} // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                            int head_dim, int max_context_len,
                                            int partition_size)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_context_len < 0 || partition_size < 0)
        return 0;
    const int parts = num_parts(max_context_len, partition_size);
    return workspace_layout(num_seqs, num_heads, num_kv_heads, head_dim, parts).total;
}

// 16-bit pools: tensor maps, then the kernel instance for (dtype, d, group).
static pa_status run_decode16(const DecodeParams &prm, const void *key_cache,
                              const void *value_cache, pa_dtype dtype, int num_seqs,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks,
                              void *stream)
{
    CUtensorMap mk, mv;
    if (!encode_pool_map(&mk, key_cache, dtype, num_blocks, block_size, num_kv_heads,
                         head_dim) ||
        !encode_pool_map(&mv, value_cache, dtype, num_blocks, block_size, num_kv_heads,
                         head_dim))
        return PA_ERR_CUDA;

    const long long max_units = (long long)num_seqs * num_kv_heads * prm.max_parts;
    cudaStream_t st = as_stream(stream);
    const bool bf = dtype == PA_BF16;
    const bool wide = prm.group > 8;
    using B16 = __nv_bfloat16;
    using F16 = __half;
    if (head_dim == 128) {
        if (bf)
            return wide ? launch_decode<B16, B16, 128, 2>(prm, mk, mv, st, max_units)
                        : launch_decode<B16, B16, 128, 1>(prm, mk, mv, st, max_units);
        return wide ? launch_decode<F16, F16, 128, 2>(prm, mk, mv, st, max_units)
                    : launch_decode<F16, F16, 128, 1>(prm, mk, mv, st, max_units);
    }
    if (bf)
        return wide ? launch_decode<B16, B16, 64, 2>(prm, mk, mv, st, max_units)
                    : launch_decode<B16, B16, 64, 1>(prm, mk, mv, st, max_units);
    return wide ? launch_decode<F16, F16, 64, 2>(prm, mk, mv, st, max_units)
                : launch_decode<F16, F16, 64, 1>(prm, mk, mv, st, max_units);
}

// FP8 (e4m3) pools, head_dim 128: scores use the K codes (the K scale folded
// into the exponent's scale), outputs and partials get the V scale.
static pa_status run_decode_fp8(DecodeParams &prm, const void *key_cache,
                                const void *value_cache, pa_dtype dtype, int num_seqs,
                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                float scale, float k_scale, float v_scale, void *stream)
{
    prm.scale_log2 = scale * k_scale * kLog2e;
    prm.out_scale = v_scale;
    CUtensorMap mk, mv;
    if (!encode_pool_map(&mk, key_cache, PA_FP8_E4M3, num_blocks, block_size, num_kv_heads,
                         head_dim) ||
        !encode_pool_map(&mv, value_cache, PA_FP8_E4M3, num_blocks, block_size, num_kv_heads,
                         head_dim))
        return PA_ERR_CUDA;
    const long long max_units = (long long)num_seqs * num_kv_heads * prm.max_parts;
    cudaStream_t st = as_stream(stream);
    const bool wide = prm.group > 8;
    using U8 = uint8_t;
    using B16 = __nv_bfloat16;
    if (head_dim == 128) {
        if (dtype == PA_BF16)
            return wide ? launch_decode<B16, U8, 128, 2>(prm, mk, mv, st, max_units)
                        : launch_decode<B16, U8, 128, 1>(prm, mk, mv, st, max_units);
        return wide ? launch_decode<__half, U8, 128, 2>(prm, mk, mv, st, max_units)
                    : launch_decode<__half, U8, 128, 1>(prm, mk, mv, st, max_units);
    }
    if (dtype == PA_BF16)
        return wide ? launch_decode<B16, U8, 64, 2>(prm, mk, mv, st, max_units)
                    : launch_decode<B16, U8, 64, 1>(prm, mk, mv, st, max_units);
    return wide ? launch_decode<__half, U8, 64, 2>(prm, mk, mv, st, max_units)
                : launch_decode<__half, U8, 64, 1>(prm, mk, mv, st, max_units);
}

static bool valid_fp8_scales(float k_scale, float v_scale)
{
    return std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f;
}

// The fused append's arguments: both new-row buffers, 16-byte aligned.
static pa_status set_append(DecodeParams *prm, void *key_cache, void *value_cache,
                            const void *new_key, const void *new_value, int32_t *slot_mapping)
{
    if (!new_key || !new_value || !aligned16(new_key) || !aligned16(new_value))
        return PA_ERR_INVALID_ARG;
    prm->key_cache = key_cache;
    prm->value_cache = value_cache;
    prm->new_key = new_key;
    prm->new_value = new_value;
    prm->slot_out = slot_mapping;
    return PA_OK;
}

extern "C" pa_status pa_decode_attention(void *out, const void *query, const void *key_cache,
                                         const void *value_cache, const int32_t *block_tables,
                                         int max_blocks_per_seq, const int32_t *context_lens,
                                         int max_context_len, int num_seqs, int num_heads,
                                         int num_kv_heads, int head_dim, int block_size,
                                         int num_blocks, float scale, int partition_size,
                                         void *workspace, size_t workspace_bytes,
                                         pa_dtype dtype, int32_t *error_word, void *stream)
{
    if (dtype != PA_F16 && dtype != PA_BF16)
        return PA_ERR_INVALID_ARG;
    DecodeParams prm{};
    const pa_status ok = prepare_decode(
        &prm, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
        context_lens, max_context_len, num_seqs, num_heads, num_kv_heads, head_dim,
        block_size, num_blocks, scale, partition_size, workspace, workspace_bytes,
        error_word);
    if (ok != PA_OK || num_seqs == 0)
        return ok;
    return run_decode16(prm, key_cache, value_cache, dtype, num_seqs, num_kv_heads, head_dim,
                        block_size, num_blocks, stream);
}

extern "C" pa_status pa_decode_attention_append(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    int partition_size, void *workspace, size_t workspace_bytes, pa_dtype dtype,
    int32_t *error_word, void *stream)
{
    if (dtype != PA_F16 && dtype != PA_BF16)
        return PA_ERR_INVALID_ARG;
    DecodeParams prm{};
    pa_status ok = prepare_decode(&prm, out, query, key_cache, value_cache, block_tables,
                                  max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                  scale, partition_size, workspace, workspace_bytes,
                                  error_word);
    if (ok != PA_OK || num_seqs == 0)
        return ok;
    ok = set_append(&prm, key_cache, value_cache, new_key, new_value, slot_mapping);
    if (ok != PA_OK)
        return ok;
    return run_decode16(prm, key_cache, value_cache, dtype, num_seqs, num_kv_heads, head_dim,
                        block_size, num_blocks, stream);
}

extern "C" pa_status pa_decode_attention_fp8(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, float k_scale, float v_scale,
    int partition_size, void *workspace, size_t workspace_bytes, pa_dtype dtype,
    int32_t *error_word, void *stream)
{
    if ((dtype != PA_F16 && dtype != PA_BF16) || !valid_fp8_scales(k_scale, v_scale))
        return PA_ERR_INVALID_ARG;
    DecodeParams prm{};
    const pa_status ok = prepare_decode(
        &prm, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
        context_lens, max_context_len, num_seqs, num_heads, num_kv_heads, head_dim,
        block_size, num_blocks, scale, partition_size, workspace, workspace_bytes,
        error_word);
    if (ok != PA_OK || num_seqs == 0)
        return ok;
    return run_decode_fp8(prm, key_cache, value_cache, dtype, num_seqs, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, k_scale, v_scale, stream);
}

extern "C" pa_status pa_decode_attention_append_fp8(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    float k_scale, float v_scale, int partition_size, void *workspace, size_t workspace_bytes,
    pa_dtype dtype, int32_t *error_word, void *stream)
{
    if ((dtype != PA_F16 && dtype != PA_BF16) || !valid_fp8_scales(k_scale, v_scale))
        return PA_ERR_INVALID_ARG;
    DecodeParams prm{};
    pa_status ok = prepare_decode(&prm, out, query, key_cache, value_cache, block_tables,
                                  max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                  scale, partition_size, workspace, workspace_bytes,
                                  error_word);
    if (ok != PA_OK || num_seqs == 0)
        return ok;
    ok = set_append(&prm, key_cache, value_cache, new_key, new_value, slot_mapping);
    if (ok != PA_OK)
        return ok;
    // the codes' contract: e4m3(x * (1 / scale)), the reciprocal taken in fp32
    prm.k_inv_scale = 1.0f / k_scale;
    prm.v_inv_scale = 1.0f / v_scale;
    return run_decode_fp8(prm, key_cache, value_cache, dtype, num_seqs, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, k_scale, v_scale, stream);
}

extern "C" size_t pa_prefix_plan_ints(int num_seqs, int num_groups, int num_members)
{
    if (num_seqs < 0 || num_groups < 0 || num_members < 0)
        return 0;
    return (size_t)num_seqs + 2 * (size_t)num_groups + 1 + (size_t)num_members;
}

extern "C" size_t pa_cascade_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                             int head_dim, int max_context_len,
                                             int partition_size)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_context_len < 0 || partition_size < 0)
        return 0;
    const int parts = num_parts(max_context_len, partition_size) + 1;
    return workspace_layout(num_seqs, num_heads, num_kv_heads, head_dim, parts).total;
}

// Prefix-aware decode; with new_key non-null, the decode step's append fused
// into its partition pass (the prefix pass reads only shared blocks, which
// never hold a new token).
static pa_status run_cascade(void *out, const void *query, void *key_cache, void *value_cache,
                             const void *new_key, const void *new_value, int32_t *slot_mapping,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, int max_context_len, int num_seqs,
                             int num_heads, int num_kv_heads, int head_dim, int block_size,
                             int num_blocks, float scale, const int32_t *prefix_plan,
                             int num_groups, int num_members, int partition_size,
                             void *workspace, size_t workspace_bytes, pa_dtype dtype,
                             bool fp8, float k_scale, float v_scale,
                             int32_t *error_word, void *stream)
{
    if (dtype != PA_F16 && dtype != PA_BF16)
        return dtype == PA_FP8_E4M3 && !fp8 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (num_groups < 0 || num_members < 0 || (num_groups > 0 && num_members < 2 * num_groups) ||
        !(scale > 0.f) || (fp8 && !valid_fp8_scales(k_scale, v_scale)))
        return PA_ERR_INVALID_ARG;
    if (num_groups == 0) {
        if (fp8) {
            if (new_key == nullptr)
                return pa_decode_attention_fp8(
                    out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                    context_lens, max_context_len, num_seqs, num_heads, num_kv_heads, head_dim,
                    block_size, num_blocks, scale, k_scale, v_scale, partition_size, workspace,
                    workspace_bytes, dtype, error_word, stream);
            return pa_decode_attention_append_fp8(
                out, query, key_cache, value_cache, new_key, new_value, slot_mapping,
                block_tables, max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, k_scale,
                v_scale, partition_size, workspace, workspace_bytes, dtype, error_word, stream);
        }
        if (new_key == nullptr)
            return pa_decode_attention(out, query, key_cache, value_cache, block_tables,
                                       max_blocks_per_seq, context_lens, max_context_len,
                                       num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                       num_blocks, scale, partition_size, workspace,
                                       workspace_bytes, dtype, error_word, stream);
        return pa_decode_attention_append(
            out, query, key_cache, value_cache, new_key, new_value, slot_mapping, block_tables,
            max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads,
            num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size, workspace,
            workspace_bytes, dtype, error_word, stream);
    }
    DecodeParams prm{};
    pa_status ok = prepare_decode(&prm, out, query, key_cache, value_cache, block_tables,
                                  max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                  scale, partition_size, workspace, workspace_bytes,
                                  error_word);
    if (ok != PA_OK || num_seqs == 0)
        return ok;
    if (prefix_plan == nullptr)
        return PA_ERR_INVALID_ARG;
    if (new_key != nullptr) {
        ok = set_append(&prm, key_cache, value_cache, new_key, new_value, slot_mapping);
        if (ok != PA_OK)
            return ok;
    }
    if (fp8) {
        // scores of the K codes (the K scale in the exponent's scale), the V
        // scale on the outputs and partials; the append's codes as
        // reshape_and_cache_fp8 computes them
        prm.scale_log2 = scale * k_scale * kLog2e;
        prm.out_scale = v_scale;
        prm.k_inv_scale = 1.0f / k_scale;
        prm.v_inv_scale = 1.0f / v_scale;
    }
    // the shared prefix [0, L) and the own tokens [L, ctx) are each cut into
    // partitions of part_tokens: ceil(L / P) + ceil((ctx - L) / P) <=
    // ceil(ctx / P) + 1 partials per (sequence, head)
    const int parts = prm.max_parts + 1;
    const WorkspaceLayout wl = workspace_layout(num_seqs, num_heads, num_kv_heads, head_dim,
                                                parts);
    if (workspace == nullptr || workspace_bytes < wl.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return PA_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    prm.part_m = reinterpret_cast<float *>(ws + wl.m_off);
    prm.part_l = reinterpret_cast<float *>(ws + wl.l_off);
    prm.part_o = reinterpret_cast<float *>(ws + wl.o_off);
    prm.max_parts = parts;
    // SMs the shared-prefix pass holds, taken as one CTA per SM for each of
    // its units with one partition of the prefix per group (its CTAs without
    // a unit end at once)
    prm.prefix_sms = (int)std::min<long long>(
        ((long long)num_members * prm.group + 127LL * num_groups) / 128 * num_kv_heads,
        1 << 30);
    prm.counters = reinterpret_cast<int32_t *>(ws + wl.cnt_off);
    prm.seq_start = prefix_plan;

    MqParams mq{};
    mq.query = query;
    mq.block_tables = block_tables;
    mq.context_lens = context_lens;
    mq.seq_start = prefix_plan;
    mq.group_start = prefix_plan + num_seqs;
    mq.group_prefix = prefix_plan + num_seqs + num_groups + 1;
    mq.group_members = prefix_plan + num_seqs + 2 * num_groups + 1;
    mq.part_m = prm.part_m;
    mq.part_l = prm.part_l;
    mq.part_o = prm.part_o;
    // sequences of up to kMergeMax partials are merged by whichever pass
    // completes their arrival counter, into the decode output
    mq.counters = prm.counters;
    mq.out = out;
    mq.error_word = error_word;
    mq.wait_ns = prm.wait_ns;
    mq.withhold_fill = prm.withhold_fill;
    mq.prefix_mode = 1;
    mq.num_segments = num_groups;
    mq.num_seqs = num_seqs;
    mq.num_heads = num_heads;
    mq.num_kv_heads = num_kv_heads;
    mq.group = prm.group;
    mq.max_blocks_per_seq = max_blocks_per_seq;
    mq.num_blocks = num_blocks;
    mq.block_size = block_size;
    mq.block_shift = prm.block_shift;
    mq.max_context_len = max_context_len;
    mq.max_parts = parts;
    mq.part_tokens = prm.part_tokens;
    mq.scale_log2 = prm.scale_log2;
    mq.out_scale = prm.out_scale;
    const long long prefix_parts = (max_context_len + prm.part_tokens - 1) / prm.part_tokens;
    const pa_dtype pool_dtype = fp8 ? PA_FP8_E4M3 : dtype;
    PrefixPass pp{&mq, pool_dtype, dtype, key_cache, value_cache,
                  ((long long)num_members * prm.group / 128 + num_groups) * prefix_parts *
                      num_kv_heads};

    CUtensorMap mk, mv;
    if (!encode_pool_map(&mk, key_cache, pool_dtype, num_blocks, block_size, num_kv_heads,
                         head_dim) ||
        !encode_pool_map(&mv, value_cache, pool_dtype, num_blocks, block_size, num_kv_heads,
                         head_dim))
        return PA_ERR_CUDA;
    const long long max_units = (long long)num_seqs * num_kv_heads * parts;
    cudaStream_t st = as_stream(stream);
    const bool bf = dtype == PA_BF16;
    const bool wide = prm.group > 8;
    using B16 = __nv_bfloat16;
    using F16 = __half;
    using U8 = uint8_t;
    if (fp8 && head_dim == 128) {
        if (bf)
            return wide ? launch_decode<B16, U8, 128, 2>(prm, mk, mv, st, max_units, &pp)
                        : launch_decode<B16, U8, 128, 1>(prm, mk, mv, st, max_units, &pp);
        return wide ? launch_decode<F16, U8, 128, 2>(prm, mk, mv, st, max_units, &pp)
                    : launch_decode<F16, U8, 128, 1>(prm, mk, mv, st, max_units, &pp);
    }
    if (fp8) {
        if (bf)
            return wide ? launch_decode<B16, U8, 64, 2>(prm, mk, mv, st, max_units, &pp)
                        : launch_decode<B16, U8, 64, 1>(prm, mk, mv, st, max_units, &pp);
        return wide ? launch_decode<F16, U8, 64, 2>(prm, mk, mv, st, max_units, &pp)
                    : launch_decode<F16, U8, 64, 1>(prm, mk, mv, st, max_units, &pp);
    }
    if (head_dim == 128) {
        if (bf)
            return wide ? launch_decode<B16, B16, 128, 2>(prm, mk, mv, st, max_units, &pp)
                        : launch_decode<B16, B16, 128, 1>(prm, mk, mv, st, max_units, &pp);
        return wide ? launch_decode<F16, F16, 128, 2>(prm, mk, mv, st, max_units, &pp)
                    : launch_decode<F16, F16, 128, 1>(prm, mk, mv, st, max_units, &pp);
    }
    if (bf)
        return wide ? launch_decode<B16, B16, 64, 2>(prm, mk, mv, st, max_units, &pp)
                    : launch_decode<B16, B16, 64, 1>(prm, mk, mv, st, max_units, &pp);
    return wide ? launch_decode<F16, F16, 64, 2>(prm, mk, mv, st, max_units, &pp)
                : launch_decode<F16, F16, 64, 1>(prm, mk, mv, st, max_units, &pp);
}

extern "C" pa_status pa_decode_attention_cascade(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, const int32_t *prefix_plan, int num_groups,
    int num_members, int partition_size, void *workspace, size_t workspace_bytes,
    pa_dtype dtype, int32_t *error_word, void *stream)
{
    return run_cascade(out, query, const_cast<void *>(key_cache),
                       const_cast<void *>(value_cache), nullptr, nullptr, nullptr,
                       block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       scale, prefix_plan, num_groups, num_members, partition_size, workspace,
                       workspace_bytes, dtype, false, 1.f, 1.f, error_word, stream);
}

extern "C" pa_status pa_decode_attention_cascade_fp8(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, float scale, float k_scale, float v_scale,
    const int32_t *prefix_plan, int num_groups, int num_members, int partition_size,
    void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *error_word, void *stream)
{
    return run_cascade(out, query, const_cast<void *>(key_cache),
                       const_cast<void *>(value_cache), nullptr, nullptr, nullptr,
                       block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       scale, prefix_plan, num_groups, num_members, partition_size, workspace,
                       workspace_bytes, dtype, true, k_scale, v_scale, error_word, stream);
}

extern "C" pa_status pa_decode_attention_cascade_append(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    const int32_t *prefix_plan, int num_groups, int num_members, int partition_size,
    void *workspace, size_t workspace_bytes, pa_dtype dtype, int32_t *error_word, void *stream)
{
    if (num_seqs > 0 && (new_key == nullptr || new_value == nullptr))
        return PA_ERR_INVALID_ARG;
    return run_cascade(out, query, key_cache, value_cache, new_key, new_value, slot_mapping,
                       block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       scale, prefix_plan, num_groups, num_members, partition_size, workspace,
                       workspace_bytes, dtype, false, 1.f, 1.f, error_word, stream);
}

extern "C" pa_status pa_decode_attention_cascade_append_fp8(
    void *out, const void *query, void *key_cache, void *value_cache, const void *new_key,
    const void *new_value, int32_t *slot_mapping, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int num_seqs,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
    float k_scale, float v_scale, const int32_t *prefix_plan, int num_groups, int num_members,
    int partition_size, void *workspace, size_t workspace_bytes, pa_dtype dtype,
    int32_t *error_word, void *stream)
{
    if (num_seqs > 0 && (new_key == nullptr || new_value == nullptr))
        return PA_ERR_INVALID_ARG;
    return run_cascade(out, query, key_cache, value_cache, new_key, new_value, slot_mapping,
                       block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       scale, prefix_plan, num_groups, num_members, partition_size, workspace,
                       workspace_bytes, dtype, true, k_scale, v_scale, error_word, stream);
}
