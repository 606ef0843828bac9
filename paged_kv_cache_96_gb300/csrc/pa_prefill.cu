// pa_prefill.cu -- multi-query paged attention for sm_103a.
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
//    blocks): the decode queries of every member of a group attend the
//    group's shared prefix [0, L) once, read through the first member's
//    table, and leave a partial (m, l, o) per (sequence, head) for the
//    split-context reduce to merge with the members' own partitions.
//
// Design (GB300): the rows of one KV head -- a chunk's tokens times the G
// query heads of the group, or the members' decode queries times G -- are
// the M dimension of mma.sync m16n8k16 tiles; 64 rows per CTA (4 warps x 16
// rows), keys and values stream through a 2-stage shared-memory ring of
// 64-token tiles fetched by 4-D TMA loads (the same 2 KB boxes and 128-byte
// swizzle as the decode pass), the score tile S = Q K^T and O += P V stay
// in registers (FA2 register reuse: the S accumulator fragment is the A
// operand of P V), softmax is online in fp32 log2 units.  Causal rows only
// fetch the tiles up to the tile's last position; tokens past a row's limit
// are masked in the scores and value rows past the key range are zeroed
// before the contraction (no poisoned slot reaches the output).
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pa_decode_common.cuh"
#include "pa_prefill.cuh"

namespace pa {

constexpr int kMqWarps = 4;
constexpr int kMqRows = 16 * kMqWarps;  // query rows per CTA
constexpr int kMqTokens = 64;           // key/value tokens per stage
constexpr int kMqSubs = kMqTokens / kTileTokens;
constexpr int kMqStages = 2;

template <int D> struct MqLayout {
    static constexpr int kSubBytes = kTileTokens * D * 2;  // one 16-token K (or V) tile
    static constexpr int kKVBytes = kMqSubs * kSubBytes;   // 64 tokens of K (or V)
    static constexpr int kStageBytes = 2 * kKVBytes;
    static constexpr int kQPitch = D + 8;                  // elements per staged query row
    static constexpr int kQ = kMqStages * kStageBytes;
    static constexpr int kRowQ = kQ + kMqRows * kQPitch * 2;  // int64 query row offsets
    static constexpr int kRowO = kRowQ + kMqRows * 8;          // int64 output offsets
    static constexpr int kRowLim = kRowO + kMqRows * 8;        // int key limits
    static constexpr int kBars = kRowLim + kMqRows * 4;
    static constexpr int kSeg = kBars + kMqStages * 8;         // int tile prefix[n + 1]
    static size_t bytes(int segments) { return 1024 + kSeg + 4 * ((size_t)segments + 1); }
    static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
    static_assert(kBars % 8 == 0, "mbarriers need 8-byte alignment");
};

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

template <typename T, int D>
__global__ void __launch_bounds__(kMqWarps * 32)
    paged_mq_kernel(const __grid_constant__ MqParams p,
                    const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v)
{
    using L = MqLayout<D>;
    using Op = MmaOp<T>;
    constexpr int KT = D / 16;  // k-steps of the score product
    constexpr int NO = D / 8;   // n-tiles of the output
    constexpr int kThreads = kMqWarps * 32;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);
    T *qs = reinterpret_cast<T *>(smem + L::kQ);
    long long *row_q = reinterpret_cast<long long *>(smem + L::kRowQ);
    long long *row_o = reinterpret_cast<long long *>(smem + L::kRowO);
    int *row_lim = reinterpret_cast<int *>(smem + L::kRowLim);
    int *pref = reinterpret_cast<int *>(smem + L::kSeg);
    auto bar_of = [&](int st) { return sbase + L::kBars + st * 8; };
    auto stage_of = [&](int st) { return sbase + st * L::kStageBytes; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int G = p.group, Hkv = p.num_kv_heads, H = p.num_heads;
    const int nseg = p.num_segments;

    if (tid == 0) {
        for (int k = 0; k < kMqStages; ++k)
            mbar_init(bar_of(k), 1);
        fence_barrier_init();
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    pdl_wait_primary();

    // ---- row tiles per segment and their prefix sums ------------------------------
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < nseg; base += 32) {
            const int sg = base + lane;
            const int n = sg < nseg ? (mq_segment_count(p, sg) * G + kMqRows - 1) / kMqRows : 0;
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, x, o);
                if (lane >= o)
                    x += y;
            }
            if (sg < nseg)
                pref[sg] = carry + x - n;
            carry += __shfl_sync(kFull, x, 31);
        }
        if (lane == 0)
            pref[nseg] = carry;
    }
    __syncthreads();
    const int total_units = pref[nseg] * Hkv;

    uint32_t phase = 0;     // parity bit per stage
    uint32_t pending = 0;   // stages with a fill not yet waited for
    bool aborted = false;

    // ldmatrix lane selectors
    const int li = lane & 7, mi = lane >> 3;
    // address of 16-byte chunk `chunk` (0..7) of d-half `half` of token `tok`
    // (0..15) in the 16-token tile at `base` (TMA 128-byte swizzle)
    auto tile_addr = [](uint32_t base, int tok, int half, int chunk) -> uint32_t {
        const int r = half * kTileTokens + tok;
        return base + r * 128 + ((chunk ^ (r & 7)) << 4);
    };

    for (int u = blockIdx.x; u < total_units && !aborted; u += gridDim.x) {
        // ---- unit -> (segment, KV head, row tile) ---------------------------------
        const int q = u / Hkv;
        const int kh = u - q * Hkv;
        int lo = 0, hi = nseg - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pref[mid] <= q)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int seg = lo;
        const int rt = q - pref[seg];
        const int count = mq_segment_count(p, seg);
        const int nrows = min(kMqRows, count * G - rt * kMqRows);

        // the table the keys are read through, and the key range of the tile
        int table_seq, kend;
        if (p.prefix_mode) {
            // a bad leader id is flagged by the plan check below
            table_seq = min(max(p.group_members[p.group_start[seg]], 0), p.num_seqs - 1);
            kend = min(max(p.group_prefix[seg], 0), p.max_blocks_per_seq * p.block_size);
        } else {
            table_seq = seg;
            const int ctx = clamp_context_mq(p, seg);
            const int last = (rt * kMqRows + nrows - 1) / G;  // chunk row of the tile's last row
            kend = max(0, ctx - count + last + 1);
        }
        const int32_t *table = p.block_tables + (size_t)table_seq * p.max_blocks_per_seq;
        const int nstages = (kend + kMqTokens - 1) / kMqTokens;

        __syncthreads();  // the previous unit is done with the stages, rows and Q tile

        // prefix pass, first KV head: check the plan for this tile's members --
        // the group's length is on the tile grid and within every member's
        // context, each member records it as its start, and each member's
        // table names the leader's blocks for the whole prefix
        if (p.prefix_mode && kh == 0 && tid < nrows && (rt * kMqRows + tid) % G == 0) {
            const int s = p.group_members[p.group_start[seg] + (rt * kMqRows + tid) / G];
            const int L = p.group_prefix[seg];
            const int leader = p.group_members[p.group_start[seg]];
            bool bad = s < 0 || s >= p.num_seqs || L <= 0 || (L & (kTileTokens - 1)) != 0 ||
                       L > p.max_blocks_per_seq * p.block_size || leader < 0 ||
                       leader >= p.num_seqs;
            if (!bad) {
                const int c = p.context_lens[s];
                bad = c < L || c > p.max_context_len || p.seq_start[s] != L;
                const int32_t *mine = p.block_tables + (size_t)s * p.max_blocks_per_seq;
                for (int b = 0; !bad && b < (L >> p.block_shift); ++b)
                    bad = __ldg(mine + b) != __ldg(table + b);
            }
            if (bad)
                flag_error(p.error_word, PA_DEVERR_PREFIX_PLAN);
        }

        auto issue = [&](int j) {  // thread 0: fetch key/value tile j into stage j % 2
            const int st = j % kMqStages;
            const int t0 = j * kMqTokens;
            const int nsub = min(kMqSubs, (kend - t0 + kTileTokens - 1) / kTileTokens);
            mbar_arrive_expect_tx(bar_of(st), (uint32_t)(nsub * 2 * L::kSubBytes));
            for (int sb = 0; sb < nsub; ++sb) {
                const int tok = t0 + sb * kTileTokens;
                int phys = __ldg(table + (tok >> p.block_shift));
                if (phys < 0 || phys >= p.num_blocks) {
                    flag_error(p.error_word, PA_DEVERR_BLOCK_RANGE);
                    phys = 0;  // stays inside the pool; the row's output is undefined
                }
                const int row = tok & (p.block_size - 1);
                const uint32_t dst = stage_of(st) + sb * L::kSubBytes;
#pragma unroll
                for (int hf = 0; hf < D / 64; ++hf) {
                    tma_load_4d(dst + hf * (L::kSubBytes / (D / 64)), &tmap_k, bar_of(st),
                                hf * 64, kh, row, phys);
                    tma_load_4d(dst + L::kKVBytes + hf * (L::kSubBytes / (D / 64)), &tmap_v,
                                bar_of(st), hf * 64, kh, row, phys);
                }
            }
        };
        if (tid == 0) {
            for (int j = 0; j < min(kMqStages, nstages); ++j)
                issue(j);
        }
        pending = (1u << min(kMqStages, nstages)) - 1u;

        // ---- row descriptors: query row, output location, key limit ----------------
        if (tid < kMqRows) {
            long long qoff = -1, ooff = -1;
            int lim = 0;
            if (tid < nrows) {
                const int r = rt * kMqRows + tid;
                const int i = r / G, hg = r - (r / G) * G;
                const int h = kh * G + hg;
                if (p.prefix_mode) {
                    int s = p.group_members[p.group_start[seg] + i];
                    s = min(max(s, 0), p.num_seqs - 1);  // a bad member id is flagged above
                    qoff = ((long long)s * H + h) * D;
                    ooff = ((long long)s * H + h) * p.max_parts;  // partial 0 of (s, h)
                    lim = kend;
                } else {
                    const long long row = (long long)p.query_start[seg] + i;
                    qoff = (row * H + h) * D;
                    ooff = qoff;
                    lim = max(0, kend - (((rt * kMqRows + nrows - 1) / G) - i));
                }
            }
            row_q[tid] = qoff;
            row_o[tid] = ooff;
            row_lim[tid] = lim;
        }
        __syncthreads();
        // ---- query tile into shared memory (zero rows past the tile) --------------
        for (int c = tid; c < kMqRows * (D / 8); c += kThreads) {
            const int r = c / (D / 8), ch = c - r * (D / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (row_q[r] >= 0)
                v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const T *>(p.query) +
                                                          row_q[r]) + ch);
            *reinterpret_cast<uint4 *>(qs + r * L::kQPitch + ch * 8) = v;
        }
        __syncthreads();
        uint32_t qa[KT][4];
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            const int r = warp * 16 + li + (mi & 1) * 8;
            const int col = kk * 16 + (mi >> 1) * 8;
            ldmatrix_x4(smem_addr(qs + r * L::kQPitch + col), qa[kk]);
        }
        const int lim0 = row_lim[warp * 16 + g], lim1 = row_lim[warp * 16 + g + 8];

        float o[NO][4];
#pragma unroll
        for (int n = 0; n < NO; ++n)
            o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

        for (int j = 0; j < nstages; ++j) {
            const int st = j % kMqStages;
            const bool ok = mbar_wait_bounded(bar_of(st), (phase >> st) & 1u, kWaitLimitNs);
            phase ^= 1u << st;
            pending &= ~(1u << st);
            if (__syncthreads_or(!ok)) {
                if (tid == 0)
                    flag_error(p.error_word, PA_DEVERR_TIMEOUT);
                aborted = true;
                break;
            }
            const uint32_t kb = stage_of(st), vb = kb + L::kKVBytes;
            const int t0 = j * kMqTokens;

            // S[16 rows x 64 tokens] = Q K^T
            float sacc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n)
                sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll
            for (int sb = 0; sb < kMqSubs; ++sb) {
                if (t0 + sb * kTileTokens >= kend)
                    break;  // sub-tile not fetched (uniform across the CTA)
#pragma unroll
                for (int kk = 0; kk < KT; ++kk) {
                    uint32_t b[4];
                    const int tok = (mi >> 1) * 8 + li;
                    const int dc = (kk & 3) * 2 + (mi & 1);
                    ldmatrix_x4(tile_addr(kb + sb * L::kSubBytes, tok, kk >> 2, dc), b);
                    Op::run(sacc[2 * sb], qa[kk], b[0], b[1]);
                    Op::run(sacc[2 * sb + 1], qa[kk], b[2], b[3]);
                }
            }

            // online softmax (log2 units) with the causal / range mask
            float mx0 = m0, mx1 = m1;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const int tk = t0 + n * 8 + 2 * t4;
                sacc[n][0] = tk < lim0 ? sacc[n][0] * p.scale_log2 : -INFINITY;
                sacc[n][1] = tk + 1 < lim0 ? sacc[n][1] * p.scale_log2 : -INFINITY;
                sacc[n][2] = tk < lim1 ? sacc[n][2] * p.scale_log2 : -INFINITY;
                sacc[n][3] = tk + 1 < lim1 ? sacc[n][3] * p.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, fmaxf(sacc[n][0], sacc[n][1]));
                mx1 = fmaxf(mx1, fmaxf(sacc[n][2], sacc[n][3]));
            }
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
            }
            const float al0 = mx0 == -INFINITY ? 1.f : exp2f(m0 - mx0);
            const float al1 = mx1 == -INFINITY ? 1.f : exp2f(m1 - mx1);
            m0 = mx0;
            m1 = mx1;
            const float mu0 = mx0 == -INFINITY ? 0.f : mx0;
            const float mu1 = mx1 == -INFINITY ? 0.f : mx1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int n = 0; n < NO; ++n) {
                o[n][0] *= al0;
                o[n][1] *= al0;
                o[n][2] *= al1;
                o[n][3] *= al1;
            }
            uint32_t pa[4][4];  // P as the A operand, one k-step per 16 tokens
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const float p0 = exp2f(sacc[n][0] - mu0), p1 = exp2f(sacc[n][1] - mu0);
                const float p2 = exp2f(sacc[n][2] - mu1), p3 = exp2f(sacc[n][3] - mu1);
                l0 += p0 + p1;
                l1 += p2 + p3;
                pa[n >> 1][(n & 1) * 2 + 0] = Op::pack(p0, p1);
                pa[n >> 1][(n & 1) * 2 + 1] = Op::pack(p2, p3);
            }

            // O[16 x D] += P V; value rows past the key range are zeroed
#pragma unroll
            for (int sb = 0; sb < kMqSubs; ++sb) {
                const int nv = kend - (t0 + sb * kTileTokens);
                if (nv <= 0)
                    break;
                const uint32_t m01 = (2 * t4 < nv ? 0x0000ffffu : 0u) |
                                     (2 * t4 + 1 < nv ? 0xffff0000u : 0u);
                const uint32_t m89 = (2 * t4 + 8 < nv ? 0x0000ffffu : 0u) |
                                     (2 * t4 + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
                for (int np = 0; np < NO / 2; ++np) {
                    uint32_t b[4];
                    const int tok = (mi & 1) * 8 + li;
                    const int d = np * 16 + (mi >> 1) * 8;
                    ldmatrix_x4_trans(tile_addr(vb + sb * L::kSubBytes, tok, d >> 6, (d & 63) >> 3),
                                      b);
                    Op::run(o[2 * np], pa[sb], b[0] & m01, b[1] & m89);
                    Op::run(o[2 * np + 1], pa[sb], b[2] & m01, b[3] & m89);
                }
            }

            // everyone is done with stage st: refill it with tile j + 2
            __syncthreads();
            if (j + kMqStages < nstages) {
                if (tid == 0)
                    issue(j + kMqStages);
                pending |= 1u << st;
            }
        }
        if (aborted)
            break;

        // ---- epilogue -------------------------------------------------------------------
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, off);
            l1 += __shfl_xor_sync(kFull, l1, off);
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = warp * 16 + g + half * 8;
            const long long ooff = row_o[r];
            if (ooff < 0)
                continue;
            const float l = half ? l1 : l0;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (p.prefix_mode) {
                float *po = p.part_o + ooff * D;
#pragma unroll
                for (int n = 0; n < NO; ++n)
                    *reinterpret_cast<float2 *>(po + n * 8 + 2 * t4) =
                        make_float2(o[n][half * 2] * inv, o[n][half * 2 + 1] * inv);
                if (t4 == 0) {
                    p.part_m[ooff] = (half ? m1 : m0) * kLn2;
                    p.part_l[ooff] = l;
                }
            } else {
                T *po = static_cast<T *>(p.out) + ooff;
#pragma unroll
                for (int n = 0; n < NO; ++n)
                    *reinterpret_cast<uint32_t *>(po + n * 8 + 2 * t4) =
                        Op::pack(o[n][half * 2] * inv, o[n][half * 2 + 1] * inv);
            }
        }
    }
    pdl_launch_dependents();

    // ---- drain: a fill still landing (only after an abort) -------------------------------
    if (tid == 0) {
        for (int st = 0; st < kMqStages; ++st)
            if (pending & (1u << st))
                mbar_wait_bounded(bar_of(st), (phase >> st) & 1u, kWaitLimitNs);
    }
}

// ---- host side -------------------------------------------------------------------

template <typename T, int D>
static pa_status launch_mq(const MqParams &prm, const CUtensorMap &mk, const CUtensorMap &mv,
                           cudaStream_t stream, long long max_units)
{
    using L = MqLayout<D>;
    auto kernel = paged_mq_kernel<T, D>;
    static KernelSetting setting[kMaxDevices];
    static std::mutex mu;
    const size_t smem = L::bytes(prm.num_segments);
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
            if (e != cudaSuccess)
                return record_cuda(e);
            ks.smem_enabled = smem;
        }
        if (smem != ks.smem_queried) {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ks.per_sm, kernel,
                                                              kMqWarps * 32, smem);
            if (e != cudaSuccess)
                return record_cuda(e);
            ks.smem_queried = smem;
        }
        per_sm = ks.per_sm;
    }
    if (per_sm < 1)
        return PA_ERR_UNSUPPORTED;
    long long grid = std::min<long long>((long long)info.sms * per_sm, max_units);
    if (grid < 1)
        grid = 1;
    return launch_pdl(kernel, dim3((unsigned)grid), dim3(kMqWarps * 32), smem, stream, prm, mk,
                      mv);
}

static pa_status dispatch_mq(const MqParams &prm, pa_dtype dtype, const void *key_cache,
                             const void *value_cache, int head_dim, cudaStream_t stream,
                             long long max_units)
{
    CUtensorMap mk, mv;
    if (!encode_pool_map(&mk, key_cache, dtype, prm.num_blocks, prm.block_size,
                         prm.num_kv_heads, head_dim) ||
        !encode_pool_map(&mv, value_cache, dtype, prm.num_blocks, prm.block_size,
                         prm.num_kv_heads, head_dim))
        return PA_ERR_CUDA;
    using B16 = __nv_bfloat16;
    if (head_dim == 128)
        return dtype == PA_BF16 ? launch_mq<B16, 128>(prm, mk, mv, stream, max_units)
                                : launch_mq<__half, 128>(prm, mk, mv, stream, max_units);
    return dtype == PA_BF16 ? launch_mq<B16, 64>(prm, mk, mv, stream, max_units)
                            : launch_mq<__half, 64>(prm, mk, mv, stream, max_units);
}

pa_status launch_prefix_pass(const MqParams &prm, pa_dtype dtype, const void *key_cache,
                             const void *value_cache, int head_dim, cudaStream_t stream,
                             long long max_units)
{
    return dispatch_mq(prm, dtype, key_cache, value_cache, head_dim, stream, max_units);
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill_attention(void *out, const void *query, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          int max_blocks_per_seq, const int32_t *query_start,
                                          const int32_t *context_lens, int max_context_len,
                                          int num_seqs, int num_tokens, int num_heads,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float scale, pa_dtype dtype,
                                          int32_t *error_word, void *stream)
{
    if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        max_context_len < 0 || !std::isfinite(scale) || num_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    if (dtype != PA_F16 && dtype != PA_BF16)
        return dtype == PA_FP8_E4M3 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_tokens == 0)
        return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !query_start ||
        !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) ||
        !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if ((head_dim != 64 && head_dim != 128) || block_size < kTileTokens || block_size > 256 ||
        (block_size & (block_size - 1)) != 0 || group > 16 ||
        (long long)num_blocks * block_size >= (1ll << 31) ||
        (long long)max_blocks_per_seq * block_size >= (1ll << 31))
        return PA_ERR_UNSUPPORTED;

    MqParams prm{};
    prm.out = out;
    prm.query = query;
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.query_start = query_start;
    prm.error_word = error_word;
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
    prm.scale_log2 = scale * kLog2e;
    // row tiles: at most one partial tile per sequence beyond the full ones
    const long long max_units =
        ((long long)num_tokens * group / kMqRows + num_seqs) * num_kv_heads;
    return dispatch_mq(prm, dtype, key_cache, value_cache, head_dim, as_stream(stream),
                       max_units);
}
