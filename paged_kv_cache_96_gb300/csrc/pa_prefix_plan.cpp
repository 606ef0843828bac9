// pa_prefix_plan.cpp -- host planner of prefix-aware decode: which
// sequences of a batch share leading physical blocks, and how long a prefix
// each group reads once ("vLLM 架构详解", "共享前缀的 Block 复用": block
// tables of requests with a common system prompt name the same physical
// blocks, whose reference counts exceed one).
//
// Sequences are ordered by their table rows, so that any set of sequences
// sharing k leading blocks is a contiguous run whose neighbouring pairs share
// at least k blocks.  A run grouped at its smallest neighbouring overlap m
// saves (size - 1) * m block reads; splitting the run where the overlap is
// exactly m gives sub-runs with longer prefixes.  The recursion keeps, for
// every run, the better of the two (ties: one group).
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/paged_attention.h"

namespace {

struct Planner {
    const int32_t *tables;
    int mb;
    std::vector<int> order;  // candidate sequences, sorted by table row
    std::vector<int> cap;    // per sequence: blocks a prefix may cover
    std::vector<int> lcp;    // lcp[i]: shared leading blocks of order[i], order[i + 1]
    int min_blocks;

    struct Group {
        int first, last, blocks;  // run [first, last) of `order`
    };

    // Best grouping of run [a, b): saved block reads, groups appended to out.
    long long solve(int a, int b, std::vector<Group> &out) const
    {
        if (b - a < 2)
            return 0;
        int m = lcp[a];
        for (int i = a + 1; i < b - 1; ++i)
            m = std::min(m, lcp[i]);
        std::vector<Group> split;
        long long saved_split = 0;
        int start = a;
        for (int i = a; i < b - 1; ++i) {
            if (lcp[i] == m) {
                saved_split += solve(start, i + 1, split);
                start = i + 1;
            }
        }
        saved_split += solve(start, b, split);
        const long long saved_whole = m >= min_blocks ? (long long)(b - a - 1) * m : 0;
        if (saved_whole > 0 && saved_whole >= saved_split) {
            out.push_back({a, b, m});
            return saved_whole;
        }
        out.insert(out.end(), split.begin(), split.end());
        return saved_split;
    }
};

}  // namespace

extern "C" pa_status pa_plan_prefix_groups(const int32_t *block_tables, int max_blocks_per_seq,
                                           const int32_t *context_lens, int num_seqs,
                                           int block_size, int min_shared_blocks, int32_t *plan,
                                           size_t plan_capacity, int *num_groups,
                                           int *num_members)
{
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || !num_groups ||
        !num_members || (num_seqs > 0 && (!block_tables || !context_lens || !plan)))
        return PA_ERR_INVALID_ARG;
    *num_groups = 0;
    *num_members = 0;
    if (plan_capacity < (size_t)num_seqs + 1)
        return PA_ERR_WORKSPACE;
    Planner pl;
    pl.tables = block_tables;
    pl.mb = max_blocks_per_seq;
    pl.min_blocks = std::max(1, min_shared_blocks);
    pl.cap.assign(num_seqs, 0);
    for (int s = 0; s < num_seqs; ++s) {
        const int ctx = context_lens[s];
        // a shared prefix ends before the sequence's last token
        pl.cap[s] = ctx > 0 ? std::min((ctx - 1) / block_size, max_blocks_per_seq) : 0;
        if (pl.cap[s] >= pl.min_blocks)
            pl.order.push_back(s);
    }
    auto row = [&](int s) { return block_tables + (size_t)s * max_blocks_per_seq; };
    std::sort(pl.order.begin(), pl.order.end(), [&](int x, int y) {
        const int n = std::min(pl.cap[x], pl.cap[y]);
        const int32_t *rx = row(x), *ry = row(y);
        for (int i = 0; i < n; ++i)
            if (rx[i] != ry[i])
                return rx[i] < ry[i];
        if (pl.cap[x] != pl.cap[y])
            return pl.cap[x] < pl.cap[y];
        return x < y;
    });
    const int n = (int)pl.order.size();
    pl.lcp.assign(n > 0 ? n - 1 : 0, 0);
    for (int i = 0; i + 1 < n; ++i) {
        const int x = pl.order[i], y = pl.order[i + 1];
        const int lim = std::min(pl.cap[x], pl.cap[y]);
        const int32_t *rx = row(x), *ry = row(y);
        int k = 0;
        while (k < lim && rx[k] == ry[k])
            ++k;
        pl.lcp[i] = k;
    }
    std::vector<Planner::Group> groups;
    pl.solve(0, n, groups);
    std::sort(groups.begin(), groups.end(),
              [](const Planner::Group &x, const Planner::Group &y) { return x.first < y.first; });

    size_t members = 0;
    for (const auto &gr : groups)
        members += (size_t)(gr.last - gr.first);
    const size_t need = (size_t)num_seqs + 2 * groups.size() + 1 + members;
    if (need > plan_capacity)
        return PA_ERR_WORKSPACE;
    const int G = (int)groups.size();
    int32_t *seq_prefix = plan;
    int32_t *gstart = plan + num_seqs;
    int32_t *gprefix = gstart + G + 1;
    int32_t *gmembers = gprefix + G;
    std::fill(seq_prefix, seq_prefix + num_seqs, 0);
    int pos = 0;
    for (int gi = 0; gi < G; ++gi) {
        const auto &gr = groups[gi];
        gstart[gi] = pos;
        gprefix[gi] = gr.blocks * block_size;
        for (int i = gr.first; i < gr.last; ++i) {
            const int s = pl.order[i];
            gmembers[pos++] = s;
            seq_prefix[s] = gr.blocks * block_size;
        }
    }
    gstart[G] = pos;
    *num_groups = G;
    *num_members = pos;
    return PA_OK;
}
