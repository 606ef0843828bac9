// pa_block_manager.cpp -- host block manager of the paged KV cache.
//
// What it keeps ("PagedAttention & Continuous Batching" §1.3-§1.5; "vLLM 架构
// 详解", "Block Table 实现" and "共享前缀的 Block 复用"; "vLLM源码解析(二)"
// §3.2 copy-on-write and §4.2 block allocation; "vLLM核心机制" §3.1): a
// reference count per physical block, and per sequence a block table and a
// token count.  Appending a token at position p opens a new block when p is
// a multiple of the block size and otherwise writes into the last block;
// a last block that other tables also name is first copied (copy-on-write:
// allocate, hand the (old, new) pair to the engine's block copy, remap, drop
// a reference).  Forking shares every block of the parent; freeing drops one
// reference per block.  Free blocks are taken lowest id first (a min-heap).
//
// Design: O(log N) allocation and release, O(1) per appended token, no
// allocation on the append path beyond a table's growth; every failing call
// checks first and changes nothing.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <new>
#include <queue>
#include <unordered_map>
#include <vector>

#include "../../include/paged_attention.h"

struct pa_block_manager {
    struct Seq {
        std::vector<int32_t> table;
        int64_t tokens = 0;
    };
    int num_blocks = 0, block_size = 0, max_blocks_per_seq = 0;
    std::vector<int32_t> ref;
    std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_heap;
    std::unordered_map<int, Seq> seqs;

    int32_t take()  // the lowest free block; the caller checked there is one
    {
        const int32_t b = free_heap.top();
        free_heap.pop();
        ref[b] = 1;
        return b;
    }
    void release(int32_t b)
    {
        if (--ref[b] == 0)
            free_heap.push(b);
    }
    // new blocks for `n` more tokens, plus 1 for a copy-on-write copy
    int64_t needed(const Seq &s, int64_t n) const
    {
        const int64_t bs = block_size;
        int64_t need = (s.tokens + n + bs - 1) / bs - (s.tokens + bs - 1) / bs;
        if (n > 0 && s.tokens % bs != 0 && ref[s.table.back()] > 1)
            ++need;
        return need;
    }
};

extern "C" pa_status pa_bm_create(int num_blocks, int block_size, int max_blocks_per_seq,
                                  pa_block_manager **out)
{
    if (!out || num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
        (int64_t)num_blocks * block_size >= (int64_t(1) << 31))
        return PA_ERR_INVALID_ARG;
    pa_block_manager *bm = new (std::nothrow) pa_block_manager();
    if (!bm)
        return PA_ERR_INVALID_ARG;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->max_blocks_per_seq = max_blocks_per_seq;
    bm->ref.assign(num_blocks, 0);
    std::vector<int32_t> ids(num_blocks);
    for (int b = 0; b < num_blocks; ++b)
        ids[b] = b;
    bm->free_heap = decltype(bm->free_heap)(std::greater<int32_t>(), std::move(ids));
    *out = bm;
    return PA_OK;
}

extern "C" void pa_bm_destroy(pa_block_manager *bm) { delete bm; }

extern "C" int pa_bm_num_free_blocks(const pa_block_manager *bm)
{
    return bm ? (int)bm->free_heap.size() : -1;
}

extern "C" pa_status pa_bm_add_sequence(pa_block_manager *bm, int seq_id)
{
    if (!bm || seq_id < 0 || bm->seqs.count(seq_id))
        return PA_ERR_INVALID_ARG;
    bm->seqs.emplace(seq_id, pa_block_manager::Seq());
    return PA_OK;
}

extern "C" pa_status pa_bm_fork(pa_block_manager *bm, int parent_id, int child_id)
{
    if (!bm || child_id < 0 || bm->seqs.count(child_id))
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq child = it->second;  // copy before inserting
    for (int32_t b : child.table)
        ++bm->ref[b];
    bm->seqs.emplace(child_id, std::move(child));
    return PA_OK;
}

extern "C" int pa_bm_blocks_needed(const pa_block_manager *bm, int seq_id, int num_tokens)
{
    if (!bm || num_tokens < 0)
        return -1;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return -1;
    return (int)bm->needed(it->second, num_tokens);
}

extern "C" pa_status pa_bm_append_tokens(pa_block_manager *bm, int seq_id, int num_tokens,
                                         int32_t *slots, int32_t *cow_pairs, int cow_capacity,
                                         int *num_cow)
{
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !slots) || cow_capacity < 0 || !num_cow)
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq &s = it->second;
    const int64_t bs = bm->block_size;
    *num_cow = 0;
    if ((s.tokens + num_tokens + bs - 1) / bs > bm->max_blocks_per_seq)
        return PA_ERR_TABLE_FULL;
    const bool cow = num_tokens > 0 && s.tokens % bs != 0 && bm->ref[s.table.back()] > 1;
    if (cow && (cow_capacity < 1 || !cow_pairs))
        return PA_ERR_WORKSPACE;
    if (bm->needed(s, num_tokens) > (int64_t)bm->free_heap.size())
        return PA_ERR_OUT_OF_BLOCKS;
    if (cow) {
        const int32_t old = s.table.back();
        const int32_t fresh = bm->take();
        cow_pairs[0] = old;
        cow_pairs[1] = fresh;
        *num_cow = 1;
        --bm->ref[old];  // still named by another table: never reaches 0 here
        s.table.back() = fresh;
    }
    for (int k = 0; k < num_tokens; ++k) {
        const int64_t pos = s.tokens;
        if (pos % bs == 0)
            s.table.push_back(bm->take());
        slots[k] = (int32_t)(s.table[pos / bs] * bs + pos % bs);
        ++s.tokens;
    }
    return PA_OK;
}

extern "C" pa_status pa_bm_append_batch(pa_block_manager *bm, const int32_t *seq_ids,
                                        const int32_t *counts, int n, int32_t *slots,
                                        int32_t *cow_pairs, int cow_capacity, int *num_cow)
{
    if (!bm || n < 0 || !num_cow || cow_capacity < 0 ||
        (n > 0 && (!seq_ids || !counts)))
        return PA_ERR_INVALID_ARG;
    *num_cow = 0;
    // check the whole batch first: the call is all or nothing
    std::unordered_map<int, int> seen;
    // partly filled shared last blocks -> batch sequences appending into them
    std::unordered_map<int32_t, int> sharers;
    int64_t need = 0, total = 0;
    const int64_t bs = bm->block_size;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || counts[i] < 0 || !seen.emplace(seq_ids[i], i).second)
            return PA_ERR_INVALID_ARG;
        const pa_block_manager::Seq &s = it->second;
        if ((s.tokens + counts[i] + bs - 1) / bs > bm->max_blocks_per_seq)
            return PA_ERR_TABLE_FULL;
        need += (s.tokens + counts[i] + bs - 1) / bs - (s.tokens + bs - 1) / bs;
        total += counts[i];
        if (counts[i] > 0 && s.tokens % bs != 0 && bm->ref[s.table.back()] > 1)
            ++sharers[s.table.back()];
    }
    if (total > 0 && !slots)
        return PA_ERR_INVALID_ARG;
    // in batch order, the first ref - 1 appenders into a shared block copy it;
    // if every table naming it appends, the last one writes in place
    int64_t cows = 0;
    for (const auto &kv : sharers)
        cows += std::min<int64_t>(kv.second, bm->ref[kv.first] - 1);
    if (cows > cow_capacity || (cows > 0 && !cow_pairs))
        return PA_ERR_WORKSPACE;
    if (need + cows > (int64_t)bm->free_heap.size())
        return PA_ERR_OUT_OF_BLOCKS;
    int64_t k = 0;
    for (int i = 0; i < n; ++i) {
        int c = 0;
        const pa_status st = pa_bm_append_tokens(bm, seq_ids[i], counts[i], slots + k,
                                                 cow_pairs + 2 * *num_cow,
                                                 cow_capacity - *num_cow, &c);
        if (st != PA_OK)  // not reached: every condition was checked above
            return st;
        *num_cow += c;
        k += counts[i];
    }
    return PA_OK;
}

extern "C" pa_status pa_bm_free_sequence(pa_block_manager *bm, int seq_id)
{
    if (!bm)
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    for (int32_t b : it->second.table)
        bm->release(b);
    bm->seqs.erase(it);
    return PA_OK;
}

extern "C" pa_status pa_bm_sequence_info(const pa_block_manager *bm, int seq_id,
                                         int *num_tokens, int *num_blocks)
{
    if (!bm || !num_tokens || !num_blocks)
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    *num_tokens = (int)it->second.tokens;
    *num_blocks = (int)it->second.table.size();
    return PA_OK;
}

extern "C" pa_status pa_bm_block_table(const pa_block_manager *bm, int seq_id, int32_t *row,
                                       int capacity)
{
    if (!bm || capacity < 0 || (capacity > 0 && !row))
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    const auto &t = it->second.table;
    if ((int64_t)t.size() > capacity)
        return PA_ERR_WORKSPACE;
    std::copy(t.begin(), t.end(), row);
    return PA_OK;
}

extern "C" int pa_bm_ref_count(const pa_block_manager *bm, int block)
{
    if (!bm || block < 0 || block >= bm->num_blocks)
        return -1;
    return bm->ref[block];
}

extern "C" pa_status pa_bm_build_batch(const pa_block_manager *bm, const int32_t *seq_ids, int n,
                                       int32_t *block_tables, int max_blocks,
                                       int32_t *context_lens, int32_t pad_block)
{
    if (!bm || n < 0 || max_blocks <= 0 ||
        (n > 0 && (!seq_ids || !block_tables || !context_lens)))
        return PA_ERR_INVALID_ARG;
    // check everything first: a failing call writes nothing
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end())
            return PA_ERR_INVALID_ARG;
        if ((int64_t)it->second.table.size() > max_blocks)
            return PA_ERR_WORKSPACE;
    }
    for (int i = 0; i < n; ++i) {
        const auto &s = bm->seqs.find(seq_ids[i])->second;
        int32_t *row = block_tables + (size_t)i * max_blocks;
        std::copy(s.table.begin(), s.table.end(), row);
        std::fill(row + s.table.size(), row + max_blocks, pad_block);
        context_lens[i] = (int32_t)s.tokens;
    }
    return PA_OK;
}
