// Host block allocator: free list, reference counts and copy-on-write.
//
// Bookkeeping follows the PagedAttention pages: blocks are handed out from a
// free list and reported exhausted when it is empty ("PagedAttention:
// virtual memory for the KV cache", scheduler sketch); a block carries a
// reference count, freeing walks a sequence's table in reverse and returns a
// block whose count reaches zero to the head of the list ("01 ·
// PagedAttention 与 KV cache 块管理" §3, §4.3); a write into a block whose
// count is above one first clones it ("4. PagedAttention原理（下）" §4.3);
// slots are table[pos / B] * B + pos % B (vLLM book chapter 4, §4.4.3).
//
// It only builds inputs (block tables, slot mappings, COW pairs) for the
// device calls; it never touches device memory.
#include <cstdint>
#include <deque>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

struct pa_allocator {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;        // head = front
    std::vector<int32_t> ref;
    struct Seq {
        std::vector<int32_t> table;
        int32_t len = 0;
    };
    std::unordered_map<int, Seq> seqs;
    int next_id = 0;

    int32_t take()
    {
        int32_t b = free_list.front();
        free_list.pop_front();
        ref[b] = 1;
        return b;
    }
    void release(int32_t b)
    {
        if (--ref[b] == 0)
            free_list.push_front(b);
    }
};

using pa::set_error;

extern "C" pa_allocator *pa_alloc_create(int num_blocks, int block_size, const int32_t *order)
{
    if (num_blocks <= 0 || block_size <= 0) {
        set_error(PA_ERR_INVALID_ARG, "pa_alloc_create: num_blocks and block_size must be > 0");
        return nullptr;
    }
    auto *a = new pa_allocator();
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
        int32_t b = order ? order[i] : i;
        if (b < 0 || b >= num_blocks || seen[b]) {
            delete a;
            set_error(PA_ERR_INVALID_ARG, "pa_alloc_create: order must list each block once");
            return nullptr;
        }
        seen[b] = 1;
        a->free_list.push_back(b);
    }
    return a;
}

extern "C" void pa_alloc_destroy(pa_allocator *a) { delete a; }

extern "C" int pa_alloc_num_free(const pa_allocator *a)
{
    if (!a)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_num_free: null allocator");
    return (int)a->free_list.size();
}

extern "C" int pa_alloc_ref_count(const pa_allocator *a, int block)
{
    if (!a || block < 0 || block >= a->num_blocks)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_ref_count: bad allocator or block %d", block);
    return a->ref[block];
}

extern "C" int pa_alloc_add_seq(pa_allocator *a, int num_tokens, int *seq_id)
{
    if (!a || !seq_id || num_tokens < 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_add_seq: bad arguments");
    long long need = ((long long)num_tokens + a->block_size - 1) / a->block_size;
    if (need > (long long)a->free_list.size())
        return set_error(PA_ERR_OUT_OF_BLOCKS, "pa_alloc_add_seq: need %lld blocks, %zu free",
                         need, a->free_list.size());
    pa_allocator::Seq s;
    s.table.reserve((size_t)need);
    for (long long i = 0; i < need; ++i)
        s.table.push_back(a->take());
    s.len = num_tokens;
    *seq_id = a->next_id++;
    a->seqs.emplace(*seq_id, std::move(s));
    return PA_OK;
}

extern "C" int pa_alloc_fork(pa_allocator *a, int parent, int *child)
{
    if (!a || !child)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_fork: bad arguments");
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end())
        return set_error(PA_ERR_NOT_FOUND, "pa_alloc_fork: unknown sequence %d", parent);
    pa_allocator::Seq s = it->second;
    for (int32_t b : s.table)
        ++a->ref[b];
    *child = a->next_id++;
    a->seqs.emplace(*child, std::move(s));
    return PA_OK;
}

extern "C" int pa_alloc_append_token(pa_allocator *a, int seq_id, int32_t *slot,
                                     int32_t *cow_src, int32_t *cow_dst)
{
    if (!a || !slot || !cow_src || !cow_dst)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_append_token: bad arguments");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end())
        return set_error(PA_ERR_NOT_FOUND, "pa_alloc_append_token: unknown sequence %d", seq_id);
    pa_allocator::Seq &s = it->second;
    const int32_t pos = s.len;
    const int B = a->block_size;
    *cow_src = *cow_dst = -1;
    if (pos % B == 0) {
        if (a->free_list.empty())
            return set_error(PA_ERR_OUT_OF_BLOCKS, "pa_alloc_append_token: no free block");
        s.table.push_back(a->take());
    } else {
        int32_t last = s.table.back();
        if (a->ref[last] > 1) {
            if (a->free_list.empty())
                return set_error(PA_ERR_OUT_OF_BLOCKS, "pa_alloc_append_token: no free block for COW");
            int32_t fresh = a->take();
            --a->ref[last];
            s.table.back() = fresh;
            *cow_src = last;
            *cow_dst = fresh;
        }
    }
    s.len = pos + 1;
    *slot = s.table[pos / B] * B + pos % B;
    return PA_OK;
}

extern "C" int pa_alloc_free_seq(pa_allocator *a, int seq_id)
{
    if (!a)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_free_seq: null allocator");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end())
        return set_error(PA_ERR_NOT_FOUND, "pa_alloc_free_seq: unknown sequence %d", seq_id);
    const std::vector<int32_t> &t = it->second.table;
    for (auto b = t.rbegin(); b != t.rend(); ++b)
        a->release(*b);
    a->seqs.erase(it);
    return PA_OK;
}

extern "C" int pa_alloc_seq_len(const pa_allocator *a, int seq_id)
{
    if (!a)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_seq_len: null allocator");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end())
        return set_error(PA_ERR_NOT_FOUND, "pa_alloc_seq_len: unknown sequence %d", seq_id);
    return it->second.len;
}

extern "C" int pa_alloc_seq_num_blocks(const pa_allocator *a, int seq_id)
{
    if (!a)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_seq_num_blocks: null allocator");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end())
        return set_error(PA_ERR_NOT_FOUND, "pa_alloc_seq_num_blocks: unknown sequence %d", seq_id);
    return (int)it->second.table.size();
}

extern "C" int pa_alloc_block_tables(const pa_allocator *a, const int *seq_ids, int n,
                                     int max_blocks_per_seq, int32_t *out)
{
    if (!a || (n > 0 && (!seq_ids || !out)) || n < 0 || max_blocks_per_seq < 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_block_tables: bad arguments");
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end())
            return set_error(PA_ERR_NOT_FOUND, "pa_alloc_block_tables: unknown sequence %d", seq_ids[i]);
        const std::vector<int32_t> &t = it->second.table;
        if ((int)t.size() > max_blocks_per_seq)
            return set_error(PA_ERR_INVALID_ARG, "pa_alloc_block_tables: sequence %d has %zu blocks > %d",
                             seq_ids[i], t.size(), max_blocks_per_seq);
        int32_t *row = out + (size_t)i * max_blocks_per_seq;
        for (int j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < (int)t.size() ? t[j] : -1;
    }
    return PA_OK;
}

extern "C" int pa_alloc_seq_lens(const pa_allocator *a, const int *seq_ids, int n, int32_t *out)
{
    if (!a || (n > 0 && (!seq_ids || !out)) || n < 0)
        return set_error(PA_ERR_INVALID_ARG, "pa_alloc_seq_lens: bad arguments");
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end())
            return set_error(PA_ERR_NOT_FOUND, "pa_alloc_seq_lens: unknown sequence %d", seq_ids[i]);
        out[i] = it->second.len;
    }
    return PA_OK;
}
