// Host-side KV block allocator: the CPU "block manager" that hands out
// fixed-size cache blocks ("Nano-vLLM Part 2" page, section 05: the control
// plane tracks block allocation and reference counts in CPU memory; "Tokenizer,
// KV Cache and RoPE" page, section 5: pages of 16 tokens allocated on demand,
// freed pages reused, allocation failures counted).
//
// A LIFO stack of free ids (a freed block is the next one handed out, which
// keeps recently touched blocks warm) plus one reference count per block.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "kvattn.h"

struct kvattn_allocator {
    std::mutex mu;
    std::vector<int32_t> free_ids;   // stack; back() is handed out next
    std::vector<int32_t> refs;       // 0 = free
    int64_t failures = 0;
};

// Removes the ids whose refcount was just set from the free stack (one pass).
static void compact_free_stack(kvattn_allocator* a)
{
    size_t w = 0;
    for (size_t r = 0; r < a->free_ids.size(); ++r)
        if (a->refs[(size_t)a->free_ids[r]] == 0) a->free_ids[w++] = a->free_ids[r];
    a->free_ids.resize(w);
}

extern "C" {

kvattn_status kvattn_allocator_create(int64_t num_blocks, kvattn_allocator** out)
{
    if (!out || num_blocks <= 0 || num_blocks > INT32_MAX) return KVATTN_ERR_INVALID_ARG;
    *out = nullptr;
    kvattn_allocator* a = new (std::nothrow) kvattn_allocator();
    if (!a) return KVATTN_ERR_INVALID_ARG;
    try {
        a->refs.assign((size_t)num_blocks, 0);
        a->free_ids.resize((size_t)num_blocks);
    } catch (...) {
        delete a;
        return KVATTN_ERR_INVALID_ARG;
    }
    // lowest id on top of the stack
    for (int64_t i = 0; i < num_blocks; ++i) a->free_ids[(size_t)i] = (int32_t)(num_blocks - 1 - i);
    *out = a;
    return KVATTN_OK;
}

void kvattn_allocator_destroy(kvattn_allocator* a) { delete a; }

kvattn_status kvattn_alloc_blocks(kvattn_allocator* a, int32_t n, int32_t* out_ids)
{
    if (!a || n < 0 || (n > 0 && !out_ids)) return KVATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    if ((size_t)n > a->free_ids.size()) {
        ++a->failures;
        return KVATTN_ERR_OUT_OF_BLOCKS;
    }
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = a->free_ids.back();
        a->free_ids.pop_back();
        a->refs[(size_t)id] = 1;
        out_ids[i] = id;
    }
    return KVATTN_OK;
}

// Validates that every id can lose one reference, counting repeats.
static bool can_release(kvattn_allocator* a, const int32_t* ids, int32_t n)
{
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (id < 0 || (size_t)id >= a->refs.size() || a->refs[(size_t)id] <= 0) return false;
    }
    // count multiplicities without touching the shared state
    std::vector<int32_t> sorted(ids, ids + n);
    std::sort(sorted.begin(), sorted.end());
    for (int32_t i = 0; i < n;) {
        int32_t j = i;
        while (j < n && sorted[(size_t)j] == sorted[(size_t)i]) ++j;
        if (j - i > a->refs[(size_t)sorted[(size_t)i]]) return false;
        i = j;
    }
    return true;
}

kvattn_status kvattn_free_blocks(kvattn_allocator* a, const int32_t* ids, int32_t n)
{
    if (!a || n < 0 || (n > 0 && !ids)) return KVATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    if (!can_release(a, ids, n)) return KVATTN_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        int32_t& r = a->refs[(size_t)ids[i]];
        if (--r == 0) a->free_ids.push_back(ids[i]);
    }
    return KVATTN_OK;
}

kvattn_status kvattn_claim_blocks(kvattn_allocator* a, const int32_t* ids, int32_t n)
{
    if (!a || n < 0 || (n > 0 && !ids)) return KVATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    std::vector<int32_t> sorted(ids, ids + n);
    std::sort(sorted.begin(), sorted.end());
    for (int32_t i = 0; i < n; ++i) {
        const int32_t id = sorted[(size_t)i];
        if (id < 0 || (size_t)id >= a->refs.size() || a->refs[(size_t)id] != 0) return KVATTN_ERR_INVALID_ARG;
        if (i > 0 && sorted[(size_t)i - 1] == id) return KVATTN_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) a->refs[(size_t)ids[i]] = 1;
    if (n > 0) compact_free_stack(a);
    return KVATTN_OK;
}

kvattn_status kvattn_share_blocks(kvattn_allocator* a, const int32_t* ids, int32_t n)
{
    if (!a || n < 0 || (n > 0 && !ids)) return KVATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (id < 0 || (size_t)id >= a->refs.size() || a->refs[(size_t)id] <= 0)
            return KVATTN_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) ++a->refs[(size_t)ids[i]];
    return KVATTN_OK;
}

int64_t kvattn_allocator_num_free(const kvattn_allocator* a)
{
    if (!a) return -1;
    auto* m = const_cast<kvattn_allocator*>(a);
    std::lock_guard<std::mutex> g(m->mu);
    return (int64_t)a->free_ids.size();
}

int64_t kvattn_allocator_num_failures(const kvattn_allocator* a)
{
    if (!a) return -1;
    auto* m = const_cast<kvattn_allocator*>(a);
    std::lock_guard<std::mutex> g(m->mu);
    return a->failures;
}

int32_t kvattn_allocator_refcount(const kvattn_allocator* a, int32_t id)
{
    if (!a || id < 0 || (size_t)id >= a->refs.size()) return -1;
    auto* m = const_cast<kvattn_allocator*>(a);
    std::lock_guard<std::mutex> g(m->mu);
    return a->refs[(size_t)id];
}

static int32_t blocks_for(int32_t len, int32_t bs) { return len <= 0 ? 0 : (len + bs - 1) / bs; }

kvattn_status kvattn_table_grow(kvattn_allocator* a, int32_t* table_row, int32_t max_blocks,
                                int32_t block_size, int32_t cur_len, int32_t new_len)
{
    if (!a || !table_row || max_blocks <= 0 || block_size <= 0 || cur_len < 0 || new_len < cur_len)
        return KVATTN_ERR_INVALID_ARG;
    int32_t have = blocks_for(cur_len, block_size), need = blocks_for(new_len, block_size);
    if (need > max_blocks) return KVATTN_ERR_INVALID_ARG;
    if (need == have) return KVATTN_OK;
    return kvattn_alloc_blocks(a, need - have, table_row + have);
}

kvattn_status kvattn_table_release(kvattn_allocator* a, int32_t* table_row, int32_t max_blocks,
                                   int32_t block_size, int32_t len)
{
    if (!a || !table_row || max_blocks <= 0 || block_size <= 0 || len < 0)
        return KVATTN_ERR_INVALID_ARG;
    int32_t have = blocks_for(len, block_size);
    if (have > max_blocks) return KVATTN_ERR_INVALID_ARG;
    kvattn_status s = kvattn_free_blocks(a, table_row, have);
    if (s != KVATTN_OK) return s;
    for (int32_t i = 0; i < have; ++i) table_row[i] = -1;
    return KVATTN_OK;
}

kvattn_status kvattn_table_fork(kvattn_allocator* a, const int32_t* src_row, int32_t* dst_row,
                                int32_t max_blocks, int32_t block_size, int32_t len)
{
    if (!a || !src_row || !dst_row || max_blocks <= 0 || block_size <= 0 || len < 0)
        return KVATTN_ERR_INVALID_ARG;
    const int32_t have = blocks_for(len, block_size);
    if (have > max_blocks) return KVATTN_ERR_INVALID_ARG;
    kvattn_status s = kvattn_share_blocks(a, src_row, have);
    if (s != KVATTN_OK) return s;
    std::copy(src_row, src_row + have, dst_row);
    return KVATTN_OK;
}

kvattn_status kvattn_table_prepare_append(kvattn_allocator* a, int32_t* table_row, int32_t max_blocks,
                                          int32_t block_size, int32_t cur_len, int32_t new_len,
                                          int32_t* cow_src, int32_t* cow_dst)
{
    if (!a || !table_row || !cow_src || !cow_dst || max_blocks <= 0 || block_size <= 0 || cur_len < 0 ||
        new_len < cur_len)
        return KVATTN_ERR_INVALID_ARG;
    const int32_t have = blocks_for(cur_len, block_size), need = blocks_for(new_len, block_size);
    if (need > max_blocks) return KVATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    // the partially filled block the first new token lands in, if any
    const bool partial = new_len > cur_len && cur_len % block_size != 0;
    int32_t old = -1;
    if (partial) {
        old = table_row[have - 1];
        if (old < 0 || (size_t)old >= a->refs.size() || a->refs[(size_t)old] <= 0) return KVATTN_ERR_INVALID_ARG;
    }
    const bool cow = partial && a->refs[(size_t)old] > 1;
    const size_t want = (size_t)(need - have) + (cow ? 1 : 0);
    if (want > a->free_ids.size()) {
        ++a->failures;
        return KVATTN_ERR_OUT_OF_BLOCKS;
    }
    auto take = [&]() {
        const int32_t id = a->free_ids.back();
        a->free_ids.pop_back();
        a->refs[(size_t)id] = 1;
        return id;
    };
    *cow_src = *cow_dst = -1;
    if (cow) {
        const int32_t fresh = take();
        --a->refs[(size_t)old];   // still >= 1: another sequence holds it
        table_row[have - 1] = fresh;
        *cow_src = old;
        *cow_dst = fresh;
    }
    for (int32_t b = have; b < need; ++b) table_row[b] = take();
    return KVATTN_OK;
}

}  // extern "C"
