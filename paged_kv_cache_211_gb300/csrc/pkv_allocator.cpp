// pkv_allocator.cpp -- host block allocator of the paged KV cache.
//
// "micro-vLLM" wiki, execution chain: the KVCacheManager hands out and takes
// back physical blocks and keeps the prefix cache; "从零手写 vLLM 核心：
// mini-vllm 项目深度解析" §2: 16-token blocks are allocated and released on
// demand, shared between sequences (prefix cache, parallel sampling), and
// admission control keeps the engine correct when only a few blocks are
// left.  Here a block is free (count 0) or referenced by one or more
// sequences; allocation is all-or-nothing so that a scheduler can refuse a
// request without rolling anything back.
#include <cstdint>
#include <new>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_allocator {
    std::vector<int32_t> free_ids;  // stack; the next id handed out is at the back
    std::vector<int32_t> refs;      // reference count per block
};

extern "C" {

pkv_status paged_kv_alloc_create(int num_blocks, pkv_allocator** out) {
    if (!out || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    pkv_allocator* a = new (std::nothrow) pkv_allocator;
    if (!a) return PKV_ERR_INVALID_ARG;
    try {
        a->refs.assign((size_t)num_blocks, 0);
        a->free_ids.resize((size_t)num_blocks);
    } catch (...) {
        delete a;
        return PKV_ERR_INVALID_ARG;
    }
    // lowest ids first: block 0 is handed out first
    for (int i = 0; i < num_blocks; ++i) a->free_ids[(size_t)i] = num_blocks - 1 - i;
    *out = a;
    return PKV_OK;
}

void paged_kv_alloc_destroy(pkv_allocator* a) { delete a; }

pkv_status paged_kv_alloc(pkv_allocator* a, int n, int32_t* out_block_ids) {
    if (!a || n < 0 || (n > 0 && !out_block_ids)) return PKV_ERR_INVALID_ARG;
    if ((size_t)n > a->free_ids.size()) return PKV_ERR_NO_BLOCKS;
    for (int i = 0; i < n; ++i) {
        const int32_t id = a->free_ids.back();
        a->free_ids.pop_back();
        a->refs[(size_t)id] = 1;
        out_block_ids[i] = id;
    }
    return PKV_OK;
}

static bool all_allocated(const pkv_allocator* a, int n, const int32_t* ids) {
    for (int i = 0; i < n; ++i) {
        const int32_t id = ids[i];
        if (id < 0 || (size_t)id >= a->refs.size() || a->refs[(size_t)id] <= 0) return false;
    }
    return true;
}

pkv_status paged_kv_share(pkv_allocator* a, int n, const int32_t* block_ids) {
    if (!a || n < 0 || (n > 0 && !block_ids)) return PKV_ERR_INVALID_ARG;
    if (!all_allocated(a, n, block_ids)) return PKV_ERR_BAD_BLOCK_ID;
    for (int i = 0; i < n; ++i) ++a->refs[(size_t)block_ids[i]];
    return PKV_OK;
}

pkv_status paged_kv_free(pkv_allocator* a, int n, const int32_t* block_ids) {
    if (!a || n < 0 || (n > 0 && !block_ids)) return PKV_ERR_INVALID_ARG;
    if (!all_allocated(a, n, block_ids)) return PKV_ERR_BAD_BLOCK_ID;
    // a list that names one block more often than it is referenced would drive
    // its count below zero: refuse it as a whole
    std::vector<int32_t> drop;
    drop.reserve((size_t)n);
    for (int i = 0; i < n; ++i) drop.push_back(block_ids[i]);
    std::vector<int32_t> seen(a->refs.size(), 0);
    for (int32_t id : drop)
        if (++seen[(size_t)id] > a->refs[(size_t)id]) return PKV_ERR_BAD_BLOCK_ID;
    for (int32_t id : drop) {
        if (--a->refs[(size_t)id] == 0) a->free_ids.push_back(id);
    }
    return PKV_OK;
}

int paged_kv_num_free(const pkv_allocator* a) { return a ? (int)a->free_ids.size() : 0; }

int paged_kv_refcount(const pkv_allocator* a, int32_t block_id) {
    if (!a || block_id < 0 || (size_t)block_id >= a->refs.size()) return -1;
    return a->refs[(size_t)block_id];
}

}  // extern "C"
