// pkv_allocator.cpp -- host block allocator of the paged KV cache, with a
// hash-indexed prefix cache, copy-on-write and rollback.
//
// "micro-vLLM" wiki, execution chain: the KVCacheManager hands out and takes
// back physical blocks and keeps the prefix cache; "从零手写 vLLM 核心：
// mini-vllm 项目深度解析" §2: 16-token blocks are allocated and released on
// demand, shared between sequences (prefix cache, parallel sampling), and
// admission control keeps the engine correct when only a few blocks are
// left; §工程启示: the KV cache can be rolled back (speculative decoding).
//
// Block states:
//   free       count 0, no cached content          -> on the free stack
//   cached     count 0, content registered by hash -> on the LRU list
//   live       count >= 1 (possibly also registered by hash)
// Allocation takes free blocks first, then evicts cached blocks oldest
// first; it is all-or-nothing, so a scheduler can refuse a request without
// rolling anything back.
#include <cstdint>
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_allocator {
    std::vector<int32_t> free_ids;  // stack; the next id handed out is at the back
    std::vector<int32_t> refs;      // reference count per block
    std::unordered_map<uint64_t, int32_t> by_hash;
    std::vector<uint64_t> hash_of;
    std::vector<uint8_t> has_hash;
    std::list<int32_t> lru;  // cached blocks with count 0, oldest first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<uint8_t> in_lru;
};

namespace {

bool valid_id(const pkv_allocator* a, int32_t id) {
    return id >= 0 && (size_t)id < a->refs.size();
}

void unregister(pkv_allocator* a, int32_t b) {
    if (!a->has_hash[(size_t)b]) return;
    auto it = a->by_hash.find(a->hash_of[(size_t)b]);
    if (it != a->by_hash.end() && it->second == b) a->by_hash.erase(it);
    a->has_hash[(size_t)b] = 0;
}

void lru_remove(pkv_allocator* a, int32_t b) {
    if (!a->in_lru[(size_t)b]) return;
    a->lru.erase(a->lru_pos[(size_t)b]);
    a->in_lru[(size_t)b] = 0;
}

// One block for a new owner (count 1): a free one, else the oldest cached.
int32_t take_one(pkv_allocator* a) {
    int32_t id;
    if (!a->free_ids.empty()) {
        id = a->free_ids.back();
        a->free_ids.pop_back();
    } else {
        id = a->lru.front();
        lru_remove(a, id);
        unregister(a, id);  // its content is about to be overwritten
    }
    a->refs[(size_t)id] = 1;
    return id;
}

// Drops one reference; at zero the block is cached (if registered) or freed.
void drop_one(pkv_allocator* a, int32_t b) {
    if (--a->refs[(size_t)b] > 0) return;
    if (a->has_hash[(size_t)b]) {
        a->lru.push_back(b);
        a->lru_pos[(size_t)b] = std::prev(a->lru.end());
        a->in_lru[(size_t)b] = 1;
    } else {
        a->free_ids.push_back(b);
    }
}

bool all_live(const pkv_allocator* a, int n, const int32_t* ids) {
    for (int i = 0; i < n; ++i)
        if (!valid_id(a, ids[i]) || a->refs[(size_t)ids[i]] <= 0) return false;
    return true;
}

// Every id live, and none named more often than it is referenced: dropping
// one reference per entry then leaves every count >= 0.
bool droppable(const pkv_allocator* a, int n, const int32_t* ids) {
    if (!all_live(a, n, ids)) return false;
    std::unordered_map<int32_t, int> seen;
    for (int i = 0; i < n; ++i)
        if (++seen[ids[i]] > a->refs[(size_t)ids[i]]) return false;
    return true;
}

// splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", 2014): a bijective 64-bit mixer.
uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

}  // namespace

extern "C" {

pkv_status paged_kv_alloc_create(int num_blocks, pkv_allocator** out) {
    if (!out || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    pkv_allocator* a = new (std::nothrow) pkv_allocator;
    if (!a) return PKV_ERR_INVALID_ARG;
    try {
        const size_t n = (size_t)num_blocks;
        a->refs.assign(n, 0);
        a->free_ids.resize(n);
        a->hash_of.assign(n, 0);
        a->has_hash.assign(n, 0);
        a->lru_pos.resize(n);
        a->in_lru.assign(n, 0);
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
    if ((size_t)n > a->free_ids.size() + a->lru.size()) return PKV_ERR_NO_BLOCKS;
    for (int i = 0; i < n; ++i) out_block_ids[i] = take_one(a);
    return PKV_OK;
}

pkv_status paged_kv_share(pkv_allocator* a, int n, const int32_t* block_ids) {
    if (!a || n < 0 || (n > 0 && !block_ids)) return PKV_ERR_INVALID_ARG;
    if (!all_live(a, n, block_ids)) return PKV_ERR_BAD_BLOCK_ID;
    for (int i = 0; i < n; ++i) ++a->refs[(size_t)block_ids[i]];
    return PKV_OK;
}

pkv_status paged_kv_free(pkv_allocator* a, int n, const int32_t* block_ids) {
    if (!a || n < 0 || (n > 0 && !block_ids)) return PKV_ERR_INVALID_ARG;
    // a list that names one block more often than it is referenced would drive
    // its count below zero: refuse it as a whole
    if (!droppable(a, n, block_ids)) return PKV_ERR_BAD_BLOCK_ID;
    for (int i = 0; i < n; ++i) drop_one(a, block_ids[i]);
    return PKV_OK;
}

int paged_kv_num_free(const pkv_allocator* a) {
    return a ? (int)(a->free_ids.size() + a->lru.size()) : 0;
}

int paged_kv_num_cached(const pkv_allocator* a) { return a ? (int)a->by_hash.size() : 0; }

int paged_kv_refcount(const pkv_allocator* a, int32_t block_id) {
    if (!a || !valid_id(a, block_id)) return -1;
    return a->refs[(size_t)block_id];
}

uint64_t paged_kv_block_hash(uint64_t parent_hash, const int32_t* tokens, int num_tokens) {
    uint64_t h = mix64(parent_hash ^ 0x9e3779b97f4a7c15ull);
    for (int i = 0; i < num_tokens; ++i)
        h = mix64(h + (uint64_t)(uint32_t)tokens[i] + 0x9e3779b97f4a7c15ull * (uint64_t)(i + 1));
    return mix64(h ^ (uint64_t)num_tokens);
}

pkv_status paged_kv_prefix_insert(pkv_allocator* a, int32_t block_id, uint64_t hash) {
    if (!a || !valid_id(a, block_id) || a->refs[(size_t)block_id] <= 0) return PKV_ERR_BAD_BLOCK_ID;
    if (a->has_hash[(size_t)block_id]) {
        return a->hash_of[(size_t)block_id] == hash ? PKV_OK : PKV_ERR_INVALID_ARG;
    }
    if (a->by_hash.count(hash)) return PKV_OK;  // another block already holds this content
    a->by_hash.emplace(hash, block_id);
    a->hash_of[(size_t)block_id] = hash;
    a->has_hash[(size_t)block_id] = 1;
    return PKV_OK;
}

pkv_status paged_kv_prefix_lookup(pkv_allocator* a, int n, const uint64_t* hashes,
                                  int32_t* out_block_ids, int* num_hits) {
    if (!a || n < 0 || !num_hits || (n > 0 && (!hashes || !out_block_ids)))
        return PKV_ERR_INVALID_ARG;
    int i = 0;
    for (; i < n; ++i) {
        auto it = a->by_hash.find(hashes[i]);
        if (it == a->by_hash.end()) break;
        const int32_t b = it->second;
        if (a->refs[(size_t)b] == 0) lru_remove(a, b);
        ++a->refs[(size_t)b];
        out_block_ids[i] = b;
    }
    *num_hits = i;
    return PKV_OK;
}

pkv_status paged_kv_cow(pkv_allocator* a, int32_t block_id, int32_t* out_block_id,
                        int* needs_copy) {
    if (!a || !out_block_id || !needs_copy) return PKV_ERR_INVALID_ARG;
    if (!valid_id(a, block_id) || a->refs[(size_t)block_id] <= 0) return PKV_ERR_BAD_BLOCK_ID;
    if (a->refs[(size_t)block_id] == 1) {
        unregister(a, block_id);  // its content is about to change
        *out_block_id = block_id;
        *needs_copy = 0;
        return PKV_OK;
    }
    if (a->free_ids.empty() && a->lru.empty()) return PKV_ERR_NO_BLOCKS;
    const int32_t fresh = take_one(a);
    --a->refs[(size_t)block_id];  // still >= 1: others keep the original
    *out_block_id = fresh;
    *needs_copy = 1;
    return PKV_OK;
}

pkv_status paged_kv_rollback(pkv_allocator* a, int32_t* block_table, int num_table_blocks,
                             int new_len, int* new_num_blocks) {
    if (!a || !new_num_blocks || num_table_blocks < 0 || new_len < 0 ||
        (num_table_blocks > 0 && !block_table))
        return PKV_ERR_INVALID_ARG;
    // blocks that hold new_len tokens (no overflow near INT_MAX)
    const int keep = new_len / PKV_BLOCK_SIZE + (new_len % PKV_BLOCK_SIZE != 0 ? 1 : 0);
    if (keep > num_table_blocks) return PKV_ERR_INVALID_ARG;
    if (!droppable(a, num_table_blocks - keep, block_table + keep)) return PKV_ERR_BAD_BLOCK_ID;
    for (int i = keep; i < num_table_blocks; ++i) {
        drop_one(a, block_table[i]);
        block_table[i] = -1;
    }
    // a now-partial last block no longer holds the full block its hash named
    if (keep > 0 && new_len % PKV_BLOCK_SIZE != 0) {
        const int32_t last = block_table[keep - 1];
        if (valid_id(a, last) && a->refs[(size_t)last] == 1) unregister(a, last);
    }
    *new_num_blocks = keep;
    return PKV_OK;
}

}  // extern "C"
