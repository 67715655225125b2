// Prefix cache: reuse of already computed KV blocks for a common prompt
// prefix.
//
// "PagedAttention Nedir?", section "Prefix Sharing Nasil Calisir?": when
// requests start with the same tokens, the KV of that common part can be
// reused instead of recomputed; matching must be exact (same tokens and same
// preceding context, not mere similarity), and vLLM's prefix caching keys
// each block by its contents together with the context before it.  The gain
// is in prefill; the blocks must still be resident.
//
// Key of full block i of a sequence: a 64-bit mix of the key of block i-1 and
// the block's token ids.  The entry also keeps the parent key and the tokens,
// so a lookup compares them exactly: a hash collision can never produce a
// false match.  Only full blocks are cached (a partial block still grows).
//
// References: the cache holds one reference (allocator refcount) on every
// block it lists; a match adds one for the caller.  Blocks whose only
// reference is the cache's are evictable, least recently used first.
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "paged_kv.h"

namespace {

// 64-bit mixing of a parent key and a block of token ids (splitmix-style
// finalisers between words).
uint64_t mix(uint64_t h) {
    h ^= h >> 30;
    h *= 0xbf58476d1ce4e5b9ull;
    h ^= h >> 27;
    h *= 0x94d049bb133111ebull;
    h ^= h >> 31;
    return h;
}

uint64_t block_key(uint64_t parent, const int32_t *tokens, int n) {
    uint64_t h = mix(parent ^ 0x9e3779b97f4a7c15ull);
    for (int i = 0; i < n; ++i) h = mix(h ^ (uint64_t)(uint32_t)tokens[i] ^ ((uint64_t)i << 40));
    return h;
}

struct Entry {
    int32_t block;
    uint64_t parent;
    std::vector<int32_t> tokens;
    std::list<uint64_t>::iterator lru;  // position in the recency list
};

}  // namespace

struct kv_prefix_cache {
    kv_allocator_t alloc = nullptr;
    int block_size = 16;
    int capacity = 0;
    std::unordered_map<uint64_t, Entry> map;
    std::list<uint64_t> lru;  // front = most recently used
    long long hits = 0, lookups = 0;
};

extern "C" {

kv_status kv_prefix_cache_create(kv_allocator_t a, int block_size, int capacity_blocks,
                                 kv_prefix_cache_t *out) {
    if (!a || !out || block_size <= 0 || capacity_blocks < 0) return KV_ERR_ARG;
    kv_prefix_cache *c = new (std::nothrow) kv_prefix_cache();
    if (!c) return KV_ERR_OOM;
    c->alloc = a;
    c->block_size = block_size;
    c->capacity = capacity_blocks;
    *out = c;
    return KV_OK;
}

kv_status kv_prefix_cache_destroy(kv_prefix_cache_t c) {
    if (!c) return KV_ERR_ARG;
    for (auto &kv : c->map) kv_allocator_free(c->alloc, 1, &kv.second.block);
    delete c;
    return KV_OK;
}

kv_status kv_prefix_cache_match(kv_prefix_cache_t c, const int32_t *tokens, int64_t n_tokens,
                                int32_t *blocks_out, int max_blocks, int *n_matched) {
    if (!c || n_tokens < 0 || !n_matched || max_blocks < 0 || (n_tokens > 0 && !tokens) ||
        (max_blocks > 0 && !blocks_out))
        return KV_ERR_ARG;
    const int bs = c->block_size;
    const int64_t full = n_tokens / bs;
    uint64_t parent = 0;
    int n = 0;
    std::vector<int32_t> found;
    for (int64_t i = 0; i < full && n < max_blocks; ++i) {
        const int32_t *blk = tokens + i * bs;
        const uint64_t key = block_key(parent, blk, bs);
        auto it = c->map.find(key);
        if (it == c->map.end() || it->second.parent != parent ||
            std::memcmp(it->second.tokens.data(), blk, sizeof(int32_t) * bs) != 0)
            break;
        found.push_back(it->second.block);
        c->lru.splice(c->lru.begin(), c->lru, it->second.lru);  // most recently used
        parent = key;
        ++n;
    }
    if (n > 0 && kv_allocator_share(c->alloc, n, found.data()) != KV_OK) return KV_ERR_STATE;
    for (int i = 0; i < n; ++i) blocks_out[i] = found[i];
    c->lookups += 1;
    c->hits += n > 0;
    *n_matched = n;
    return KV_OK;
}

kv_status kv_prefix_cache_insert(kv_prefix_cache_t c, const int32_t *tokens, int64_t n_tokens,
                                 const int32_t *blocks, int n_blocks, int *n_inserted) {
    if (!c || n_tokens < 0 || n_blocks < 0 || (n_tokens > 0 && !tokens) ||
        (n_blocks > 0 && !blocks))
        return KV_ERR_ARG;
    const int bs = c->block_size;
    int64_t full = n_tokens / bs;
    if (full > n_blocks) full = n_blocks;
    uint64_t parent = 0;
    int added = 0;
    for (int64_t i = 0; i < full; ++i) {
        const int32_t *blk = tokens + i * bs;
        const uint64_t key = block_key(parent, blk, bs);
        auto it = c->map.find(key);
        if (it != c->map.end()) {
            if (it->second.parent != parent ||
                std::memcmp(it->second.tokens.data(), blk, sizeof(int32_t) * bs) != 0)
                break;  // a different block hashes here: stop rather than alias
            parent = key;  // already cached (possibly another physical copy): keep the old one
            continue;
        }
        if ((int)c->map.size() >= c->capacity) {
            int freed = 0;
            kv_prefix_cache_evict(c, 1, &freed);
            if ((int)c->map.size() >= c->capacity) break;  // nothing evictable: stop caching
        }
        if (kv_allocator_share(c->alloc, 1, blocks + i) != KV_OK) return KV_ERR_ARG;
        c->lru.push_front(key);
        Entry e;
        e.block = blocks[i];
        e.parent = parent;
        e.tokens.assign(blk, blk + bs);
        e.lru = c->lru.begin();
        c->map.emplace(key, std::move(e));
        parent = key;
        ++added;
    }
    if (n_inserted) *n_inserted = added;
    return KV_OK;
}

kv_status kv_prefix_cache_evict(kv_prefix_cache_t c, int n_blocks, int *n_freed) {
    if (!c || n_blocks < 0 || !n_freed) return KV_ERR_ARG;
    int freed = 0;
    // Least recently used first; only blocks nobody but the cache holds.
    for (auto it = c->lru.end(); it != c->lru.begin() && freed < n_blocks;) {
        --it;
        auto e = c->map.find(*it);
        int rc = 0;
        kv_allocator_refcount(c->alloc, e->second.block, &rc);
        if (rc != 1) continue;
        kv_allocator_free(c->alloc, 1, &e->second.block);
        c->map.erase(e);
        it = c->lru.erase(it);
        ++freed;
    }
    *n_freed = freed;
    return KV_OK;
}

kv_status kv_prefix_cache_stats(kv_prefix_cache_t c, int *cached_blocks, int64_t *lookups,
                                int64_t *hits) {
    if (!c) return KV_ERR_ARG;
    if (cached_blocks) *cached_blocks = (int)c->map.size();
    if (lookups) *lookups = c->lookups;
    if (hits) *hits = c->hits;
    return KV_OK;
}

}  // extern "C"
