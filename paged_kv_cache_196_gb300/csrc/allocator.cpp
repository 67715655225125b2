// Host block manager: free list, reference counts, copy-on-write planning.
//
// "Makale Bulteni -- PagedAttention ve vLLM", section "Iddia ve Gerceklik":
// blocks come from a free pool as sequences grow, the page table maps logical
// to physical blocks, and parallel samples / branches share blocks by pointer
// with copy-on-write.  "PagedAttention Nedir?", "Nasil Calisir?" steps 2, 3
// and 5: allocate on demand, keep the mapping, reuse freed blocks.
//
// Free blocks sit in a FIFO ring: alloc pops from the head, free pushes at
// the tail, so blocks are handed out in the configured order and reused
// least-recently-freed first.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "paged_kv.h"

struct kv_allocator {
    int num_blocks = 0;
    std::vector<int32_t> ring;      // capacity num_blocks
    int head = 0, count = 0;        // free ids are ring[head .. head+count) mod num_blocks
    std::vector<int32_t> refcount;  // 0 = free
};

extern "C" {

const char *kv_status_string(kv_status s) {
    switch (s) {
        case KV_OK: return "ok";
        case KV_ERR_ARG: return "invalid argument";
        case KV_ERR_OOM: return "out of blocks or memory";
        case KV_ERR_UNSUPPORTED: return "unsupported shape or type";
        case KV_ERR_CUDA: return "CUDA call failed";
        case KV_ERR_DEVICE_BOUNDS: return "GPU met an out-of-range block id, slot or position";
        case KV_ERR_TIMEOUT: return "a pipeline wait inside a kernel timed out";
        case KV_ERR_STATE: return "call not valid in the current state";
    }
    return "unknown status";
}

kv_status kv_blocks_for_tokens(int64_t n_tokens, int block_size, int64_t *blocks,
                               int64_t *unused_slots) {
    if (n_tokens < 0 || block_size <= 0) return KV_ERR_ARG;
    int64_t nb = (n_tokens + block_size - 1) / block_size;
    if (blocks) *blocks = nb;
    if (unused_slots) *unused_slots = nb * block_size - n_tokens;
    return KV_OK;
}

kv_status kv_allocator_create(int num_blocks, kv_allocator_t *out) {
    if (!out || num_blocks <= 0) return KV_ERR_ARG;
    kv_allocator *a = new (std::nothrow) kv_allocator();
    if (!a) return KV_ERR_OOM;
    try {
        a->num_blocks = num_blocks;
        a->ring.resize(num_blocks);
        a->refcount.assign(num_blocks, 0);
    } catch (...) {
        delete a;
        return KV_ERR_OOM;
    }
    for (int i = 0; i < num_blocks; ++i) a->ring[i] = i;
    a->head = 0;
    a->count = num_blocks;
    *out = a;
    return KV_OK;
}

kv_status kv_allocator_destroy(kv_allocator_t a) {
    delete a;
    return KV_OK;
}

kv_status kv_allocator_set_order(kv_allocator_t a, const int32_t *order, int n) {
    if (!a || !order || n != a->num_blocks) return KV_ERR_ARG;
    if (a->count != a->num_blocks) return KV_ERR_STATE;
    std::vector<char> seen(n, 0);
    for (int i = 0; i < n; ++i) {
        if (order[i] < 0 || order[i] >= n || seen[order[i]]) return KV_ERR_ARG;
        seen[order[i]] = 1;
    }
    std::memcpy(a->ring.data(), order, sizeof(int32_t) * n);
    a->head = 0;
    return KV_OK;
}

kv_status kv_allocator_alloc(kv_allocator_t a, int n, int32_t *ids_out) {
    if (!a || n < 0 || (n > 0 && !ids_out)) return KV_ERR_ARG;
    if (n > a->count) return KV_ERR_OOM;
    for (int i = 0; i < n; ++i) {
        int32_t id = a->ring[a->head];
        a->head = (a->head + 1) % a->num_blocks;
        a->refcount[id] = 1;
        ids_out[i] = id;
    }
    a->count -= n;
    return KV_OK;
}

kv_status kv_allocator_share(kv_allocator_t a, int n, const int32_t *ids) {
    if (!a || n < 0 || (n > 0 && !ids)) return KV_ERR_ARG;
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= a->num_blocks || a->refcount[ids[i]] <= 0) return KV_ERR_ARG;
    for (int i = 0; i < n; ++i) a->refcount[ids[i]] += 1;
    return KV_OK;
}

kv_status kv_allocator_free(kv_allocator_t a, int n, const int32_t *ids) {
    if (!a || n < 0 || (n > 0 && !ids)) return KV_ERR_ARG;
    // Validate against the counts as they would evolve, so a list naming a
    // block more often than it is referenced is rejected without change.
    std::vector<std::pair<int32_t, int>> dec;
    for (int i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (id < 0 || id >= a->num_blocks) return KV_ERR_ARG;
        int times = 0;
        for (int j = 0; j < i; ++j) times += ids[j] == id;
        if (a->refcount[id] - times <= 0) return KV_ERR_ARG;
    }
    for (int i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (--a->refcount[id] == 0) {
            a->ring[(a->head + a->count) % a->num_blocks] = id;
            a->count += 1;
        }
    }
    return KV_OK;
}

kv_status kv_allocator_refcount(kv_allocator_t a, int32_t id, int *refcount) {
    if (!a || !refcount || id < 0 || id >= a->num_blocks) return KV_ERR_ARG;
    *refcount = a->refcount[id];
    return KV_OK;
}

kv_status kv_allocator_num_free(kv_allocator_t a, int *num_free) {
    if (!a || !num_free) return KV_ERR_ARG;
    *num_free = a->count;
    return KV_OK;
}

kv_status kv_prepare_append(kv_allocator_t a, int block_size, int32_t *table_row,
                            int max_blocks, int *num_blocks, int64_t cur_len, int n_new,
                            int64_t *slots_out, int32_t *cow_src, int32_t *cow_dst,
                            int *n_cow) {
    if (!a || block_size <= 0 || !table_row || !num_blocks || cur_len < 0 || n_new < 0 ||
        (n_new > 0 && !slots_out) || !n_cow || *n_cow < 0)
        return KV_ERR_ARG;
    const int nb = *num_blocks;
    if (nb < 0 || nb > max_blocks) return KV_ERR_ARG;
    if ((cur_len + block_size - 1) / block_size > nb) return KV_ERR_ARG;  // row too short for cur_len
    for (int i = 0; i < nb; ++i)
        if (table_row[i] < 0 || table_row[i] >= a->num_blocks || a->refcount[table_row[i]] <= 0)
            return KV_ERR_ARG;
    if (n_new == 0) {
        *n_cow = 0;
        return KV_OK;
    }
    const int64_t end = cur_len + n_new;
    const int64_t first_block = cur_len / block_size;
    const int64_t last_block = (end - 1) / block_size;
    if (last_block >= max_blocks) return KV_ERR_ARG;
    // Plan: blocks already in the row that receive new tokens and are shared
    // need a private copy; blocks past the row's end are fresh.
    int need_cow = 0, need_new = 0;
    for (int64_t bi = first_block; bi <= last_block; ++bi) {
        if (bi < nb) need_cow += a->refcount[table_row[bi]] > 1;
        else need_new += 1;
    }
    if (need_cow > *n_cow || (need_cow > 0 && (!cow_src || !cow_dst))) return KV_ERR_ARG;
    if (need_cow + need_new > a->count) return KV_ERR_OOM;
    int k = 0;
    for (int64_t bi = first_block; bi <= last_block; ++bi) {
        int32_t id;
        if (bi < nb) {
            if (a->refcount[table_row[bi]] <= 1) continue;
            kv_allocator_alloc(a, 1, &id);
            cow_src[k] = table_row[bi];
            cow_dst[k] = id;
            ++k;
            a->refcount[table_row[bi]] -= 1;  // still > 0: another sequence holds it
            table_row[bi] = id;
        } else {
            kv_allocator_alloc(a, 1, &id);
            table_row[bi] = id;
        }
    }
    *num_blocks = (int)(last_block + 1 > nb ? last_block + 1 : nb);
    for (int i = 0; i < n_new; ++i) {
        int64_t pos = cur_len + i;
        slots_out[i] = (int64_t)table_row[pos / block_size] * block_size + pos % block_size;
    }
    *n_cow = k;
    return KV_OK;
}

kv_status kv_prepare_append_batch(kv_allocator_t a, int block_size, int batch, int32_t *tables,
                                  int max_blocks, int32_t *num_blocks, const int64_t *cur_lens,
                                  const int32_t *n_new, int64_t *slots_out, int32_t *cow_src,
                                  int32_t *cow_dst, int *n_cow) {
    if (!a || block_size <= 0 || batch < 0 || max_blocks < 0 || !n_cow || *n_cow < 0) return KV_ERR_ARG;
    if (batch > 0 && (!tables || !num_blocks || !cur_lens || !n_new)) return KV_ERR_ARG;
    // Plan first, change nothing: blocks to take and copies to make for the
    // whole batch.  A block shared by several sequences of this batch is
    // copied by all but the last writer (whose write finds it private).
    std::vector<int> pending;  // refcount drops planned per block
    long long need_new = 0, need_cow = 0, total_slots = 0;
    for (int b = 0; b < batch; ++b) {
        const int32_t *row = tables + (size_t)b * max_blocks;
        const int nb = num_blocks[b];
        const int64_t len = cur_lens[b];
        if (nb < 0 || nb > max_blocks || len < 0 || n_new[b] < 0) return KV_ERR_ARG;
        if ((len + block_size - 1) / block_size > nb) return KV_ERR_ARG;
        for (int i = 0; i < nb; ++i)
            if (row[i] < 0 || row[i] >= a->num_blocks || a->refcount[row[i]] <= 0) return KV_ERR_ARG;
        total_slots += n_new[b];
        if (n_new[b] == 0) continue;
        const int64_t first = len / block_size, last = (len + n_new[b] - 1) / block_size;
        if (last >= max_blocks) return KV_ERR_ARG;
        for (int64_t bi = first; bi <= last; ++bi) {
            if (bi >= nb) {
                need_new += 1;
                continue;
            }
            const int32_t id = row[bi];
            if (pending.empty()) pending.assign(a->num_blocks, 0);
            const int left = a->refcount[id] - pending[id];
            if (left > 1) {  // still shared when this sequence writes: copy
                need_cow += 1;
                pending[id] += 1;
            }
        }
    }
    if (total_slots > 0 && !slots_out) return KV_ERR_ARG;
    if (need_cow > *n_cow || (need_cow > 0 && (!cow_src || !cow_dst))) return KV_ERR_ARG;
    if (need_new + need_cow > a->count) return KV_ERR_OOM;
    // Apply, sequence by sequence (the single-sequence planner makes the same
    // decisions in the same order).
    int k = 0;
    long long off = 0;
    for (int b = 0; b < batch; ++b) {
        int cap = *n_cow - k;
        int nb = num_blocks[b];
        const kv_status st = kv_prepare_append(a, block_size, tables + (size_t)b * max_blocks,
                                               max_blocks, &nb, cur_lens[b], n_new[b],
                                               slots_out ? slots_out + off : nullptr,
                                               cow_src ? cow_src + k : nullptr,
                                               cow_dst ? cow_dst + k : nullptr, &cap);
        if (st != KV_OK) return st;  // not reached: the plan above checked every condition
        num_blocks[b] = nb;
        k += cap;
        off += n_new[b];
    }
    *n_cow = k;
    return KV_OK;
}

}  // extern "C"
