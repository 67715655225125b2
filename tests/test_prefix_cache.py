"""Prefix cache (host): exact reuse of full blocks keyed by their tokens and
everything before them.  "PagedAttention Nedir?", "Prefix Sharing Nasil
Calisir?": reuse needs the same tokens and the same preceding context."""
import numpy as np
import pytest

import paged_kv_cache_196_gb300 as pk
import workloads as W

BS = 16


def _seq(a, n_tokens):
    row = np.full(64, -1, np.int32)
    nb, _ = pk.kv_prepare_append(a, row, 0, 0, n_tokens, np.zeros(n_tokens, np.int64),
                                 np.zeros(0, np.int32), np.zeros(0, np.int32))
    return row[:nb].copy()


def test_match_returns_longest_cached_prefix_with_references():
    a = pk.kv_allocator_create(64)
    c = pk.kv_prefix_cache_create(a, 32)
    toks = W.rng(1).integers(0, 32000, 100).astype(np.int32)  # 6 full blocks + 4 tokens
    blocks = _seq(a, 100)
    assert pk.kv_prefix_cache_insert(c, toks, blocks) == 6       # the partial block is not listed
    out = np.zeros(16, np.int32)
    # same prompt: all 6 full blocks, in order, one more reference each
    assert pk.kv_prefix_cache_match(c, toks, out) == 6
    np.testing.assert_array_equal(out[:6], blocks[:6])
    assert [pk.kv_allocator_refcount(a, int(b)) for b in blocks[:6]] == [3] * 6
    assert pk.kv_allocator_refcount(a, int(blocks[6])) == 1
    # a prompt sharing the first 50 tokens: 3 full blocks
    other = toks.copy()
    other[50:] += 1
    assert pk.kv_prefix_cache_match(c, other, out) == 3
    # the same block contents after a different first block: no match at all
    shifted = toks.copy()
    shifted[0] += 1
    assert pk.kv_prefix_cache_match(c, shifted, out) == 0
    assert pk.kv_prefix_cache_match(c, toks[:15], out) == 0       # not even one full block
    assert pk.kv_prefix_cache_stats(c) == (6, 4, 2)
    pk.kv_prefix_cache_destroy(c)
    pk.kv_allocator_destroy(a)


def test_eviction_frees_only_blocks_nobody_else_holds_lru_first():
    a = pk.kv_allocator_create(32)
    c = pk.kv_prefix_cache_create(a, 32)
    g = W.rng(2)
    t1 = g.integers(0, 1000, 32).astype(np.int32)
    t2 = g.integers(0, 1000, 32).astype(np.int32)
    b1, b2 = _seq(a, 32), _seq(a, 32)
    pk.kv_prefix_cache_insert(c, t1, b1)
    pk.kv_prefix_cache_insert(c, t2, b2)
    pk.kv_allocator_free(a, b1)          # request 1 finished: only the cache holds b1
    free0 = pk.kv_allocator_num_free(a)
    out = np.zeros(4, np.int32)
    assert pk.kv_prefix_cache_match(c, t1, out) == 2   # t1 becomes most recently used; user ref
    assert pk.kv_prefix_cache_evict(c, 10) == 0        # b1 in use by the matcher, b2 by request 2
    pk.kv_allocator_free(a, out[:2])
    pk.kv_allocator_free(a, b2)
    pk.kv_prefix_cache_match(c, t1, out)               # touch t1 again, then release
    pk.kv_allocator_free(a, out[:2])
    assert pk.kv_prefix_cache_evict(c, 2) == 2         # least recently used first: request 2's blocks
    assert pk.kv_prefix_cache_match(c, t2, out) == 0
    assert pk.kv_prefix_cache_match(c, t1, out) == 2
    pk.kv_allocator_free(a, out[:2])
    assert pk.kv_allocator_num_free(a) == free0 + 2
    pk.kv_prefix_cache_destroy(c)
    assert pk.kv_allocator_num_free(a) == 32
    pk.kv_allocator_destroy(a)


def test_capacity_evicts_idle_entries_and_stops_when_none_can_go():
    a = pk.kv_allocator_create(64)
    c = pk.kv_prefix_cache_create(a, 4)
    g = W.rng(3)
    toks = [g.integers(0, 1000, 32).astype(np.int32) for _ in range(3)]
    rows = [_seq(a, 32) for _ in range(3)]
    assert pk.kv_prefix_cache_insert(c, toks[0], rows[0]) == 2
    assert pk.kv_prefix_cache_insert(c, toks[1], rows[1]) == 2
    # full, and both entries are still held by their requests: nothing is listed
    assert pk.kv_prefix_cache_insert(c, toks[2], rows[2]) == 0
    pk.kv_allocator_free(a, rows[0])
    assert pk.kv_prefix_cache_insert(c, toks[2], rows[2]) == 2   # request 0's blocks evicted
    out = np.zeros(4, np.int32)
    assert pk.kv_prefix_cache_match(c, toks[0], out) == 0
    assert pk.kv_prefix_cache_stats(c)[0] == 4
    pk.kv_prefix_cache_destroy(c)
    pk.kv_allocator_destroy(a)
