"""Prefix cache on the GPU.  A request whose prompt starts like an earlier one
takes that request's full KV blocks from the cache and appends only its own
suffix; its decode must equal attention over its logical KV (the first
request's rows for the shared blocks, its own rows after them).
"PagedAttention Nedir?", "Prefix Sharing Nasil Calisir?": reuse needs the same
tokens and the same preceding context, and the reused blocks stay resident."""
import numpy as np
import pytest
import torch

import oracle as O
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, bf16_to_f64, dev, host, pool_views, require_cuda

pytestmark = pytest.mark.gpu


def test_matched_prefix_blocks_decode_like_their_logical_kv():
    require_cuda()
    nb, hkv, hq, d, bs = 64, 2, 8, 128, 16
    g = W.rng(91)
    pool = pk.kv_pool_create(nb, bs, hkv, d, pk.KV_BF16)
    a = pk.kv_pool_allocator(pool)
    pk.kv_allocator_set_order(a, W.permutation(g, nb))
    cache = pk.kv_prefix_cache_create(a, 32)
    maxb = 8

    # request 1: a 100-token prompt, written through its slot mapping
    toks1 = g.integers(0, 32000, 100).astype(np.int32)
    row1 = np.full(maxb, -1, np.int32)
    slots1 = np.zeros(100, np.int64)
    nb1, _ = pk.kv_prepare_append(a, row1, 0, 0, 100, slots1, np.zeros(0, np.int32),
                                  np.zeros(0, np.int32))
    k1 = W.normal(g, (100, hkv, d), "bf16")
    v1 = W.normal(g, (100, hkv, d), "bf16")
    pk.kv_append(pool, dev(k1), dev(v1), dev(slots1), 100)
    assert pk.kv_prefix_cache_insert(cache, toks1, row1[:nb1]) == 6

    # request 2 shares the first 70 prompt tokens: the first 4 full blocks match
    toks2 = np.concatenate([toks1[:70], g.integers(0, 32000, 50).astype(np.int32)])
    row2 = np.full(maxb, -1, np.int32)
    n_match = pk.kv_prefix_cache_match(cache, toks2, row2)
    assert n_match == 4
    np.testing.assert_array_equal(row2[:4], row1[:4])
    assert [pk.kv_allocator_refcount(a, int(x)) for x in row2[:4]] == [3] * 4
    cached = n_match * bs
    n_new = len(toks2) - cached
    slots2 = np.zeros(n_new, np.int64)
    nb2, ncow = pk.kv_prepare_append(a, row2, n_match, cached, n_new, slots2,
                                     np.zeros(0, np.int32), np.zeros(0, np.int32))
    assert ncow == 0 and nb2 == 8
    assert not np.isin(row2[4:nb2], row1[:nb1]).any()   # the suffix got blocks of its own
    k2 = W.normal(g, (n_new, hkv, d), "bf16")
    v2 = W.normal(g, (n_new, hkv, d), "bf16")
    pk.kv_append(pool, dev(k2), dev(v2), dev(slots2), n_new)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0

    # the shared blocks still hold request 1's rows, bit for bit
    kv, vv = pool_views(pool, nb, hkv, d, True)
    kp = host(kv, like_bf16=True)
    for i in range(4):
        np.testing.assert_array_equal(kp[row1[i]].transpose(1, 0, 2), k1[16 * i:16 * i + 16])

    # decode both requests in one batch
    q = W.normal(g, (2, hq, d), "bf16")
    lens = np.array([100, 120], np.int32)
    tables = np.stack([row1, row2]).astype(np.int32)
    out = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
    ws_bytes = pk.kv_decode_workspace_size(2, hq, hkv, d, maxb, 0)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device="cuda")
    scale = 1.0 / np.sqrt(d)
    pk.paged_decode_attention(pool, dev(q), dev(tables), maxb, dev(lens), 2, hq, scale, out,
                              pk.KV_F32, None, 0, ws, ws_bytes)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    got = host(out)

    # oracle over the explicit logical KV of each request
    K = [bf16_to_f64(k1), bf16_to_f64(np.concatenate([k1[:cached], k2]))]
    V = [bf16_to_f64(v1), bf16_to_f64(np.concatenate([v1[:cached], v2]))]
    qf = bf16_to_f64(q)
    ref = np.empty((2, hq, d))
    for b in range(2):
        for h in range(hq):
            ref[b, h], _ = O.attend_logical(qf[b, h], K[b], V[b], h // (hq // hkv), scale)
    assert_close_scaled(got, ref, 2e-3, "prefix-cache decode")

    # request 1 finishes; its blocks stay resident for the cache and request 2
    pk.kv_allocator_free(a, row1[:nb1])
    assert pk.kv_prefix_cache_evict(cache, 10) == 2     # blocks 4, 5: only the cache held them
    pk.kv_prefix_cache_destroy(cache)
    pk.kv_pool_destroy(pool)
