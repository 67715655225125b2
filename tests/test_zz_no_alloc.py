"""The decode entry point for callers that cannot allocate device memory.

Such callers (a plugin whose host framework owns all device memory, a
serving loop that must not call cudaMalloc after start-up) use
paged_decode_attention_noalloc: the split-KV scratch lives in a fixed array
inside the library instead of a caller-supplied workspace.  Its results must
match the regular entry point's within the attention tolerance, on two calls
in a row (the second call reuses the scratch the first one left behind).

This file is collected last on purpose, and it builds its own inputs so it
also passes when run alone in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_196_gb300 as pk
import workloads as W

pytestmark = pytest.mark.gpu


def _setup(lens, hq, hkv, d, seed):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    g = W.rng(seed)
    lens = np.asarray(lens, np.int32)
    need = int(sum((int(L) + 15) // 16 for L in lens))
    nb = need + 4
    max_blocks = int(max((int(L) + 15) // 16 for L in lens))
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    alloc = pk.kv_pool_allocator(pool)
    pk.kv_allocator_set_order(alloc, W.permutation(g, nb))
    tables = np.full((len(lens), max_blocks), -1, np.int32)
    for b, L in enumerate(lens):
        slots = np.zeros(int(L), np.int64)
        pk.kv_prepare_append(alloc, tables[b], 0, 0, int(L), slots, np.zeros(0, np.int32),
                             np.zeros(0, np.int32))
        k = torch.from_numpy(W.normal(g, (int(L), hkv, d), "bf16").view(np.int16)).cuda()
        v = torch.from_numpy(W.normal(g, (int(L), hkv, d), "bf16").view(np.int16)).cuda()
        pk.kv_append(pool, k, v, torch.from_numpy(slots).cuda(), int(L))
    q = torch.from_numpy(W.normal(g, (len(lens), hq, d), "bf16").view(np.int16)).cuda()
    return pool, q, torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), max_blocks


@pytest.mark.parametrize("splits", [4, 0])
def test_noalloc_decode_matches_regular_entry_point_twice(splits):
    lens = [1500, 35, 4096, 700, 17, 2049, 1, 3000]
    hq, hkv, d = 32, 8, 128
    pool, q, tables, seq_lens, max_blocks = _setup(lens, hq, hkv, d, seed=2024)
    B, scale = len(lens), 1 / math.sqrt(d)
    try:
        wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, max_blocks, splits)
        assert wsb > 0  # the plan really uses scratch
        ws = torch.empty(wsb // 4, dtype=torch.float32, device="cuda")
        ref = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
        ref_lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
        pk.paged_decode_attention(pool, q, tables, max_blocks, seq_lens, B, hq, scale, ref,
                                  pk.KV_F32, ref_lse, splits, ws, wsb)
        torch.cuda.synchronize()
        ref_np, ref_lse_np = ref.cpu().numpy(), ref_lse.cpu().numpy()
        tol = 2e-3 * float(np.max(np.abs(ref_np)))
        for _ in range(2):
            out = torch.full((B, hq, d), float("nan"), dtype=torch.float32, device="cuda")
            lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
            pk.paged_decode_attention_noalloc(pool, q, tables, max_blocks, seq_lens, B, hq, scale,
                                              out, pk.KV_F32, lse, splits)
            torch.cuda.synchronize()
            assert pk.kv_get_device_error(pool) == 0
            o = out.cpu().numpy()
            assert np.all(np.isfinite(o))
            assert float(np.max(np.abs(o - ref_np))) <= tol
            np.testing.assert_allclose(lse.cpu().numpy(), ref_lse_np, atol=1e-3)
    finally:
        pk.kv_pool_destroy(pool)


def test_noalloc_rejects_plans_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    pool = pk.kv_pool_create(8, 16, 8, 128, pk.KV_BF16)
    try:
        B, hq, max_blocks, splits = 512, 64, 4096, 64   # about 1.1 GB of partials
        assert pk.kv_decode_workspace_size(B, hq, 8, 128, max_blocks, splits) > (8 << 20)
        with pytest.raises(pk.KVError) as e:
            pk.paged_decode_attention_noalloc(pool, 0, 0, max_blocks, 0, B, hq, 0.1, 0,
                                              pk.KV_F32, None, splits)
        assert e.value.status == -3  # KV_ERR_UNSUPPORTED, nothing launched
    finally:
        pk.kv_pool_destroy(pool)
