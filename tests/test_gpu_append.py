"""KV append (slot-mapping write) and copy-on-write block copy on the GPU:
bit-exact against the oracle's byte copy, every untouched slot unchanged."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import dev, host, pool_views, require_cuda

pytestmark = pytest.mark.gpu


def _sentinel_pool(nb, hkv, d, dtype):
    return W.empty_pool(nb, hkv, d, dtype, W.NAN_BF16 if dtype == "bf16" else W.NAN_F32)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 128)])
def test_append_bit_exact_with_sentinel(dtype, d):
    require_cuda()
    nb, hkv, T = 40, 4, 300
    g = W.rng(31)
    slots = g.permutation(nb * 16)[:T].astype(np.int64)
    slots[::17] = -1                                   # skipped tokens
    k = W.normal(g, (T, hkv, d), dtype)
    v = W.normal(g, (T, hkv, d), dtype)
    ref_k, ref_v = _sentinel_pool(nb, hkv, d, dtype), _sentinel_pool(nb, hkv, d, dtype)
    oracle.append(ref_k, ref_v, k, v, slots)
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16 if dtype == "bf16" else pk.KV_F32)
    kv, vv = pool_views(pool, nb, hkv, d, dtype == "bf16")
    kv.copy_(dev(_sentinel_pool(nb, hkv, d, dtype)))
    vv.copy_(dev(_sentinel_pool(nb, hkv, d, dtype)))
    pk.kv_append(pool, dev(k), dev(v), dev(slots), T)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    bits = np.uint16 if dtype == "bf16" else np.uint32
    np.testing.assert_array_equal(host(kv).view(bits), ref_k.view(bits))
    np.testing.assert_array_equal(host(vv).view(bits), ref_v.view(bits))
    pk.kv_pool_destroy(pool)


def test_append_out_of_range_slot_is_flagged_and_skipped():
    require_cuda()
    nb, hkv, d = 4, 2, 64
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_F32)
    kv, vv = pool_views(pool, nb, hkv, d, False)
    kv.zero_(); vv.zero_()
    k = np.ones((2, hkv, d), np.float32)
    pk.kv_append(pool, dev(k), dev(k), dev(np.array([5, nb * 16 + 3], np.int64)), 2)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0x2
    assert pk.kv_get_device_error(pool) == 0   # cleared by the read
    got = host(kv)
    assert np.all(got[0, :, 5] == 1) and got.sum() == hkv * d
    pk.kv_pool_destroy(pool)


def test_append_llama_sized_chunk():
    # 8192 tokens x 8 heads x 128 dims: the prefill chunk size.
    require_cuda()
    nb, hkv, d, T = 1024, 8, 128, 8192
    g = W.rng(32)
    slots = g.permutation(nb * 16)[:T].astype(np.int64)
    k = W.normal(g, (T, hkv, d), "bf16")
    v = W.normal(g, (T, hkv, d), "bf16")
    ref_k, ref_v = W.empty_pool(nb, hkv, d, "bf16"), W.empty_pool(nb, hkv, d, "bf16")
    oracle.append(ref_k, ref_v, k, v, slots)
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    kv, vv = pool_views(pool, nb, hkv, d, True)
    kv.zero_(); vv.zero_()
    pk.kv_append(pool, dev(k), dev(v), dev(slots), T)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(kv).view(np.uint16), ref_k)
    np.testing.assert_array_equal(host(vv).view(np.uint16), ref_v)
    pk.kv_pool_destroy(pool)


def test_copy_blocks_exact_and_flags_bad_ids():
    require_cuda()
    nb, hkv, d = 12, 2, 128
    g = W.rng(33)
    pk_ = W.normal(g, (nb, hkv, 16, d), "bf16")
    pv_ = W.normal(g, (nb, hkv, 16, d), "bf16")
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    kv, vv = pool_views(pool, nb, hkv, d, True)
    kv.copy_(dev(pk_)); vv.copy_(dev(pv_))
    src = np.array([1, 4, 7], np.int32)
    dst = np.array([9, 10, 11], np.int32)
    pk.kv_copy_blocks(pool, dev(src), dev(dst), 3)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    ek, ev = pk_.copy(), pv_.copy()
    ek[dst] = pk_[src]; ev[dst] = pv_[src]
    np.testing.assert_array_equal(host(kv).view(np.uint16), ek)
    np.testing.assert_array_equal(host(vv).view(np.uint16), ev)
    pk.kv_copy_blocks(pool, dev(np.array([0, nb], np.int32)), dev(np.array([nb + 1, 2], np.int32)), 2)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0x1
    np.testing.assert_array_equal(host(kv).view(np.uint16), ek)  # nothing written
    pk.kv_pool_destroy(pool)
