"""Swap / preemption block copies between the pool and pinned host memory:
bit-exact round trip, out-of-range ids flagged and skipped."""
import numpy as np
import pytest
import torch

import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import dev, host, pool_views, require_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,d,hkv", [("bf16", 128, 8), ("f32", 64, 2)])
def test_swap_out_and_in_round_trip(dtype, d, hkv):
    require_cuda()
    nb = 64
    g = W.rng(81)
    pk_ = W.normal(g, (nb, hkv, 16, d), dtype)
    pv_ = W.normal(g, (nb, hkv, 16, d), dtype)
    bf = dtype == "bf16"
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16 if bf else pk.KV_F32)
    kv, vv = pool_views(pool, nb, hkv, d, bf)
    kv.copy_(dev(pk_)); vv.copy_(dev(pv_))
    ids = np.array([5, 17, 3, 40, 63], np.int32)
    nbytes = pk.kv_swap_bytes(pool, len(ids))
    buf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    pk.kv_swap_out(pool, dev(ids), len(ids), buf)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    dt = np.uint16 if bf else np.float32
    got = buf.numpy().view(dt).reshape(len(ids), 2, hkv, 16, d)
    bits = np.uint16 if bf else np.uint32
    np.testing.assert_array_equal(got[:, 0].view(bits), pk_[ids].view(bits))
    np.testing.assert_array_equal(got[:, 1].view(bits), pv_[ids].view(bits))
    # swap back into other blocks of an emptied pool
    kv.zero_(); vv.zero_()
    ids2 = np.array([0, 1, 2, 62, 33], np.int32)
    pk.kv_swap_in(pool, dev(ids2), len(ids2), buf)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    k_after = host(kv).view(bits)
    v_after = host(vv).view(bits)
    np.testing.assert_array_equal(k_after[ids2], pk_[ids].view(bits))
    np.testing.assert_array_equal(v_after[ids2], pv_[ids].view(bits))
    others = np.setdiff1d(np.arange(nb), ids2)
    assert not k_after[others].any() and not v_after[others].any()
    pk.kv_pool_destroy(pool)


def test_swap_rejects_out_of_range_ids():
    require_cuda()
    pool = pk.kv_pool_create(8, 16, 2, 64, pk.KV_F32)
    kv, vv = pool_views(pool, 8, 2, 64, False)
    kv.fill_(1.0); vv.fill_(1.0)
    buf = torch.zeros(pk.kv_swap_bytes(pool, 2), dtype=torch.uint8).pin_memory()
    pk.kv_swap_out(pool, dev(np.array([3, 9], np.int32)), 2, buf)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0x1
    half = buf.numel() // 2
    assert torch.all(buf[:half].view(torch.float32) == 1.0) and not buf[half:].any()
    pk.kv_swap_in(pool, dev(np.array([-1, 2], np.int32)), 2, torch.zeros_like(buf).pin_memory())
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0x1
    assert torch.all(kv[2] == 0) and torch.all(kv[3] == 1.0)
    pk.kv_pool_destroy(pool)
