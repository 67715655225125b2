"""A pool or contiguous context used while another GPU is current.

Its memory lives on the device that was current at creation; a call made with
another device current must be refused (KV_ERR_ARG, nothing launched) instead
of launching there against memory of another GPU.  Needs two visible GPUs.
"""
import pytest
import torch

import paged_kv_cache_196_gb300 as pk

pytestmark = pytest.mark.gpu


def _two_gpus():
    if not torch.cuda.is_available() or torch.cuda.device_count() < 2:
        pytest.skip("needs two visible CUDA devices")
    pk.lib()


def test_pool_calls_on_another_device_are_refused():
    _two_gpus()
    torch.cuda.set_device(0)
    pool = pk.kv_pool_create(8, 16, 2, 64, pk.KV_F32)
    k = torch.zeros((1, 2, 64), dtype=torch.float32, device="cuda:0")
    slots = torch.zeros(1, dtype=torch.int64, device="cuda:0")
    try:
        torch.cuda.set_device(1)
        with pytest.raises(pk.KVError) as e:
            pk.kv_append(pool, k, k, slots, 1)
        assert e.value.status == -1
        with pytest.raises(pk.KVError) as e:
            pk.kv_get_device_error(pool)
        assert e.value.status == -1
        torch.cuda.set_device(0)
        pk.kv_append(pool, k, k, slots, 1)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        torch.cuda.set_device(1)
    finally:
        pk.kv_pool_destroy(pool)  # frees on device 0 and leaves device 1 current
    assert torch.cuda.current_device() == 1
    torch.cuda.set_device(0)


def test_contig_calls_on_another_device_are_refused():
    _two_gpus()
    torch.cuda.set_device(0)
    ctx = pk.kv_contig_create(2, 1000, 2, 64, pk.KV_F32)
    try:
        pk.kv_contig_reserve(ctx, 0)
        torch.cuda.set_device(1)
        with pytest.raises(pk.KVError) as e:
            pk.kv_contig_ensure(ctx, 0, 10)
        assert e.value.status == -1
        torch.cuda.set_device(0)
        pk.kv_contig_ensure(ctx, 0, 10)
        assert pk.kv_contig_stats(ctx, 0)[0] > 0
    finally:
        torch.cuda.set_device(0)
        pk.kv_contig_destroy(ctx)
