"""Block manager calls on a pool: allocation, sharing, freeing and the
copy-on-write of one block before a write ("Makale Bulteni -- PagedAttention
ve vLLM", "Iddia ve Gerceklik": blocks are shared by reference and copied on
write)."""
import numpy as np
import pytest

import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import dev, host, pool_views, require_cuda

pytestmark = pytest.mark.gpu


def test_alloc_share_free_track_references():
    require_cuda()
    pool = pk.kv_pool_create(8, 16, 2, 64, pk.KV_F32)
    a = pk.kv_pool_allocator(pool)
    ids = np.zeros(3, np.int32)
    pk.kv_alloc_blocks(pool, ids)
    assert len(set(ids.tolist())) == 3 and pk.kv_allocator_num_free(a) == 5
    pk.kv_share_blocks(pool, ids[:2])
    assert [pk.kv_allocator_refcount(a, int(i)) for i in ids] == [2, 2, 1]
    pk.kv_free_blocks(pool, ids)
    assert [pk.kv_allocator_refcount(a, int(i)) for i in ids] == [1, 1, 0]
    assert pk.kv_allocator_num_free(a) == 6
    with pytest.raises(pk.KVError):  # more blocks than are free: nothing taken
        pk.kv_alloc_blocks(pool, np.zeros(7, np.int32))
    assert pk.kv_allocator_num_free(a) == 6
    pk.kv_pool_destroy(pool)


@pytest.mark.parametrize("dtype,d,hkv", [("bf16", 128, 8), ("f32", 64, 2)])
def test_cow_if_shared_copies_only_shared_blocks(dtype, d, hkv):
    require_cuda()
    nb = 16
    g = W.rng(77)
    bf = dtype == "bf16"
    kp_ = W.normal(g, (nb, hkv, 16, d), dtype)
    vp_ = W.normal(g, (nb, hkv, 16, d), dtype)
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16 if bf else pk.KV_F32)
    a = pk.kv_pool_allocator(pool)
    kv, vv = pool_views(pool, nb, hkv, d, bf)
    kv.copy_(dev(kp_))
    vv.copy_(dev(vp_))
    ids = np.zeros(2, np.int32)
    pk.kv_alloc_blocks(pool, ids)
    shared, private = int(ids[0]), int(ids[1])
    pk.kv_share_blocks(pool, ids[:1])                      # a second sequence holds block 0
    # private block: written in place
    assert pk.kv_cow_if_shared(pool, private) == (private, False)
    # shared block: a copy for the writer, the other holder keeps the original
    new_id, copied = pk.kv_cow_if_shared(pool, shared)
    assert copied and new_id not in (shared, private)
    assert pk.kv_allocator_refcount(a, shared) == 1 and pk.kv_allocator_refcount(a, new_id) == 1
    bits = np.uint16 if bf else np.uint32
    k_after = host(kv).view(bits)
    v_after = host(vv).view(bits)
    np.testing.assert_array_equal(k_after[new_id], kp_[shared].view(bits))
    np.testing.assert_array_equal(v_after[new_id], vp_[shared].view(bits))
    others = [i for i in range(nb) if i != new_id]
    np.testing.assert_array_equal(k_after[others], kp_[others].view(bits))  # nothing else moved
    assert pk.kv_get_device_error(pool) == 0
    with pytest.raises(pk.KVError):  # a free block cannot be written
        pk.kv_cow_if_shared(pool, int(np.setdiff1d(np.arange(nb), [shared, private, new_id])[0]))
    pk.kv_pool_destroy(pool)
