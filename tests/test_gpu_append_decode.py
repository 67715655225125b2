"""One decode step in one call: paged_append_and_decode against kv_append
followed by paged_decode_attention, and against the oracle on the appended
content.  "PagedAttention Nedir?", "Nasil Calisir?": the new token's KV is
written into its block, then the step attends all tokens."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, dev, host, pool_views, require_cuda

pytestmark = pytest.mark.gpu


def _setup(lens_after, hq, hkv, d, dtype, seed):
    """Pool content before the step (the new token's slot holds NaN), tables,
    the new token per sequence and its slot."""
    g = W.rng(seed)
    lens = np.asarray(lens_after, np.int32)
    need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
    nb = need + 5
    maxb = max(oracle.blocks_needed(int(L), 16) for L in lens)
    tables = oracle.build_block_tables(lens, 16, W.permutation(g, nb), maxb)
    pool_k = W.normal(g, (nb, hkv, 16, d), dtype)
    pool_v = W.normal(g, (nb, hkv, 16, d), dtype)
    slots = np.array([int(tables[b, (L - 1) // 16]) * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                     np.int64)
    nan = W.NAN_BF16 if dtype == "bf16" else W.NAN_F32
    raw = np.uint16 if dtype == "bf16" else np.uint32
    for s in slots:  # before the step the new slots hold garbage
        pool_k.view(raw)[s // 16, :, s % 16, :] = nan
        pool_v.view(raw)[s // 16, :, s % 16, :] = nan
    k_new = W.normal(g, (len(lens), hkv, d), dtype)
    v_new = W.normal(g, (len(lens), hkv, d), dtype)
    q = W.normal(g, (len(lens), hq, d), dtype)
    return lens, tables, pool_k, pool_v, slots, k_new, v_new, q


def _run(fused, lens, tables, pool_k, pool_v, slots, k_new, v_new, q, splits, order=None):
    bf = pool_k.dtype == np.uint16
    nb, hkv, _, d = pool_k.shape
    B, hq, _ = q.shape
    maxb = tables.shape[1]
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16 if bf else pk.KV_F32)
    kv, vv = pool_views(pool, nb, hkv, d, bf)
    kv.copy_(dev(pool_k))
    vv.copy_(dev(pool_v))
    out = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    args = (dev(tables), maxb, dev(lens), B, hq, 1.0 / math.sqrt(d), out, pk.KV_F32, lse, splits,
            ws, wsb)
    if fused:
        pk.paged_append_and_decode(pool, dev(q), dev(k_new), dev(v_new), dev(slots), *args,
                                   seq_order=None if order is None else dev(order))
    else:
        pk.kv_append(pool, dev(k_new), dev(v_new), dev(slots), B)
        pk.paged_decode_attention(pool, dev(q), *args)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    res = host(out), host(lse), host(kv, like_bf16=bf), host(vv, like_bf16=bf)
    pk.kv_pool_destroy(pool)
    return res


@pytest.mark.parametrize("shape", [(32, 8, 128, "bf16", 0), (32, 8, 128, "bf16", 3),
                                   (56, 8, 128, "bf16", 2), (4, 2, 64, "f32", 0)])
def test_fused_step_equals_append_then_decode(shape):
    """bf16 / d128 / >= 3 heads per kv head is the fused kernel (4 and 7 heads
    per kv head, several split plans); fp32 / d64 / 2 heads takes the two calls."""
    require_cuda()
    hq, hkv, d, dtype, splits = shape
    lens = [1, 16, 17, 33, 300, 511, 1024, 1025, 2000, 47]
    case = _setup(lens, hq, hkv, d, dtype, seed=hq + d + splits)
    a = _run(False, *case, splits=splits)
    b = _run(True, *case, splits=splits)
    bits = np.uint16 if dtype == "bf16" else np.uint32
    np.testing.assert_array_equal(a[0], b[0])  # output, bit for bit
    np.testing.assert_array_equal(a[1], b[1])  # lse
    np.testing.assert_array_equal(a[2].view(bits), b[2].view(bits))  # K pool after the step
    np.testing.assert_array_equal(a[3].view(bits), b[3].view(bits))  # V pool
    # and the oracle on the appended content
    lens_, tables, pool_k, pool_v, slots, k_new, v_new, q = case
    pk_, pv_ = pool_k.copy(), pool_v.copy()
    oracle.append(pk_, pv_, k_new, v_new, slots)
    ref, ref_lse = oracle.paged_decode(pk_, pv_, tables, lens_, q, 1.0 / math.sqrt(d))
    assert_close_scaled(b[0], ref, 2e-3 if dtype == "bf16" else 1e-5, "fused step")


def test_sequence_order_changes_no_result():
    """The grid may take the sequences in any order (kv_decode_order: longest
    first); output, lse and pool bytes stay bit-identical."""
    require_cuda()
    lens = [700, 33, 2000, 1, 1500, 16, 900, 260]
    case = _setup(lens, 32, 8, 128, "bf16", seed=5)
    order = np.zeros(len(lens), np.int32)
    pk.kv_decode_order(np.asarray(lens, np.int32), order)
    assert order.tolist() == [2, 4, 6, 0, 7, 1, 5, 3]
    for splits in (0, 3):
        a = _run(True, *case, splits=splits)
        b = _run(True, *case, splits=splits, order=order)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x.view(np.uint32) if x.dtype == np.float32 else x, y.view(np.uint32) if y.dtype == np.float32 else y)


def test_launch_overlap_keeps_step_order():
    """With kv_pool_set_launch_overlap, back-to-back decode steps may start
    before the previous one has finished; each waits for it before touching
    memory.  Two steps: the second attends the token the first appended (its
    slot held NaN before), so a step that read early would show it.  Output,
    lse and pool bytes bit-identical to ordinary launches, and the oracle."""
    require_cuda()
    g = W.rng(77)
    hq, hkv, d = 32, 8, 128
    lens2 = np.array([1025, 17, 300, 2000, 16, 47, 511, 1024], np.int32)  # after both steps
    lens1 = lens2 - 1
    nb = sum(oracle.blocks_needed(int(L), 16) for L in lens2) + 5
    maxb = max(oracle.blocks_needed(int(L), 16) for L in lens2)
    tables = oracle.build_block_tables(lens2, 16, W.permutation(g, nb), maxb)
    pool_k = W.normal(g, (nb, hkv, 16, d), "bf16")
    pool_v = W.normal(g, (nb, hkv, 16, d), "bf16")

    def slot(b, pos):
        return int(tables[b, pos // 16]) * 16 + pos % 16

    s1 = np.array([slot(b, int(L) - 1) for b, L in enumerate(lens1)], np.int64)
    s2 = np.array([slot(b, int(L) - 1) for b, L in enumerate(lens2)], np.int64)
    for s in np.concatenate([s1, s2]):  # both new slots hold NaN before the steps
        pool_k.view(np.uint16)[s // 16, :, s % 16, :] = W.NAN_BF16
        pool_v.view(np.uint16)[s // 16, :, s % 16, :] = W.NAN_BF16
    kn = [W.normal(g, (len(lens2), hkv, d), "bf16") for _ in range(2)]
    vn = [W.normal(g, (len(lens2), hkv, d), "bf16") for _ in range(2)]
    q = [W.normal(g, (len(lens2), hq, d), "bf16") for _ in range(2)]

    def run(overlap):
        pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
        pk.kv_pool_set_launch_overlap(pool, overlap)
        kv, vv = pool_views(pool, nb, hkv, d, True)
        kv.copy_(dev(pool_k))
        vv.copy_(dev(pool_v))
        B = len(lens2)
        wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, 0)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        outs = [torch.empty((B, hq, d), dtype=torch.float32, device="cuda") for _ in range(2)]
        lses = [torch.empty((B, hq), dtype=torch.float32, device="cuda") for _ in range(2)]
        args = [(dev(q[i]), dev(kn[i]), dev(vn[i]), dev(s), dev(tables), maxb, dev(L))
                for i, (s, L) in enumerate(((s1, lens1), (s2, lens2)))]
        torch.cuda.synchronize()
        for i in range(2):  # back to back on one stream
            qq, kk, vvv, ss, tt, mb, ll = args[i]
            pk.paged_append_and_decode(pool, qq, kk, vvv, ss, tt, mb, ll, B, hq, 1 / math.sqrt(d),
                                       outs[i], pk.KV_F32, lses[i], 0, ws, wsb)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        res = [host(o) for o in outs] + [host(x) for x in lses] + [host(kv, like_bf16=True),
                                                                   host(vv, like_bf16=True)]
        pk.kv_pool_destroy(pool)
        return res

    a, b = run(False), run(True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                                      y.view(np.uint32) if y.dtype == np.float32 else y)
    pk_, pv_ = pool_k.copy(), pool_v.copy()
    oracle.append(pk_, pv_, kn[0], vn[0], s1)
    oracle.append(pk_, pv_, kn[1], vn[1], s2)
    np.testing.assert_array_equal(b[4], pk_)
    ref, ref_lse = oracle.paged_decode(pk_, pv_, tables, lens2, q[1], 1 / math.sqrt(d))
    assert_close_scaled(b[1], ref, 2e-3, "second step with launch overlap")
    np.testing.assert_allclose(b[3], ref_lse, atol=1e-3)
