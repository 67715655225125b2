"""IEEE half-precision (KV_F16) pools on the GPU against the oracle.

The boundary's element types include fp16 beside fp32 and bf16.  An fp16 pool
takes fp16 q / k_new / v_new and writes fp32 or fp16 output.  Checked here:
  * the append, bit for bit, every untouched slot keeping its NaN sentinel;
  * decode on the CUDA-core kernel (1-2 query heads per kv head, head_dim 64)
    and the tensor-core kernel (3-8 heads, head_dim 128: fp16 QK^T and one PV
    product with fp16 weights), ragged lengths with NaN-poisoned unused slots,
    several split plans, within 2e-3 of the output scale (fp32 output; fp16
    output also allows its own rounding, 2^-11 relative);
  * the fused decode step (append folded into the decode kernel), bit for bit
    against kv_append + decode and against the oracle;
  * the chunked causal prefill (fp16 QK^T and PV on tcgen05, no V conversion);
  * the contiguous path, bit-identical to the paged decode under the same plan.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, dev, require_cuda, view

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _f16_pool_views(pool, nb, hkv, d):
    kp, vp = pk.kv_pool_ptrs(pool)
    shape = (nb, hkv, 16, d)
    return view(kp, shape, False, "<f2"), view(vp, shape, False, "<f2")


def _h(t):
    return t.detach().cpu().numpy()


def _poisoned_case(lens, hq, hkv, d, seed, extra=3):
    g = W.rng(seed)
    lens = np.asarray(lens, np.int32)
    need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
    nb = need + extra
    maxb = max(1, max(oracle.blocks_needed(int(L), 16) for L in lens))
    tables = oracle.build_block_tables(lens, 16, W.permutation(g, nb), maxb)
    pool_k = W.normal(g, (nb, hkv, 16, d), "f16")
    pool_v = W.normal(g, (nb, hkv, 16, d), "f16")
    used = np.zeros((nb, 16), bool)
    for b, L in enumerate(lens):
        for j in range(L):
            used[tables[b, j // 16], j % 16] = True
    pool_k.view(np.uint16).transpose(0, 2, 1, 3)[~used] = W.NAN_F16
    pool_v.view(np.uint16).transpose(0, 2, 1, 3)[~used] = W.NAN_F16
    q = W.normal(g, (len(lens), hq, d), "f16")
    return lens, tables, pool_k, pool_v, q, nb


def _pool_with(pool_k, pool_v):
    nb, hkv, _, d = pool_k.shape
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_F16)
    kv, vv = _f16_pool_views(pool, nb, hkv, d)
    kv.copy_(dev(pool_k))
    vv.copy_(dev(pool_v))
    return pool, kv, vv


def _decode(pool, q, tables, lens, hkv, splits, out_f16=False):
    B, hq, d = q.shape
    maxb = tables.shape[1]
    out = torch.empty((B, hq, d), dtype=torch.float16 if out_f16 else torch.float32, device="cuda")
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    pk.paged_decode_attention(pool, dev(q), dev(tables), maxb, dev(lens), B, hq, 1 / math.sqrt(d),
                              out, pk.KV_F16 if out_f16 else pk.KV_F32, lse, splits, ws, wsb)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    return _h(out).astype(np.float64), _h(lse).astype(np.float64)


def test_f16_append_bit_exact_with_sentinel():
    require_cuda()
    nb, hkv, d, T = 40, 4, 128, 300
    g = W.rng(601)
    slots = g.permutation(nb * 16)[:T].astype(np.int64)
    slots[::13] = -1
    k = W.normal(g, (T, hkv, d), "f16")
    v = W.normal(g, (T, hkv, d), "f16")
    ref_k = W.empty_pool(nb, hkv, d, "f16", W.NAN_F16)
    ref_v = W.empty_pool(nb, hkv, d, "f16", W.NAN_F16)
    oracle.append(ref_k, ref_v, k, v, slots)
    pool, kv, vv = _pool_with(W.empty_pool(nb, hkv, d, "f16", W.NAN_F16),
                              W.empty_pool(nb, hkv, d, "f16", W.NAN_F16))
    try:
        pk.kv_append(pool, dev(k), dev(v), dev(slots), T)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        np.testing.assert_array_equal(_h(kv).view(np.uint16), ref_k.view(np.uint16))
        np.testing.assert_array_equal(_h(vv).view(np.uint16), ref_v.view(np.uint16))
    finally:
        pk.kv_pool_destroy(pool)


@pytest.mark.parametrize("g,d", [(1, 64), (2, 128), (4, 64), (3, 128), (4, 128), (8, 128)])
def test_f16_decode_matches_oracle(g, d):
    require_cuda()
    hkv = 2
    lens, tables, pool_k, pool_v, q, _ = _poisoned_case([1, 15, 16, 17, 35, 300, 777, 0, 64],
                                                        hq=g * hkv, hkv=hkv, d=d, seed=610 + g + d)
    ref, ref_lse = oracle.paged_decode(pool_k, pool_v, tables, lens, q, 1 / math.sqrt(d))
    pool, _, _ = _pool_with(pool_k, pool_v)
    try:
        for splits in (1, 4, 0):
            out, lse = _decode(pool, q, tables, lens, hkv, splits)
            assert_close_scaled(out, ref, TOL, f"f16 g={g} d={d} splits={splits}")
            fin = np.isfinite(ref_lse)
            np.testing.assert_allclose(lse[fin], ref_lse[fin], atol=1e-3)
            assert np.all(np.isneginf(lse[~fin]))
        out16, _ = _decode(pool, q, tables, lens, hkv, 0, out_f16=True)
        scale = np.max(np.abs(ref))
        assert np.all(np.abs(out16 - ref) <= TOL * scale + 2.0 ** -11 * np.abs(ref))
    finally:
        pk.kv_pool_destroy(pool)


def test_f16_fused_step_equals_append_then_decode_and_oracle():
    require_cuda()
    hq, hkv, d = 32, 8, 128
    lens, tables, pool_k, pool_v, q, nb = _poisoned_case([40, 1500, 17, 3000, 256, 1],
                                                         hq=hq, hkv=hkv, d=d, seed=620)
    g = W.rng(621)
    k_new = W.normal(g, (len(lens), hkv, d), "f16")
    v_new = W.normal(g, (len(lens), hkv, d), "f16")
    slots = np.array([int(tables[b, (L - 1) // 16]) * 16 + (L - 1) % 16 for b, L in enumerate(lens)],
                     np.int64)
    B, maxb = len(lens), tables.shape[1]
    results = []
    for fused in (True, False):
        pool, kv, vv = _pool_with(pool_k, pool_v)
        try:
            out = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
            wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, 2)
            ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
            args = (dev(tables), maxb, dev(lens), B, hq, 1 / math.sqrt(d), out, pk.KV_F32, None, 2,
                    ws, wsb)
            if fused:
                pk.paged_append_and_decode(pool, dev(q), dev(k_new), dev(v_new), dev(slots), *args)
            else:
                pk.kv_append(pool, dev(k_new), dev(v_new), dev(slots), B)
                pk.paged_decode_attention(pool, dev(q), *args)
            torch.cuda.synchronize()
            assert pk.kv_get_device_error(pool) == 0
            results.append((_h(out), _h(kv).view(np.uint16), _h(vv).view(np.uint16)))
        finally:
            pk.kv_pool_destroy(pool)
    for a, b in zip(results[0], results[1]):
        np.testing.assert_array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                      b.view(np.uint32) if b.dtype == np.float32 else b)
    ref_k, ref_v = pool_k.copy(), pool_v.copy()
    oracle.append(ref_k, ref_v, k_new, v_new, slots)
    np.testing.assert_array_equal(results[0][1], ref_k.view(np.uint16))
    ref, _ = oracle.paged_decode(ref_k, ref_v, tables, lens, q, 1 / math.sqrt(d))
    assert_close_scaled(results[0][0], ref, TOL, "f16 fused step")


@pytest.mark.parametrize("cached,chunk", [([0], [200]), ([37, 512, 300], [77, 256, 130])])
def test_f16_prefill_matches_oracle(cached, chunk):
    require_cuda()
    hq, hkv, d = 8, 2, 128
    g = W.rng(630 + len(chunk))
    cached = np.asarray(cached, np.int32)
    chunk = np.asarray(chunk, np.int32)
    lens = (cached + chunk).astype(np.int32)
    need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
    nb = need + 3
    maxb = max(oracle.blocks_needed(int(L), 16) for L in lens)
    tables = oracle.build_block_tables(lens, 16, W.permutation(g, nb), maxb)
    pool_k = W.normal(g, (nb, hkv, 16, d), "f16")
    pool_v = W.normal(g, (nb, hkv, 16, d), "f16")
    used = np.zeros((nb, 16), bool)
    for b, L in enumerate(lens):
        for j in range(L):
            used[tables[b, j // 16], j % 16] = True
    pool_k.view(np.uint16).transpose(0, 2, 1, 3)[~used] = W.NAN_F16
    pool_v.view(np.uint16).transpose(0, 2, 1, 3)[~used] = W.NAN_F16
    T = int(chunk.sum())
    q = W.normal(g, (T, hq, d), "f16")
    cu = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    ref, ref_lse = oracle.paged_prefill(pool_k, pool_v, tables, lens, cu, q, 1 / math.sqrt(d))
    pool, _, _ = _pool_with(pool_k, pool_v)
    try:
        for out_f16 in (False, True):
            out = torch.full((T, hq, d), float("nan"),
                             dtype=torch.float16 if out_f16 else torch.float32, device="cuda")
            lse = torch.empty((T, hq), dtype=torch.float32, device="cuda")
            pk.paged_prefill_attention(pool, dev(q), dev(cu), T, int(chunk.max()), dev(tables), maxb,
                                       dev(lens), len(lens), hq, 1 / math.sqrt(d), out,
                                       pk.KV_F16 if out_f16 else pk.KV_F32, lse)
            torch.cuda.synchronize()
            assert pk.kv_get_device_error(pool) == 0
            got = _h(out).astype(np.float64)
            if out_f16:
                scale = np.max(np.abs(ref))
                assert np.all(np.abs(got - ref) <= TOL * scale + 2.0 ** -11 * np.abs(ref))
            else:
                assert_close_scaled(got, ref, TOL, f"f16 prefill cached={cached.tolist()}")
                np.testing.assert_allclose(_h(lse), ref_lse, atol=1e-3)
    finally:
        pk.kv_pool_destroy(pool)


@pytest.mark.parametrize("hq", [4, 32])   # CUDA-core and tensor-core kernels
def test_f16_contiguous_equals_paged(hq):
    require_cuda()
    hkv, d = 4, 128
    lens = np.array([35, 17, 1, 300, 777, 64], np.int32)
    B = len(lens)
    g = W.rng(640 + hq)
    K = [W.normal(g, (int(L), hkv, d), "f16") for L in lens]
    V = [W.normal(g, (int(L), hkv, d), "f16") for L in lens]
    q = W.normal(g, (B, hq, d), "f16")
    ctx = pk.kv_contig_create(B, 800, hkv, d, pk.KV_F16)
    pool = None
    try:
        for b, L in enumerate(lens):
            pk.kv_contig_reserve(ctx, b)
            pk.kv_contig_ensure(ctx, b, int(L))
            pk.kv_contig_append(ctx, dev(K[b]), dev(V[b]), dev(np.full(int(L), b, np.int32)),
                                dev(np.arange(int(L), dtype=np.int32)), int(L))
        maxb = -(-800 // 16)
        need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
        tables = oracle.build_block_tables(lens, 16, W.permutation(g, need + 5), maxb)
        pool = pk.kv_pool_create(need + 5, 16, hkv, d, pk.KV_F16)
        for b, L in enumerate(lens):
            j = np.arange(int(L))
            pk.kv_append(pool, dev(K[b]), dev(V[b]),
                         dev(tables[b, j // 16].astype(np.int64) * 16 + j % 16), int(L))
        n = int(lens.max())
        kb = [np.zeros((hkv, n, d), np.float16) for _ in range(B)]
        vb = [np.zeros((hkv, n, d), np.float16) for _ in range(B)]
        for b, L in enumerate(lens):
            kb[b][:, :L] = K[b].transpose(1, 0, 2)
            vb[b][:, :L] = V[b].transpose(1, 0, 2)
        ref, _ = oracle.linear_decode(kb, vb, np.arange(B), lens, q, 1 / math.sqrt(d))
        for splits in (1, 4, 0):
            wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
            ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
            oc = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
            op = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
            pk.contig_decode_attention(ctx, dev(q), dev(np.arange(B, dtype=np.int32)), dev(lens), B, hq,
                                       1 / math.sqrt(d), oc, pk.KV_F32, None, splits, ws, wsb)
            pk.paged_decode_attention(pool, dev(q), dev(tables), maxb, dev(lens), B, hq,
                                      1 / math.sqrt(d), op, pk.KV_F32, None, splits, ws, wsb)
            torch.cuda.synchronize()
            assert pk.kv_contig_get_device_error(ctx) == 0
            assert pk.kv_get_device_error(pool) == 0
            np.testing.assert_array_equal(_h(oc).view(np.uint32), _h(op).view(np.uint32))
            assert_close_scaled(_h(oc), ref, TOL, f"f16 contiguous splits={splits}")
    finally:
        if pool is not None:
            pk.kv_pool_destroy(pool)
        pk.kv_contig_destroy(ctx)


def test_f16_llama3_8b_step_full_size():
    """The benchmark's fp16 Llama-3-8B-shaped step at full size
    (`bench.py --kv-dtype f16`): paged_append_and_decode with the planner's
    split count, the grid longest first and launch overlap on.  The pool after
    the step bit for bit against the oracle's append; sampled (sequence, query
    head) items against the oracle."""
    require_cuda()
    name = "llama3_8b_decode"
    cfg = W.CONFIGS[name]
    lens = W.decode_lengths(name)
    nb = int(math.ceil(cfg["pool_factor"] * sum(oracle.blocks_needed(int(L), 16) for L in lens)))
    inp = W.decode_inputs(name, nb, dtype="f16")
    maxb = oracle.blocks_needed(cfg["len_hi"], 16)
    tables = oracle.build_block_tables(lens, 16, inp["perm"], maxb)
    B, hq, hkv, d = len(lens), cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    g = W.rng(cfg["seed"] + 1000)
    k_new = W.normal(g, (B, hkv, d), "f16")
    v_new = W.normal(g, (B, hkv, d), "f16")
    last = lens.astype(np.int64) - 1
    slots = tables[np.arange(B), last // 16].astype(np.int64) * 16 + last % 16
    order = np.zeros(B, np.int32)
    pk.kv_decode_order(lens, order)
    splits = pk.kv_decode_plan(lens, hkv, maxb)
    scale = 1 / math.sqrt(d)
    pool, kv, vv = _pool_with(inp["pool_k"], inp["pool_v"])
    try:
        pk.kv_pool_set_launch_overlap(pool, True)
        wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        out = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
        lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
        pk.paged_append_and_decode(pool, dev(inp["q"]), dev(k_new), dev(v_new), dev(slots),
                                   dev(tables), maxb, dev(lens), B, hq, scale, out, pk.KV_F32, lse,
                                   splits, ws, wsb, seq_order=dev(order))
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        exp_k, exp_v = inp["pool_k"].copy(), inp["pool_v"].copy()
        oracle.append(exp_k, exp_v, k_new, v_new, slots)
        np.testing.assert_array_equal(_h(kv).view(np.uint16), exp_k.view(np.uint16))
        np.testing.assert_array_equal(_h(vv).view(np.uint16), exp_v.view(np.uint16))
        gi = W.rng(7)
        items = sorted({(int(b), int(h)) for b, h in zip(gi.integers(0, B, 128), gi.integers(0, hq, 128))})
        ref, ref_lse = oracle.paged_decode(exp_k, exp_v, tables, lens, inp["q"], scale, items=items)
        o = _h(out)
        assert_close_scaled(np.array([o[b, h] for b, h in items]), ref, TOL, "f16 llama3-8b step")
        np.testing.assert_allclose([_h(lse)[b, h] for b, h in items], ref_lse, atol=1e-3)
        assert np.all(np.isfinite(o))
    finally:
        pk.kv_pool_destroy(pool)


@pytest.mark.slow
def test_f16_yi34b_prefill_full_size_sampled():
    """The benchmark's fp16 Yi-34B-shaped prefill at full size (4 x (8192
    cached + 2048 new) tokens, 56 query / 8 kv heads): one complete 256-row
    slab for every query head, every row of the first query tile, and random
    items, against the oracle."""
    require_cuda()
    cfg = W.CONFIGS["yi34b_prefill"]
    B, hq, hkv, d = cfg["batch"], cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    c_len, t_len = cfg["cached_len"], cfg["chunk_len"]
    L = c_len + t_len
    maxb = oracle.blocks_needed(L, 16)
    nb = B * maxb
    inp = W.prefill_inputs("yi34b_prefill", nb, dtype="f16")
    lens = np.full(B, L, np.int32)
    tables = oracle.build_block_tables(lens, 16, inp["perm"], maxb)
    slots = []
    for b in range(B):
        pos = np.arange(c_len, L)
        slots.append(tables[b, pos // 16].astype(np.int64) * 16 + pos % 16)
    slots = np.concatenate(slots)
    T = B * t_len
    cu = np.arange(0, T + 1, t_len, dtype=np.int32)
    scale = 1 / math.sqrt(d)
    pool, _, _ = _pool_with(inp["pool_k"], inp["pool_v"])
    try:
        pk.kv_append(pool, dev(inp["k_new"]), dev(inp["v_new"]), dev(slots), T)
        out = torch.empty((T, hq, d), dtype=torch.float32, device="cuda")
        lse = torch.empty((T, hq), dtype=torch.float32, device="cuda")
        pk.paged_prefill_attention(pool, dev(inp["q"]), dev(cu), T, t_len, dev(tables), maxb,
                                   dev(lens), B, hq, scale, out, pk.KV_F32, lse)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        ref_k, ref_v = inp["pool_k"].copy(), inp["pool_v"].copy()
        oracle.append(ref_k, ref_v, inp["k_new"], inp["v_new"], slots)
        gi = W.rng(8)
        items = {(int(r), int(h)) for r, h in zip(gi.integers(0, T, 48), gi.integers(0, hq, 48))}
        items |= {(2 * t_len + t_len - 256 + r, h) for r in range(256) for h in range(hq)}
        items |= {(r, h) for r in range(128) for h in range(hq)}
        items = sorted(items)
        ref, ref_lse = oracle.paged_prefill(ref_k, ref_v, tables, lens, cu, inp["q"], scale,
                                            items=items)
        o, l = _h(out), _h(lse)
        assert_close_scaled(np.array([o[r, h] for r, h in items]), ref, TOL, "f16 yi34b prefill")
        np.testing.assert_allclose([l[r, h] for r, h in items], ref_lse, atol=1e-3)
    finally:
        pk.kv_pool_destroy(pool)
