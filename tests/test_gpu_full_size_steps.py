"""Decode steps at full workload size, in the launch configurations the
benchmark times.

A decode step writes each sequence's new token into its block through the
slot mapping and then attends all of the sequence's tokens through its block
table ("PagedAttention Nedir?", section "PagedAttention Nasil Calisir?", steps
1-4).  The vAttention variant runs the same step over per-request virtual
ranges ("Makale Bulteni -- vAttention", section "Iddia ve Gerceklik:
vAttention").  Each test checks:
  * the pool after the step, bit for bit, against the oracle's append;
  * outputs on sampled (sequence, query head) items against the oracle, within
    2e-3 of the output scale (fp32 output), and bf16 output within that plus
    its own rounding;
  * two steps queued back to back with launch overlap on, as the benchmark runs
    them: the second must see the first's writes and nothing else.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, bf16_to_f64, dev, host, pool_views, require_cuda
from test_gpu_contig_pages import linear_oracle_items

pytestmark = pytest.mark.gpu


def _workload(name):
    cfg = W.CONFIGS[name]
    lens = W.decode_lengths(name)
    need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
    nb = int(math.ceil(cfg["pool_factor"] * need))
    inp = W.decode_inputs(name, nb)
    maxb = oracle.blocks_needed(cfg["len_hi"], 16)
    tables = oracle.build_block_tables(inp["lens"], 16, inp["perm"], maxb)
    g = W.rng(cfg["seed"] + 1000)   # the step's new tokens
    B, hkv, d = len(lens), cfg["num_kv_heads"], cfg["head_dim"]
    new = [(W.normal(g, (B, hkv, d), "bf16"), W.normal(g, (B, hkv, d), "bf16")) for _ in range(2)]
    return cfg, nb, inp, maxb, tables, new


def _items(B, hq, n, seed, lens):
    g = W.rng(seed)
    items = {(int(b), int(h)) for b, h in zip(g.integers(0, B, n), g.integers(0, hq, n))}
    items |= {(int(np.argmax(lens)), 0), (int(np.argmin(lens)), hq - 1)}
    return sorted(items)


def _pool(nb, hkv, d, pool_k, pool_v):
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    kv, vv = pool_views(pool, nb, hkv, d, True)
    kv.copy_(dev(pool_k))
    vv.copy_(dev(pool_v))
    return pool, kv, vv


def _assert_pool(kv, vv, exp_k, exp_v):
    assert torch.equal(kv, dev(exp_k)), "K pool differs from the oracle's append"
    assert torch.equal(vv, dev(exp_v)), "V pool differs from the oracle's append"


def _check_bf16_out(out_bf16, ref, items, what):
    got = np.array([bf16_to_f64(out_bf16[b, h]) for b, h in items])
    scale = float(np.max(np.abs(ref)))
    assert np.all(np.abs(got - ref) <= 2e-3 * scale + 2.0 ** -8 * np.abs(ref)), what


def test_llama3_8b_fused_step_full_size():
    """paged_append_and_decode with the planner's split count, the grid
    longest first and launch overlap on: the benchmark's default step."""
    require_cuda()
    cfg, nb, inp, maxb, tables, new = _workload("llama3_8b_decode")
    lens, q = inp["lens"], inp["q"]
    B, hq, hkv, d = len(lens), cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    scale = 1 / math.sqrt(d)
    last = lens.astype(np.int64) - 1
    slots = tables[np.arange(B), last // 16].astype(np.int64) * 16 + last % 16
    order = np.zeros(B, np.int32)
    pk.kv_decode_order(lens, order)
    splits = pk.kv_decode_plan(lens, hkv, maxb)
    pool, kv, vv = _pool(nb, hkv, d, inp["pool_k"], inp["pool_v"])
    try:
        pk.kv_pool_set_launch_overlap(pool, True)
        wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        t = dict(q=dev(q), tables=dev(tables), lens=dev(lens), slots=dev(slots), order=dev(order))
        k0, v0 = dev(new[0][0]), dev(new[0][1])
        outs = [torch.empty((B, hq, d), dtype=torch.float32, device="cuda") for _ in range(2)]
        lses = [torch.empty((B, hq), dtype=torch.float32, device="cuda") for _ in range(2)]
        out_bf16 = torch.empty((B, hq, d), dtype=torch.int16, device="cuda")
        torch.cuda.synchronize()
        # two identical steps back to back (the same token rewritten into the
        # same slot), then the benchmark's bf16-output form
        for o, l in zip(outs + [out_bf16], lses + [None]):
            pk.paged_append_and_decode(pool, t["q"], k0, v0, t["slots"], t["tables"], maxb,
                                       t["lens"], B, hq, scale, o,
                                       pk.KV_F32 if o.dtype == torch.float32 else pk.KV_BF16, l,
                                       splits, ws, wsb, seq_order=t["order"])
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        exp_k, exp_v = inp["pool_k"].copy(), inp["pool_v"].copy()
        oracle.append(exp_k, exp_v, new[0][0], new[0][1], slots)
        _assert_pool(kv, vv, exp_k, exp_v)
        o0, o1 = host(outs[0]), host(outs[1])
        np.testing.assert_array_equal(o0.view(np.uint32), o1.view(np.uint32))
        np.testing.assert_array_equal(host(lses[0]).view(np.uint32), host(lses[1]).view(np.uint32))
        items = _items(B, hq, 128, 5, lens)
        ref, ref_lse = oracle.paged_decode(exp_k, exp_v, tables, lens, q, scale, items=items)
        assert_close_scaled(np.array([o0[b, h] for b, h in items]), ref, 2e-3,
                            "llama3-8b fused step, sampled")
        np.testing.assert_allclose([host(lses[0])[b, h] for b, h in items], ref_lse, atol=1e-3)
        assert np.all(np.isfinite(o0))
        _check_bf16_out(host(out_bf16, like_bf16=True), ref, items, "bf16 output")
    finally:
        pk.kv_pool_destroy(pool)


@pytest.mark.slow
def test_yi6b_step_full_size_scheduled_grid_and_contiguous():
    """The Yi-6B-shaped step at full size (contexts 32K-192K) three ways:
      1. paged, balanced schedule with the append fused (the benchmark's path
         for this workload), checked against the oracle and the pool bit for bit;
      2. paged, grid-indexed plan from the planner over the same pool;
      3. contiguous: the same logical content in per-request virtual ranges
         (each head region 4 to 24 mapped 2 MiB pages), two append + decode
         steps back to back with launch overlap on.  Step 1 must equal (2) bit
         for bit (same split plan); step 2 attends the token step 1 appended
         and one more, checked against the oracle's linear-layout decode."""
    require_cuda()
    cfg, nb, inp, maxb, tables, new = _workload("yi6b_long_decode")
    lens, q = inp["lens"], inp["q"]
    B, hq, hkv, d = len(lens), cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    scale = 1 / math.sqrt(d)
    last = lens.astype(np.int64) - 1
    slots = tables[np.arange(B), last // 16].astype(np.int64) * 16 + last % 16
    items = _items(B, hq, 24, 6, lens)
    t_q, t_lens, t_tables = dev(q), dev(lens), dev(tables)
    k0, v0 = new[0]

    # ---- 1. balanced schedule, the append fused
    pool, kv, vv = _pool(nb, hkv, d, inp["pool_k"], inp["pool_v"])
    try:
        pk.kv_pool_set_launch_overlap(pool, True)
        h_sched = pk.kv_decode_schedule(lens, hkv, maxb)
        assert int(h_sched[4]) == 1   # runs long enough for the deep ring
        wss = pk.kv_decode_schedule_workspace_size(h_sched, hq, d)
        ws = torch.empty(max(wss // 4, 1), dtype=torch.float32, device="cuda")
        o_s = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
        l_s = torch.empty((B, hq), dtype=torch.float32, device="cuda")
        pk.paged_decode_attention_scheduled(pool, t_q, t_tables, maxb, t_lens, B, hq, scale, h_sched,
                                            dev(h_sched), o_s, pk.KV_F32, l_s, ws, wss,
                                            k_new=dev(k0), v_new=dev(new[0][1]),
                                            slot_mapping=dev(slots))
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        exp_k, exp_v = inp["pool_k"].copy(), inp["pool_v"].copy()
        oracle.append(exp_k, exp_v, k0, v0, slots)
        _assert_pool(kv, vv, exp_k, exp_v)
        ref, ref_lse = oracle.paged_decode(exp_k, exp_v, tables, lens, q, scale, items=items)
        o_s, l_s = host(o_s), host(l_s)
        assert_close_scaled(np.array([o_s[b, h] for b, h in items]), ref, 2e-3,
                            "yi-6b balanced schedule, sampled")
        np.testing.assert_allclose([l_s[b, h] for b, h in items], ref_lse, atol=1e-3)
        assert np.all(np.isfinite(o_s))

        # ---- 2. grid-indexed plan over the same pool (the token already appended)
        splits = pk.kv_decode_plan(lens, hkv, maxb)
        wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        o_g = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
        l_g = torch.empty((B, hq), dtype=torch.float32, device="cuda")
        pk.paged_decode_attention(pool, t_q, t_tables, maxb, t_lens, B, hq, scale, o_g, pk.KV_F32,
                                  l_g, splits, ws, wsb)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(pool) == 0
        o_g, l_g = host(o_g), host(l_g)
        assert_close_scaled(np.array([o_g[b, h] for b, h in items]), ref, 2e-3,
                            "yi-6b grid plan, sampled")
        assert_close_scaled(o_g, o_s, 1e-5, "grid plan vs balanced schedule")
    finally:
        pk.kv_pool_destroy(pool)
    del exp_k, exp_v, kv, vv

    # ---- 3. contiguous: logical content = each sequence's blocks in table order
    K, V = [], []
    for b, L in enumerate(lens):
        j = np.arange(int(L))
        K.append(np.ascontiguousarray(inp["pool_k"][tables[b, j // 16], :, j % 16]))
        V.append(np.ascontiguousarray(inp["pool_v"][tables[b, j // 16], :, j % 16]))
        K[b][-1], V[b][-1] = k0[b], v0[b]     # the token step 1 writes
    # reserved at the workload's maximum context, so the contiguous decode
    # plans on the same table width (and partitions) as the paged grid plan
    assert int(lens.max()) + 1 <= cfg["len_hi"]
    ctx = pk.kv_contig_create(B, cfg["len_hi"], hkv, d, pk.KV_BF16)
    try:
        pk.kv_contig_set_launch_overlap(ctx, True)
        req = dev(np.arange(B, dtype=np.int32))
        for b, L in enumerate(lens):
            pk.kv_contig_reserve(ctx, b)
            pk.kv_contig_ensure(ctx, b, int(L) + 1)
            pk.kv_contig_append(ctx, dev(K[b][:-1]), dev(V[b][:-1]),
                                dev(np.full(int(L) - 1, b, np.int32)),
                                dev(np.arange(int(L) - 1, dtype=np.int32)), int(L) - 1)
            torch.cuda.synchronize()
        assert pk.kv_contig_get_device_error(ctx) == 0
        k1, v1 = new[1]
        steps = [(k0, v0, last.astype(np.int32), lens), (k1, v1, lens.copy(), lens + 1)]
        dargs = [(dev(k), dev(v), dev(pos), dev(ln.astype(np.int32))) for k, v, pos, ln in steps]
        outs = [torch.empty((B, hq, d), dtype=torch.float32, device="cuda") for _ in range(2)]
        lses = [torch.empty((B, hq), dtype=torch.float32, device="cuda") for _ in range(2)]
        torch.cuda.synchronize()
        for (k, v, pos, ln), o, l in zip(dargs, outs, lses):   # back to back, overlapped
            pk.kv_contig_append(ctx, k, v, req, pos, B)
            pk.contig_decode_attention(ctx, t_q, req, ln, B, hq, scale, o, pk.KV_F32, l, splits,
                                       ws, wsb)
        torch.cuda.synchronize()
        assert pk.kv_contig_get_device_error(ctx) == 0
        oc1, lc1 = host(outs[0]), host(lses[0])
        np.testing.assert_array_equal(oc1.view(np.uint32), o_g.view(np.uint32))
        np.testing.assert_array_equal(lc1.view(np.uint32), l_g.view(np.uint32))
        ref1, _ = linear_oracle_items(K, V, lens, q, items, scale)
        assert_close_scaled(np.array([oc1[b, h] for b, h in items]), ref1, 2e-3,
                            "contiguous step 1, sampled")
        for b in range(B):
            K[b] = np.concatenate([K[b], k1[b:b + 1]])
            V[b] = np.concatenate([V[b], v1[b:b + 1]])
        ref2, ref2_lse = linear_oracle_items(K, V, lens + 1, q, items, scale)
        oc2, lc2 = host(outs[1]), host(lses[1])
        assert_close_scaled(np.array([oc2[b, h] for b, h in items]), ref2, 2e-3,
                            "contiguous step 2, sampled")
        np.testing.assert_allclose([lc2[b, h] for b, h in items], ref2_lse, atol=1e-3)
        assert np.all(np.isfinite(oc2))
    finally:
        pk.kv_contig_destroy(ctx)
