"""A decode step whose per-step arguments live in pinned host memory.

On a GB300 the GPU reads and writes pinned host memory directly over
NVLink-C2C, so a serving loop can hand a step's query, new K/V rows, slots or
positions, lengths, order or schedule, and its output buffer to the library
without staging copies.  Each step path the benchmark drives must give the
bits the same call gives with device buffers: output, log-sum-exp and the
appended cache.  ("PagedAttention Nedir?", "Nasil Calisir?": the new token's
KV is written into its block, then the step attends all tokens.)"""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import dev, host, pool_views, read_linear, require_cuda
from test_gpu_append_decode import _setup
from test_gpu_contig import ContigCase

pytestmark = pytest.mark.gpu


def pinned(a: np.ndarray) -> torch.Tensor:
    """A pinned host copy of a numpy array (bf16 bit patterns travel as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a.copy()).pin_memory()


def _buffers(where, shapes):
    if where == "device":
        return [torch.empty(s, dtype=torch.float32, device="cuda") for s in shapes]
    return [torch.empty(s, dtype=torch.float32).pin_memory() for s in shapes]


def _paged_steps(where, case, scheduled, steps=3):
    """`steps` identical fused steps (append + decode) with launch overlap on."""
    lens, tables, pool_k, pool_v, slots, k_new, v_new, q = case
    place = dev if where == "device" else pinned
    nb, hkv, _, d = pool_k.shape
    B, hq, _ = q.shape
    maxb = tables.shape[1]
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    pk.kv_pool_set_launch_overlap(pool, True)
    kv, vv = pool_views(pool, nb, hkv, d, True)
    kv.copy_(dev(pool_k))
    vv.copy_(dev(pool_v))
    out, lse = _buffers(where, [(B, hq, d), (B, hq)])
    t_tables = dev(tables)  # the block tables are the cache's own state, on the device
    t_q, t_k, t_v, t_slots, t_lens = place(q), place(k_new), place(v_new), place(slots), place(lens)
    scale = 1.0 / math.sqrt(d)
    if scheduled:
        s = pk.kv_decode_schedule(lens, hkv, maxb, 3)  # few CTAs: several pieces each
        t_s = place(s)
        wsb = pk.kv_decode_schedule_workspace_size(s, hq, d)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        for _ in range(steps):
            pk.paged_decode_attention_scheduled(pool, t_q, t_tables, maxb, t_lens, B, hq, scale, s,
                                                t_s, out, pk.KV_F32, lse, ws, wsb, k_new=t_k,
                                                v_new=t_v, slot_mapping=t_slots)
    else:
        splits = pk.kv_decode_plan(lens, hkv, maxb)
        order = np.zeros(B, np.int32)
        pk.kv_decode_order(lens, order)
        t_order = place(order)
        wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        for _ in range(steps):
            pk.paged_append_and_decode(pool, t_q, t_k, t_v, t_slots, t_tables, maxb, t_lens, B, hq,
                                       scale, out, pk.KV_F32, lse, splits, ws, wsb,
                                       seq_order=t_order)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    res = (out.cpu().numpy().copy(), lse.cpu().numpy().copy(), host(kv, like_bf16=True),
           host(vv, like_bf16=True))
    pk.kv_pool_destroy(pool)
    return res


@pytest.mark.parametrize("scheduled", [False, True])
def test_paged_step_with_host_buffers_is_bit_identical(scheduled):
    """The grid-indexed fused step (longest-first order, planner's splits) and
    the balanced schedule with the append fused; 7 and 4 query heads per kv
    head."""
    require_cuda()
    hq = 32 if scheduled else 56
    lens = [1, 16, 17, 33, 300, 511, 1024, 1025, 2000, 47, 4096, 5]
    case = _setup(lens, hq, 8, 128, "bf16", seed=900 + int(scheduled))
    a = _paged_steps("device", case, scheduled)
    b = _paged_steps("host", case, scheduled)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert np.all(np.isfinite(a[0]))


def _contig_step(where, seed, fused):
    """Append one token per request at position L, then decode L + 1 tokens:
    contig_append_and_decode, or kv_contig_append then contig_decode_attention."""
    lens = [35, 17, 1, 300, 777, 64]
    c = ContigCase(lens, 800, hq=32, hkv=4, d=128, dtype="bf16", seed=seed)
    pk.kv_contig_set_launch_overlap(c.ctx, True)
    place = dev if where == "device" else pinned
    g = W.rng(seed + 1)
    k_new = W.normal(g, (c.B, c.hkv, c.d), "bf16")
    v_new = W.normal(g, (c.B, c.hkv, c.d), "bf16")
    for b, L in enumerate(c.lens):
        pk.kv_contig_ensure(c.ctx, int(c.req[b]), int(L) + 1)
    t_req = dev(c.req)  # request ids are the context's own state, on the device
    t_k, t_v, t_pos = place(k_new), place(v_new), place(c.lens.astype(np.int32))
    t_q, t_lens = place(c.q), place((c.lens + 1).astype(np.int32))
    out, lse = _buffers(where, [(c.B, c.hq, c.d), (c.B, c.hq)])
    maxb = -(-c.max_tokens // 16)
    wsb = pk.kv_decode_workspace_size(c.B, c.hq, c.hkv, c.d, maxb, 0)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    if fused:
        pk.contig_append_and_decode(c.ctx, t_q, t_k, t_v, t_req, t_lens, c.B, c.hq,
                                    1 / math.sqrt(c.d), out, pk.KV_F32, lse, 0, ws, wsb)
    else:
        pk.kv_contig_append(c.ctx, t_k, t_v, t_req, t_pos, c.B)
        pk.contig_decode_attention(c.ctx, t_q, t_req, t_lens, c.B, c.hq, 1 / math.sqrt(c.d), out,
                                   pk.KV_F32, lse, 0, ws, wsb)
    torch.cuda.synchronize()
    assert pk.kv_contig_get_device_error(c.ctx) == 0
    rows = []
    for b, L in enumerate(c.lens):
        k_ptr, v_ptr = pk.kv_contig_ptrs(c.ctx, int(c.req[b]))
        rows.append(read_linear(k_ptr, c.hkv, c.head_stride, int(L) + 1, c.d, True))
        rows.append(read_linear(v_ptr, c.hkv, c.head_stride, int(L) + 1, c.d, True))
    res = [out.cpu().numpy().copy(), lse.cpu().numpy().copy()] + rows
    c.close()
    return res


@pytest.mark.parametrize("fused", [True, False])
def test_contig_step_with_host_buffers_is_bit_identical(fused):
    """The contiguous path's step (the fused call, and the append and decode
    calls), its arguments in pinned host memory, against the same step with
    device buffers."""
    require_cuda()
    a = _contig_step("device", 910, fused)
    b = _contig_step("host", 910, fused)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert np.all(np.isfinite(a[0]))
