"""Failure detection, exercised without faulting or hanging a GPU.

Every pipeline wait inside the kernels is bounded: when one runs out the
kernel records KV_DEVERR_TIMEOUT, runs to its end, and the host reads
KV_ERR_TIMEOUT; the context stays usable.  These tests shorten the limit with
kv_debug_set_wait_limit_ns(0), so that any wait not satisfied at its first
poll gives up, then check the reported status and that the next call with
the default limit is correct again (the split-merge counters a timed-out call may
leave behind are cleared by kv_get_device_error).  A warp's wait for its own
copies and tensor-core operations before its CTA ends keeps the full limit, so
nothing is in flight when the kernels exit.

The contiguous path's page creation is made to fail on the host
(kv_debug_fail_page_create): kv_contig_ensure must return KV_ERR_OOM and leave
nothing of that call mapped ("Makale Bulteni -- vAttention", section "Iddia ve
Gerceklik: vAttention": physical pages are created and mapped on demand).
"""
import contextlib
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, dev, host, read_linear, require_cuda
from test_gpu_decode import random_case
from test_gpu_prefill import PrefillCase

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 0x4


@contextlib.contextmanager
def short_waits():
    pk.kv_debug_set_wait_limit_ns(0)
    try:
        yield
    finally:
        pk.kv_debug_set_wait_limit_ns(pk.KV_WAIT_LIMIT_DEFAULT_NS)


def _lens(n, seed):
    return W.rng(seed).integers(300, 4000, size=n, endpoint=True).astype(np.int32)


def _decode(c, splits, out, lse):
    maxb = c.tables.shape[1]
    wsb = pk.kv_decode_workspace_size(c.B, c.hq, c.hkv, c.d, maxb, splits)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    pk.paged_decode_attention(c.pool, c.t_q, c.t_tables, maxb, c.t_lens, c.B, c.hq,
                              1 / math.sqrt(c.d), out, pk.KV_F32, lse, splits, ws, wsb)
    torch.cuda.synchronize()


def test_decode_wait_timeout_is_reported_and_the_next_call_is_correct():
    require_cuda()
    c = random_case(_lens(24, 500), hq=32, hkv=8, d=128, dtype="bf16", seed=501)
    try:
        ref, ref_lse = c.oracle()
        first, first_lse = c.run(2)          # two splits: the fused merge and its counters
        assert_close_scaled(first, ref, 2e-3, "before the timeout")
        out = torch.empty((c.B, c.hq, c.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((c.B, c.hq), dtype=torch.float32, device="cuda")
        with short_waits():
            _decode(c, 2, out, lse)
        assert pk.kv_get_device_error(c.pool) & TIMEOUT_BIT
        again, again_lse = c.run(2)          # asserts a clean device error word
        np.testing.assert_array_equal(again, first)
        np.testing.assert_array_equal(again_lse, first_lse)
    finally:
        c.close()


@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 4)])
def test_scheduled_decode_wait_timeout_then_correct(hq, hkv):
    """The balanced-schedule kernel (4 and 8 query heads per kv head):
    consumers and the producer meet on a named barrier at every piece
    boundary whether or not a wait ran out."""
    require_cuda()
    c = random_case(_lens(16, 502), hq=hq, hkv=hkv, d=128, dtype="bf16", seed=503 + hkv)
    try:
        maxb = c.tables.shape[1]
        h_sched = pk.kv_decode_schedule(c.lens, c.hkv, maxb)
        d_sched = dev(h_sched)
        wsb = pk.kv_decode_schedule_workspace_size(h_sched, c.hq, c.d)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")

        def run():
            out = torch.empty((c.B, c.hq, c.d), dtype=torch.float32, device="cuda")
            pk.paged_decode_attention_scheduled(c.pool, c.t_q, c.t_tables, maxb, c.t_lens, c.B,
                                                c.hq, 1 / math.sqrt(c.d), h_sched, d_sched, out,
                                                pk.KV_F32, None, ws, wsb)
            torch.cuda.synchronize()
            return host(out).astype(np.float64)

        with short_waits():
            run()
        assert pk.kv_get_device_error(c.pool) & TIMEOUT_BIT
        out = run()
        assert pk.kv_get_device_error(c.pool) == 0
        ref, _ = c.oracle()
        assert_close_scaled(out, ref, 2e-3, "scheduled decode after a timeout")
    finally:
        c.close()


def test_prefill_wait_timeout_is_reported_and_the_next_call_is_correct():
    """The tcgen05 prefill: after a timed-out call (its MMAs drained before the
    tensor memory is freed) the same call gives the oracle's result."""
    c = PrefillCase([300, 0, 1000], [200, 256, 77], hq=8, hkv=2, seed=504)
    try:
        out = torch.empty((c.total_q, c.hq, c.d), dtype=torch.float32, device="cuda")
        with short_waits():
            pk.paged_prefill_attention(c.pool, dev(c.q), dev(c.cu), c.total_q,
                                       int(c.chunk.max()), dev(c.tables), c.maxb, dev(c.lens),
                                       c.B, c.hq, 1 / math.sqrt(c.d), out, pk.KV_F32, None)
            torch.cuda.synchronize()
        assert pk.kv_get_device_error(c.pool) & TIMEOUT_BIT
        got, lse = c.run()                    # asserts a clean device error word
        ref, ref_lse = c.oracle()
        assert_close_scaled(got, ref, 2e-3, "prefill after a timeout")
        np.testing.assert_allclose(lse, ref_lse, atol=1e-3)
    finally:
        c.close()


def test_timeout_status_maps_to_kv_err_timeout():
    require_cuda()
    c = random_case(_lens(8, 505), hq=32, hkv=8, d=128, dtype="bf16", seed=506)
    try:
        out = torch.empty((c.B, c.hq, c.d), dtype=torch.float32, device="cuda")
        with short_waits():
            _decode(c, 1, out, None)
        # the raw call: status KV_ERR_TIMEOUT (-6) with the timeout bit in the code
        import ctypes
        code = ctypes.c_int()
        st = pk.lib().kv_get_device_error(c.pool, ctypes.byref(code), None)
        assert st == -6 and code.value & TIMEOUT_BIT
        st = pk.lib().kv_get_device_error(c.pool, ctypes.byref(code), None)
        assert st == 0 and code.value == 0   # read and cleared
    finally:
        c.close()


def test_contig_page_creation_failure_leaves_nothing_mapped():
    require_cuda()
    ctx = pk.kv_contig_create(2, 100000, 4, 128, pk.KV_BF16)
    try:
        _, page, _ = pk.kv_contig_layout(ctx)
        tpp = page // (128 * 2)
        pk.kv_contig_reserve(ctx, 0)
        pk.kv_contig_ensure(ctx, 0, tpp)                 # one page per head region: 8 pages
        before = pk.kv_contig_stats(ctx, 0)
        assert before == (tpp, 8 * page)
        pk.kv_debug_fail_page_create(5)                  # the sixth creation from now fails
        with pytest.raises(pk.KVError) as e:
            pk.kv_contig_ensure(ctx, 0, 3 * tpp)         # needs 16 more pages
        assert e.value.status == -2                      # KV_ERR_OOM
        assert pk.kv_contig_stats(ctx, 0) == before      # the five it had mapped are undone
        # the failure was used up: the same call now succeeds and the range works
        pk.kv_contig_ensure(ctx, 0, 3 * tpp)
        assert pk.kv_contig_stats(ctx, 0) == (3 * tpp, 24 * page)
        k = W.normal(W.rng(7), (2, 4, 128), "bf16")
        pos = np.array([tpp - 1, 3 * tpp - 1], np.int32)
        pk.kv_contig_append(ctx, dev(k), dev(k), dev(np.zeros(2, np.int32)), dev(pos), 2)
        torch.cuda.synchronize()
        assert pk.kv_contig_get_device_error(ctx) == 0
        k_ptr, _ = pk.kv_contig_ptrs(ctx, 0)
        hs, _, _ = pk.kv_contig_layout(ctx)
        got = read_linear(k_ptr, 4, hs, 3 * tpp, 128, True)
        np.testing.assert_array_equal(got[:, pos], k.transpose(1, 0, 2))
    finally:
        pk.kv_debug_fail_page_create(-1)
        pk.kv_contig_destroy(ctx)
