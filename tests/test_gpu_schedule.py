"""Decode on a balanced schedule (kv_decode_schedule +
paged_decode_attention_scheduled) against the oracle, against the
grid-indexed decode, and with the decode step's append fused in.

The maths is the pages' ("PagedAttention Nedir?", "Nasil Calisir?": the query
attends every token of its sequence through the block table); only the cut of
each sequence into split-KV partitions differs, so outputs agree with the
oracle within the bf16 tolerance and with each other within rounding.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, dev, host, pool_views, require_cuda
from test_gpu_append_decode import _setup
from test_gpu_decode import TOL, _full_decode_case, _sample_items, random_case

pytestmark = pytest.mark.gpu


def _sched_run(case, num_sms, lens_dev=None, expect_err=0, flags=0, ring_stages=0):
    """Scheduled decode of a test_gpu_decode Case (no append)."""
    hq, hkv, d = case.hq, case.hkv, case.d
    maxb = case.tables.shape[1]
    s = pk.kv_decode_schedule(case.lens, hkv, maxb, num_sms, ring_stages=ring_stages, flags=flags)
    wsb = pk.kv_decode_schedule_workspace_size(s, hq, d)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    out = torch.empty((case.B, hq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((case.B, hq), dtype=torch.float32, device="cuda")
    pk.paged_decode_attention_scheduled(case.pool, case.t_q, case.t_tables, maxb,
                                        case.t_lens if lens_dev is None else lens_dev, case.B, hq,
                                        1.0 / math.sqrt(d), s, dev(s), out, pk.KV_F32, lse, ws,
                                        wsb)
    torch.cuda.synchronize()
    err = pk.kv_get_device_error(case.pool)
    assert (err != 0) if expect_err else (err == 0), err
    return host(out).astype(np.float64), host(lse).astype(np.float64), s


@pytest.mark.parametrize("num_sms,hq,hkv", [(0, 32, 8), (3, 32, 8), (16, 32, 8), (3, 24, 8),
                                             (3, 32, 4), (16, 32, 4)])
def test_scheduled_decode_matches_oracle(num_sms, hq, hkv):
    """Ragged lengths (one-token, exact-block and block+1 sequences, an empty
    one).  num_sms = 3 packs many pieces into each of few CTAs; 0 plans for
    the device.  3, 4 and 8 query heads per kv head."""
    require_cuda()
    lens = [1, 16, 17, 33, 300, 511, 1024, 1025, 2000, 47, 0, 4096, 5]
    c = random_case(lens, hq, hkv, 128, "bf16", seed=700 + num_sms + hq + hkv)
    out, lse, s = _sched_run(c, num_sms)
    if num_sms == 3:
        assert s[0] <= 15 and s[1] > 2 * s[0]  # several pieces per CTA
    ref, ref_lse = c.oracle()
    assert_close_scaled(out, ref, TOL["bf16"], "scheduled decode")
    live = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[live], ref_lse[live], atol=1e-3)
    # the empty sequence: zero output, lse = -inf
    assert np.all(out[10] == 0) and np.all(np.isneginf(lse[10]))
    # same schedule, same bits
    out2, lse2, _ = _sched_run(c, num_sms)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)
    # and the grid-indexed decode, within rounding
    g_out, g_lse = c.run(0)
    assert_close_scaled(out, g_out, 1e-5, "scheduled vs grid-indexed")
    c.close()


@pytest.mark.parametrize("num_sms", [0, 3])
def test_whole_piece_schedule_matches_oracle(num_sms):
    """One piece per CTA, pieces of near-equal length, longest first."""
    require_cuda()
    lens = [1, 16, 17, 33, 300, 511, 1024, 1025, 2000, 47, 0, 4096, 5]
    c = random_case(lens, 32, 8, 128, "bf16", seed=730 + num_sms)
    out, lse, s = _sched_run(c, num_sms, flags=pk.KV_SCHED_WHOLE_PIECES)
    assert s[0] == s[1]  # one piece per CTA
    ref, ref_lse = c.oracle()
    assert_close_scaled(out, ref, TOL["bf16"], "whole-piece schedule")
    live = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[live], ref_lse[live], atol=1e-3)
    assert np.all(out[10] == 0) and np.all(np.isneginf(lse[10]))
    c.close()


def test_wide_schedule_with_long_pieces_matches_oracle():
    """Four ring stages forced on pieces of several hundred blocks (the wide
    kernel with table slices of about a thousand entries)."""
    require_cuda()
    lens = [9000, 7001, 8192, 5000, 33]
    c = random_case(lens, 32, 8, 128, "bf16", seed=712)
    out, lse, s = _sched_run(c, 3, ring_stages=4)
    assert s[4] == 0 and s[3] >= 300
    ref, ref_lse = c.oracle()
    assert_close_scaled(out, ref, TOL["bf16"], "wide schedule, long pieces")
    np.testing.assert_allclose(lse, ref_lse, atol=1e-3)
    c.close()


def test_scheduled_deep_ring_matches_oracle():
    """Runs of >= 256 blocks take the deep-ring kernel (8 stages)."""
    require_cuda()
    lens = [9000, 7001, 8192, 5000]
    c = random_case(lens, 16, 4, 128, "bf16", seed=711)
    out, lse, s = _sched_run(c, 8)
    assert s[4] == 1 and s[3] >= 256
    ref, ref_lse = c.oracle()
    assert_close_scaled(out, ref, TOL["bf16"], "scheduled decode, deep ring")
    np.testing.assert_allclose(lse, ref_lse, atol=1e-3)
    c.close()


def test_schedule_that_does_not_match_device_lengths_is_flagged():
    """Device lengths longer or shorter than the schedule's are reported as a
    device error; every read stays inside the sequence's table row."""
    require_cuda()
    lens = [100, 1600, 1000, 33]
    c = random_case(lens, 32, 8, 128, "bf16", seed=712, extra_blocks=8)
    for delta in (-40, 40):
        wrong = np.asarray(lens, np.int32).copy()
        # 960 / 1040 tokens: within the table's width (100 blocks); the two
        # blocks past the 63 the sequence holds have table entry -1, which the
        # kernel flags and does not read
        wrong[2] += delta
        _sched_run(c, 4, lens_dev=dev(wrong), expect_err=1)
    # the pool stays usable: a matching call is clean again
    out, _, _ = _sched_run(c, 4)
    ref, _ = c.oracle()
    assert_close_scaled(out, ref, TOL["bf16"], "after a flagged call")
    c.close()


def _fused(case, num_sms, fused):
    lens, tables, pool_k, pool_v, slots, k_new, v_new, q = case
    nb, hkv, _, d = pool_k.shape
    B, hq, _ = q.shape
    maxb = tables.shape[1]
    pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
    kv, vv = pool_views(pool, nb, hkv, d, True)
    kv.copy_(dev(pool_k))
    vv.copy_(dev(pool_v))
    s = pk.kv_decode_schedule(lens, hkv, maxb, num_sms)
    wsb = pk.kv_decode_schedule_workspace_size(s, hq, d)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    out = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    if fused:
        extra = dict(k_new=dev(k_new), v_new=dev(v_new), slot_mapping=dev(slots))
    else:
        pk.kv_append(pool, dev(k_new), dev(v_new), dev(slots), B)
        extra = {}
    pk.paged_decode_attention_scheduled(pool, dev(q), dev(tables), maxb, dev(lens), B, hq,
                                        1.0 / math.sqrt(d), s, dev(s), out, pk.KV_F32, lse, ws,
                                        wsb, **extra)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(pool) == 0
    res = host(out), host(lse), host(kv, like_bf16=True), host(vv, like_bf16=True)
    pk.kv_pool_destroy(pool)
    return res


@pytest.mark.parametrize("num_sms", [0, 3])
def test_scheduled_step_fuses_the_append(num_sms):
    """With k_new the scheduled call also appends one token per sequence:
    output, lse and pool bytes bit-identical to kv_append followed by the
    scheduled decode, and the oracle on the appended content."""
    require_cuda()
    lens = [1, 16, 17, 33, 300, 511, 1024, 1025, 2000, 47]
    case = _setup(lens, 32, 8, 128, "bf16", seed=720 + num_sms)
    a = _fused(case, num_sms, False)
    b = _fused(case, num_sms, True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                                      y.view(np.uint32) if y.dtype == np.float32 else y)
    lens_, tables, pool_k, pool_v, slots, k_new, v_new, q = case
    pk_, pv_ = pool_k.copy(), pool_v.copy()
    oracle.append(pk_, pv_, k_new, v_new, slots)
    np.testing.assert_array_equal(b[2], pk_)  # the pool after the step, bit for bit
    np.testing.assert_array_equal(b[3], pv_)
    ref, ref_lse = oracle.paged_decode(pk_, pv_, tables, lens_, q, 1.0 / math.sqrt(128))
    assert_close_scaled(b[0], ref, TOL["bf16"], "scheduled fused step")
    np.testing.assert_allclose(b[1], ref_lse, atol=1e-3)


def test_llama3_8b_scheduled_full_size_sampled():
    """The Llama-3-8B-shaped decode at full size on a balanced schedule,
    sampled against the oracle.  (The benchmark runs this shape on the
    grid-indexed plan; it takes the schedule for long contexts.)"""
    c = _full_decode_case("llama3_8b_decode")
    out, lse, s = _sched_run(c, 0)
    items = _sample_items(c.B, c.hq, 96, 3)
    ref, ref_lse = c.oracle(items)
    got = np.array([out[b, h] for b, h in items])
    assert_close_scaled(got, ref, TOL["bf16"], "llama3-8b scheduled, sampled")
    np.testing.assert_allclose([lse[b, h] for b, h in items], ref_lse, atol=1e-3)
    assert np.all(np.isfinite(out))
    c.close()
