"""The decode entry point for callers that cannot allocate device memory.

Such callers (a plugin whose host framework owns all device memory, a
serving loop that must not call cudaMalloc after start-up) use
paged_decode_attention_noalloc: the split-KV scratch lives in a fixed array
inside the library instead of a caller-supplied workspace.  It runs the same
kernels on the same split plan as paged_decode_attention, so its output and
lse must be bit-identical to the workspace call's, on two calls in a row (the
second call reuses the scratch the first one left behind), and within the
attention tolerance of the oracle.

This file is collected last on purpose, and it builds its own inputs so it
also passes when run alone in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W

pytestmark = pytest.mark.gpu


def _dev(a):
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()


class _Case:
    """A shuffled bf16 pool filled through kv_append, with the oracle's copy of it."""

    def __init__(self, lens, hq, hkv, d, seed):
        if not torch.cuda.is_available():
            pytest.skip("needs a CUDA device")
        g = W.rng(seed)
        self.lens = np.asarray(lens, np.int32)
        self.B, self.hq, self.hkv, self.d = len(lens), hq, hkv, d
        need = sum(oracle.blocks_needed(int(L), 16) for L in self.lens)
        nb = need + 4
        self.max_blocks = max(oracle.blocks_needed(int(L), 16) for L in self.lens)
        self.tables = oracle.build_block_tables(self.lens, 16, W.permutation(g, nb),
                                                self.max_blocks)
        self.ref_k = W.empty_pool(nb, hkv, d, "bf16")
        self.ref_v = W.empty_pool(nb, hkv, d, "bf16")
        self.pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
        for b, L in enumerate(self.lens):
            k = W.normal(g, (int(L), hkv, d), "bf16")
            v = W.normal(g, (int(L), hkv, d), "bf16")
            j = np.arange(int(L))
            slots = self.tables[b, j // 16].astype(np.int64) * 16 + j % 16
            oracle.append(self.ref_k, self.ref_v, k, v, slots)
            pk.kv_append(self.pool, _dev(k), _dev(v), _dev(slots), int(L))
        self.qs = [W.normal(g, (self.B, hq, d), "bf16") for _ in range(2)]
        self.t_tables, self.t_lens = _dev(self.tables), _dev(self.lens)
        self.scale = 1 / math.sqrt(d)
        torch.cuda.synchronize()

    def buffers(self):
        out = torch.full((self.B, self.hq, self.d), float("nan"), dtype=torch.float32,
                         device="cuda")
        lse = torch.full((self.B, self.hq), float("nan"), dtype=torch.float32, device="cuda")
        return out, lse

    def workspace_call(self, q, splits):
        wsb = pk.kv_decode_workspace_size(self.B, self.hq, self.hkv, self.d, self.max_blocks,
                                          splits)
        assert wsb > 0  # the plan really uses scratch
        ws = torch.empty(wsb // 4, dtype=torch.float32, device="cuda")
        out, lse = self.buffers()
        pk.paged_decode_attention(self.pool, q, self.t_tables, self.max_blocks, self.t_lens,
                                  self.B, self.hq, self.scale, out, pk.KV_F32, lse, splits, ws,
                                  wsb)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(self.pool) == 0
        return out.cpu().numpy(), lse.cpu().numpy()

    def noalloc_call(self, q, splits, out=None, lse=None):
        if out is None:
            out, lse = self.buffers()
        pk.paged_decode_attention_noalloc(self.pool, q, self.t_tables, self.max_blocks,
                                          self.t_lens, self.B, self.hq, self.scale, out,
                                          pk.KV_F32, lse, splits)
        return out, lse

    def check_oracle(self, out, lse, q):
        ref, ref_lse = oracle.paged_decode(self.ref_k, self.ref_v, self.tables, self.lens, q,
                                           self.scale)
        err = float(np.max(np.abs(out.astype(np.float64) - ref)))
        assert err <= 2e-3 * float(np.max(np.abs(ref))), f"max|err| {err:.3e} vs the oracle"
        np.testing.assert_allclose(lse, ref_lse, atol=1e-3)

    def close(self):
        pk.kv_pool_destroy(self.pool)


def _same_bits(a, b):
    np.testing.assert_array_equal(np.asarray(a, np.float32).view(np.uint32),
                                  np.asarray(b, np.float32).view(np.uint32))


@pytest.mark.parametrize("splits", [4, 0])
def test_noalloc_decode_matches_regular_entry_point_twice(splits):
    c = _Case([1500, 35, 4096, 700, 17, 2049, 1, 3000], hq=32, hkv=8, d=128, seed=2024)
    try:
        q = _dev(c.qs[0])
        ref, ref_lse = c.workspace_call(q, splits)
        for i in range(2):
            out, lse = c.noalloc_call(q, splits)
            torch.cuda.synchronize()
            assert pk.kv_get_device_error(c.pool) == 0
            _same_bits(out.cpu().numpy(), ref)
            _same_bits(lse.cpu().numpy(), ref_lse)
            if i == 0:
                c.check_oracle(out.cpu().numpy(), lse.cpu().numpy(), c.qs[0])
    finally:
        c.close()


def test_noalloc_plan_with_a_separate_merge_kernel():
    """More than 32 splits: the partial results are merged by their own kernel,
    which reads them back out of the library's scratch array."""
    c = _Case([4096, 3000], hq=32, hkv=8, d=128, seed=2025)
    try:
        splits = 64
        _, ms = pk.kv_decode_split_plan(c.B, c.hkv, c.max_blocks, splits)
        assert ms > 32
        assert pk.kv_decode_workspace_size(c.B, c.hq, c.hkv, c.d, c.max_blocks, splits) <= 8 << 20
        q = _dev(c.qs[0])
        ref, ref_lse = c.workspace_call(q, splits)
        for _ in range(2):
            out, lse = c.noalloc_call(q, splits)
            torch.cuda.synchronize()
            assert pk.kv_get_device_error(c.pool) == 0
            _same_bits(out.cpu().numpy(), ref)
            _same_bits(lse.cpu().numpy(), ref_lse)
        c.check_oracle(out.cpu().numpy(), lse.cpu().numpy(), c.qs[0])
    finally:
        c.close()


def test_noalloc_back_to_back_calls_with_launch_overlap():
    """Two calls with different queries queued on one stream with no wait
    between them, each decode launch overlapping the previous one's tail: the
    second call reuses the scratch the first is still finishing with, so each
    must still equal its own workspace call exactly."""
    c = _Case([1500, 35, 4096, 700, 17, 2049, 1, 3000], hq=32, hkv=8, d=128, seed=2026)
    try:
        qs = [_dev(x) for x in c.qs]
        refs = [c.workspace_call(q, 4) for q in qs]
        pk.kv_pool_set_launch_overlap(c.pool, True)
        bufs = [c.buffers() for _ in qs]
        torch.cuda.synchronize()
        for q, (out, lse) in zip(qs, bufs):
            c.noalloc_call(q, 4, out, lse)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(c.pool) == 0
        for (ref, ref_lse), (out, lse) in zip(refs, bufs):
            _same_bits(out.cpu().numpy(), ref)
            _same_bits(lse.cpu().numpy(), ref_lse)
        c.check_oracle(bufs[1][0].cpu().numpy(), bufs[1][1].cpu().numpy(), c.qs[1])
    finally:
        c.close()


def test_noalloc_rejects_plans_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    pool = pk.kv_pool_create(8, 16, 8, 128, pk.KV_BF16)
    try:
        B, hq, max_blocks, splits = 512, 64, 4096, 64   # about 1.1 GB of partials
        assert pk.kv_decode_workspace_size(B, hq, 8, 128, max_blocks, splits) > (8 << 20)
        with pytest.raises(pk.KVError) as e:
            pk.paged_decode_attention_noalloc(pool, 0, 0, max_blocks, 0, B, hq, 0.1, 0,
                                              pk.KV_F32, None, splits)
        assert e.value.status == -3  # KV_ERR_UNSUPPORTED, nothing launched
    finally:
        pk.kv_pool_destroy(pool)
