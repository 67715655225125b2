"""The contiguous (vAttention-style) decode across many separately mapped pages.

A request's K and V regions are virtual ranges backed by 2 MiB physical pages
that are created and mapped one by one as the context grows ("Makale Bulteni
-- vAttention", section "Iddia ve Gerceklik: vAttention"; "PagedAttention
Nedir?", section "vAttention Nasil Farklilasiyor?").  At bf16 and head_dim 128
one page holds 8192 tokens of one head, so only contexts longer than that make
the kernel read across independently mapped allocations.  These tests decode
20K-70K-token contexts (up to 9 pages per head region) with split plans that
reach both ring depths of the tensor-core kernel and the separate merge
kernel, and check:
  * each output against the oracle's linear-layout decode, on sampled
    (sequence, query head) items, within 2e-3 of the output scale;
  * bit identity with the paged decode of the same logical content under the
    same split plan.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, dev, host, require_cuda

pytestmark = pytest.mark.gpu


def linear_oracle_items(K, V, lens, q, items, scale):
    """The oracle's linear-layout decode on sampled (b, hq) items, one
    sequence at a time: K[b], V[b] are the logical [L][Hkv][D] contents, laid
    out as the request's own [Hkv][L][D] buffer."""
    d = q.shape[2]
    out = np.zeros((len(items), d))
    lse = np.zeros(len(items))
    by_seq = {}
    for i, (b, h) in enumerate(items):
        by_seq.setdefault(int(b), []).append((i, int(h)))
    for b, lst in by_seq.items():
        L = int(lens[b])
        n = max(L, 1)
        kb = np.zeros((K[b].shape[1], n, d), K[b].dtype)
        vb = np.zeros_like(kb)
        kb[:, :L] = K[b][:L].transpose(1, 0, 2)
        vb[:, :L] = V[b][:L].transpose(1, 0, 2)
        o, l = oracle.linear_decode([kb], [vb], np.zeros(1, np.int32), np.array([L], np.int32),
                                    q[b:b + 1], scale, items=[(0, h) for _, h in lst])
        for (i, _), oo, ll in zip(lst, o, l):
            out[i] = oo
            lse[i] = ll
    return out, lse


def sample_items(lens, hq, per_seq, seed):
    g = W.rng(seed)
    items = []
    for b in range(len(lens)):
        hs = {0, hq - 1} | {int(h) for h in g.integers(0, hq, per_seq)}
        items += [(b, h) for h in sorted(hs)]
    return items


@pytest.mark.parametrize("hq", [16, 32])   # 4 and 8 query heads per kv head
def test_contig_decode_across_mapped_pages(hq):
    require_cuda()
    hkv, d, max_tokens = 4, 128, 70000
    lens = np.array([20000, 45000, 70000, 8192, 8193, 1], np.int32)
    B, scale = len(lens), 1 / math.sqrt(d)
    g = W.rng(3100 + hq)
    K = [W.normal(g, (int(L), hkv, d), "bf16") for L in lens]
    V = [W.normal(g, (int(L), hkv, d), "bf16") for L in lens]
    q = W.normal(g, (B, hq, d), "bf16")

    ctx = pk.kv_contig_create(B, max_tokens, hkv, d, pk.KV_BF16)
    pool = None
    try:
        _, page, _ = pk.kv_contig_layout(ctx)
        tpp = page // (d * 2)                             # tokens of one head per page
        assert tpp == 8192
        pages = 0
        for b, L in enumerate(lens):
            pk.kv_contig_reserve(ctx, b)
            pk.kv_contig_ensure(ctx, b, int(L))
            # every head region of K and V is its own run of ceil(L / tpp) pages
            pages += 2 * hkv * -(-int(L) // tpp)
            assert pk.kv_contig_stats(ctx, b) == (-(-int(L) // tpp) * tpp, pages * page)
            pk.kv_contig_append(ctx, dev(K[b]), dev(V[b]), dev(np.full(int(L), b, np.int32)),
                                dev(np.arange(int(L), dtype=np.int32)), int(L))
        torch.cuda.synchronize()
        assert pk.kv_contig_get_device_error(ctx) == 0

        # the same logical content in a shuffled paged pool
        maxb = -(-max_tokens // 16)   # the contiguous path plans on this table width
        need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
        tables = oracle.build_block_tables(lens, 16, W.permutation(g, need + 7), maxb)
        pool = pk.kv_pool_create(need + 7, 16, hkv, d, pk.KV_BF16)
        for b, L in enumerate(lens):
            j = np.arange(int(L))
            slots = tables[b, j // 16].astype(np.int64) * 16 + j % 16
            pk.kv_append(pool, dev(K[b]), dev(V[b]), dev(slots), int(L))

        items = sample_items(lens, hq, 4, seed=hq)
        ref, ref_lse = linear_oracle_items(K, V, lens, q, items, scale)
        t_q, t_lens, t_tables = dev(q), dev(lens), dev(tables)
        req = dev(np.arange(B, dtype=np.int32))
        planned = pk.kv_decode_plan(lens, hkv, maxb)
        seen_deep = seen_merge_kernel = False
        for splits in (8, 32, 48, planned):
            pb, ms = pk.kv_decode_split_plan(B, hkv, maxb, splits)
            seen_deep |= pb >= 256         # the 8-stage ring instantiation
            seen_merge_kernel |= ms > 32   # partial results merged by their own kernel
            wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, splits)
            ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
            outs = []
            for contig in (True, False):
                out = torch.empty((B, hq, d), dtype=torch.float32, device="cuda")
                lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
                if contig:
                    pk.contig_decode_attention(ctx, t_q, req, t_lens, B, hq, scale, out, pk.KV_F32,
                                               lse, splits, ws, wsb)
                else:
                    pk.paged_decode_attention(pool, t_q, t_tables, maxb, t_lens, B, hq, scale, out,
                                              pk.KV_F32, lse, splits, ws, wsb)
                torch.cuda.synchronize()
                outs.append((host(out), host(lse)))
            assert pk.kv_contig_get_device_error(ctx) == 0
            assert pk.kv_get_device_error(pool) == 0
            (oc, lc), (op, lp) = outs
            np.testing.assert_array_equal(oc.view(np.uint32), op.view(np.uint32))
            np.testing.assert_array_equal(lc.view(np.uint32), lp.view(np.uint32))
            got = np.array([oc[b, h] for b, h in items], np.float64)
            assert_close_scaled(got, ref, 2e-3, f"contiguous, splits={splits} (pb={pb}, ms={ms})")
            np.testing.assert_allclose([lc[b, h] for b, h in items], ref_lse, atol=1e-3)
            assert np.all(np.isfinite(oc))
        assert seen_deep and seen_merge_kernel
    finally:
        if pool is not None:
            pk.kv_pool_destroy(pool)
        pk.kv_contig_destroy(ctx)
