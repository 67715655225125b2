"""Contiguous (vAttention-style) path on the GPU: virtual ranges reserved per
request, physical pages mapped on demand, the same decode maths without a
block table.  Checked against the oracle's linear-layout decode and, bit for
bit, against the paged path on the same logical data and split plan."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, dev, host, pool_views, read_linear, require_cuda

pytestmark = pytest.mark.gpu


class ContigCase:
    def __init__(self, lens, max_tokens, hq, hkv, d, dtype, seed, req_order=None):
        require_cuda()
        self.bf16 = dtype == "bf16"
        self.lens = np.asarray(lens, np.int32)
        self.B, self.hq, self.hkv, self.d, self.max_tokens = len(lens), hq, hkv, d, max_tokens
        g = W.rng(seed)
        # logical content per sequence
        self.K = [W.normal(g, (int(L), hkv, d), dtype) for L in lens]
        self.V = [W.normal(g, (int(L), hkv, d), dtype) for L in lens]
        self.q = W.normal(g, (self.B, hq, d), dtype)
        self.req = np.asarray(req_order if req_order is not None else np.arange(self.B), np.int32)
        self.ctx = pk.kv_contig_create(self.B + 2, max_tokens, hkv, d,
                                       pk.KV_BF16 if self.bf16 else pk.KV_F32)
        self.head_stride, self.page, self.reserved = pk.kv_contig_layout(self.ctx)
        for b, L in enumerate(lens):
            r = int(self.req[b])
            pk.kv_contig_reserve(self.ctx, r)
            pk.kv_contig_ensure(self.ctx, r, int(L))
            if L:
                pos = np.arange(L, dtype=np.int32)
                pk.kv_contig_append(self.ctx, dev(self.K[b]), dev(self.V[b]),
                                    dev(np.full(L, r, np.int32)), dev(pos), int(L))
        torch.cuda.synchronize()
        assert pk.kv_contig_get_device_error(self.ctx) == 0

    def run(self, splits=0):
        out = torch.empty((self.B, self.hq, self.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((self.B, self.hq), dtype=torch.float32, device="cuda")
        maxb = -(-self.max_tokens // 16)
        wsb = pk.kv_decode_workspace_size(self.B, self.hq, self.hkv, self.d, maxb, splits)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        pk.contig_decode_attention(self.ctx, dev(self.q), dev(self.req), dev(self.lens), self.B,
                                   self.hq, 1 / math.sqrt(self.d), out, pk.KV_F32, lse, splits,
                                   ws, wsb)
        torch.cuda.synchronize()
        assert pk.kv_contig_get_device_error(self.ctx) == 0
        return host(out).astype(np.float64), host(lse).astype(np.float64)

    def oracle_linear(self):
        # The oracle's linear-layout decode on the generated logical content
        # (one [Hkv][L][D] buffer per sequence); nothing is read back from the GPU.
        n = max(1, int(self.lens.max()))
        kb, vb = [], []
        for k, v in zip(self.K, self.V):
            kp = np.zeros((self.hkv, n, self.d), k.dtype)
            vp = np.zeros((self.hkv, n, self.d), v.dtype)
            kp[:, :len(k)] = k.transpose(1, 0, 2)
            vp[:, :len(v)] = v.transpose(1, 0, 2)
            kb.append(kp)
            vb.append(vp)
        return oracle.linear_decode(kb, vb, np.arange(self.B), self.lens, self.q,
                                    1 / math.sqrt(self.d))

    def close(self):
        pk.kv_contig_destroy(self.ctx)


def test_contig_append_lands_at_linear_positions():
    c = ContigCase([35, 17, 0], 100, hq=4, hkv=2, d=64, dtype="f32", seed=40)
    for b, L in enumerate(c.lens):
        k_ptr, _ = pk.kv_contig_ptrs(c.ctx, int(c.req[b]))
        got = read_linear(k_ptr, c.hkv, c.head_stride, int(L), c.d, False)
        np.testing.assert_array_equal(got, c.K[b].transpose(1, 0, 2))
    c.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_contig_decode_matches_oracle(dtype):
    c = ContigCase([35, 17, 1, 300, 0, 1000], 1024, hq=16, hkv=2, d=128, dtype=dtype, seed=41,
                   req_order=[3, 0, 5, 1, 2, 4])
    ref, ref_lse = c.oracle_linear()
    for splits in (1, 3, 0):
        out, lse = c.run(splits)
        assert_close_scaled(out, ref, 1e-5 if dtype == "f32" else 2e-3, f"splits={splits}")
    c.close()


@pytest.mark.parametrize("hq", [16, 32])  # g = 4 (CUDA cores) and g = 8 (tensor cores)
def test_contig_equals_paged_bit_for_bit(hq):
    lens = [35, 17, 1, 300, 777, 64]
    c = ContigCase(lens, 800, hq=hq, hkv=4, d=128, dtype="bf16", seed=42)
    # the same logical data in a shuffled paged pool
    need = sum(oracle.blocks_needed(L, 16) for L in lens)
    perm = W.permutation(W.rng(43), need + 5)
    maxb = -(-800 // 16)
    tables = oracle.build_block_tables(np.array(lens, np.int32), 16, perm, maxb)
    pool = pk.kv_pool_create(need + 5, 16, 4, 128, pk.KV_BF16)
    kv, vv = pool_views(pool, need + 5, 4, 128, True)
    kv.zero_(); vv.zero_()
    for b, L in enumerate(lens):
        j = np.arange(L)
        slots = (tables[b, j // 16].astype(np.int64) * 16 + j % 16)
        pk.kv_append(pool, dev(c.K[b]), dev(c.V[b]), dev(slots), L)
    for splits in (1, 4, 0):
        out_c, lse_c = c.run(splits)
        out_p = torch.empty((len(lens), hq, 128), dtype=torch.float32, device="cuda")
        lse_p = torch.empty((len(lens), hq), dtype=torch.float32, device="cuda")
        wsb = pk.kv_decode_workspace_size(len(lens), hq, 4, 128, maxb, splits)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        pk.paged_decode_attention(pool, dev(c.q), dev(tables), maxb, dev(np.array(lens, np.int32)),
                                  len(lens), hq, 1 / math.sqrt(128), out_p, pk.KV_F32, lse_p,
                                  splits, ws, wsb)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(out_p), out_c.astype(np.float32))
        np.testing.assert_array_equal(host(lse_p), lse_c.astype(np.float32))
    pk.kv_pool_destroy(pool)
    c.close()


def test_pages_are_mapped_on_demand_and_released():
    require_cuda()
    ctx = pk.kv_contig_create(4, 100000, 4, 128, pk.KV_BF16)
    head_stride, page, reserved = pk.kv_contig_layout(ctx)
    tpp = page // (128 * 2)                                  # tokens per page
    assert head_stride % tpp == 0 and head_stride >= 100000
    assert reserved == 2 * 4 * head_stride * 128 * 2
    pk.kv_contig_reserve(ctx, 1)
    assert pk.kv_contig_stats(ctx, 1) == (0, 0)              # reserving maps nothing
    pk.kv_contig_ensure(ctx, 1, 1)
    assert pk.kv_contig_stats(ctx, 1) == (tpp, 2 * 4 * page)
    pk.kv_contig_ensure(ctx, 1, tpp + 1)
    assert pk.kv_contig_stats(ctx, 1) == (2 * tpp, 2 * 2 * 4 * page)
    pk.kv_contig_ensure(ctx, 1, 5)                          # never shrinks
    assert pk.kv_contig_stats(ctx, 1)[0] == 2 * tpp
    with pytest.raises(pk.KVError):
        pk.kv_contig_reserve(ctx, 1)                         # already reserved
    with pytest.raises(pk.KVError):
        pk.kv_contig_ensure(ctx, 2, 10)                      # not reserved
    with pytest.raises(pk.KVError):
        pk.kv_contig_ensure(ctx, 1, 100001)                  # beyond max_tokens
    # a write past the mapped range is skipped and flagged, not faulted
    k = np.zeros((1, 4, 128), np.uint16)
    pk.kv_contig_append(ctx, dev(k), dev(k), dev(np.array([1], np.int32)),
                        dev(np.array([2 * tpp], np.int32)), 1)
    torch.cuda.synchronize()
    assert pk.kv_contig_get_device_error(ctx) == 0x8
    pk.kv_contig_release(ctx, 1)
    assert pk.kv_contig_stats(ctx, 1) == (0, 0)
    pk.kv_contig_reserve(ctx, 1)                             # reusable after release
    pk.kv_contig_destroy(ctx)


def test_page_pool_prefetches_and_recycles_pages():
    import time
    require_cuda()
    ctx = pk.kv_contig_create(4, 100000, 4, 128, pk.KV_BF16)
    _, page, _ = pk.kv_contig_layout(ctx)
    pages_per_req = 2 * 4 * -(-30000 * 128 * 2 // page)   # K and V regions of 4 heads
    pk.kv_contig_page_pool(ctx, pages_per_req, 2 * pages_per_req)
    t0 = time.time()
    while pk.kv_contig_page_stats(ctx)["spare"] < pages_per_req and time.time() - t0 < 10:
        time.sleep(0.01)
    st0 = pk.kv_contig_page_stats(ctx)
    assert st0["spare"] >= pages_per_req                  # created ahead, off the request path
    pk.kv_contig_reserve(ctx, 0)
    pk.kv_contig_ensure(ctx, 0, 30000)
    st1 = pk.kv_contig_page_stats(ctx)
    assert st1["reused"] - st0["reused"] == pages_per_req    # every mapped page came from the pool
    # the request works as usual: write and read back through the mapping
    k = W.normal(W.rng(5), (3, 4, 128), "bf16")
    pk.kv_contig_append(ctx, dev(k), dev(k), dev(np.zeros(3, np.int32)),
                        dev(np.array([0, 1, 29999], np.int32)), 3)
    torch.cuda.synchronize()
    assert pk.kv_contig_get_device_error(ctx) == 0
    k_ptr, _ = pk.kv_contig_ptrs(ctx, 0)
    hs, _, _ = pk.kv_contig_layout(ctx)
    got = read_linear(k_ptr, 4, hs, 30000, 128, True)
    np.testing.assert_array_equal(got[:, [0, 1, 29999]], k.transpose(1, 0, 2))
    # deferred reclamation: released pages stay spare and serve the next request
    pk.kv_contig_release(ctx, 0)
    created = pk.kv_contig_page_stats(ctx)["created"]
    pk.kv_contig_reserve(ctx, 1)
    pk.kv_contig_ensure(ctx, 1, 30000)
    st2 = pk.kv_contig_page_stats(ctx)
    assert st2["created"] == created or st2["created"] - created <= pages_per_req
    assert st2["reused"] - st1["reused"] == pages_per_req
    pk.kv_contig_page_pool(ctx, 0, 0)                      # stop the thread, drop spare pages
    assert pk.kv_contig_page_stats(ctx)["spare"] == 0
    pk.kv_contig_destroy(ctx)


def test_contig_launch_overlap_keeps_step_order():
    """kv_contig_set_launch_overlap: two append + decode steps back to back on
    one stream (the second step attends the token the first appended);
    outputs bit-identical to ordinary launches, and the oracle."""
    require_cuda()
    lens = [35, 17, 300, 777, 64, 1]
    B, hq, hkv, d = len(lens), 32, 4, 128
    g = W.rng(45)
    kn = [W.normal(g, (B, hkv, d), "bf16") for _ in range(2)]
    vn = [W.normal(g, (B, hkv, d), "bf16") for _ in range(2)]
    res = []
    for overlap in (False, True):
        c = ContigCase(lens, 800, hq=hq, hkv=hkv, d=d, dtype="bf16", seed=44)
        pk.kv_contig_set_launch_overlap(c.ctx, overlap)
        for b, L in enumerate(lens):
            pk.kv_contig_ensure(c.ctx, int(c.req[b]), int(L) + 2)
        maxb = -(-c.max_tokens // 16)
        wsb = pk.kv_decode_workspace_size(B, hq, hkv, d, maxb, 0)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        args = [(dev(kn[i]), dev(vn[i]), dev(c.req), dev((c.lens + i).astype(np.int32)),
                 dev(c.q), dev((c.lens + i + 1).astype(np.int32))) for i in range(2)]
        outs = [torch.empty((B, hq, d), dtype=torch.float32, device="cuda") for _ in range(2)]
        lses = [torch.empty((B, hq), dtype=torch.float32, device="cuda") for _ in range(2)]
        torch.cuda.synchronize()
        for i in range(2):  # back to back, nothing else in the stream between the launches
            k_, v_, req, pos, q, ln = args[i]
            pk.kv_contig_append(c.ctx, k_, v_, req, pos, B)
            pk.contig_decode_attention(c.ctx, q, req, ln, B, hq, 1 / math.sqrt(d), outs[i],
                                       pk.KV_F32, lses[i], 0, ws, wsb)
        torch.cuda.synchronize()
        assert pk.kv_contig_get_device_error(c.ctx) == 0
        res.append([host(o) for o in outs] + [host(x) for x in lses])
        q_case = c.q
        K2 = [np.concatenate([c.K[b], kn[0][b:b + 1], kn[1][b:b + 1]]) for b in range(B)]
        V2 = [np.concatenate([c.V[b], vn[0][b:b + 1], vn[1][b:b + 1]]) for b in range(B)]
        c.close()
    for x, y in zip(res[0], res[1]):
        np.testing.assert_array_equal(x.view(np.uint32), y.view(np.uint32))
    # the oracle's linear-layout decode over each request's content after both steps
    n = int(max(lens)) + 2
    kb, vb = [], []
    for k, v in zip(K2, V2):
        kp = np.zeros((hkv, n, d), k.dtype)
        vp = np.zeros((hkv, n, d), v.dtype)
        kp[:, :len(k)] = k.transpose(1, 0, 2)
        vp[:, :len(v)] = v.transpose(1, 0, 2)
        kb.append(kp)
        vb.append(vp)
    lens2 = np.asarray(lens, np.int32) + 2
    ref, ref_lse = oracle.linear_decode(kb, vb, np.arange(B), lens2, q_case, 1 / math.sqrt(d))
    assert_close_scaled(res[1][1], ref, 2e-3, "second contiguous step with launch overlap")
    np.testing.assert_allclose(res[1][3], ref_lse, atol=1e-3)


def _contig_step(fused, hq, d, dtype, seed):
    """One decode step on a ContigCase: a new token per request at position
    seq_lens - 1 (request 2 takes none: its step length is 0), then a decode
    of the step lengths.  Returns out, lse, each request's K and V rows after
    the step, and the logical content the oracle attends."""
    lens = [35, 17, 0, 300, 777, 64]
    c = ContigCase(lens, 800, hq=hq, hkv=4, d=d, dtype=dtype, seed=seed)
    g = W.rng(seed + 1)
    k_new = W.normal(g, (c.B, c.hkv, c.d), dtype)
    v_new = W.normal(g, (c.B, c.hkv, c.d), dtype)
    step = (c.lens + 1).astype(np.int32)
    step[2] = 0
    for b, L in enumerate(step):
        pk.kv_contig_ensure(c.ctx, int(c.req[b]), int(L))
    out = torch.empty((c.B, c.hq, c.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((c.B, c.hq), dtype=torch.float32, device="cuda")
    maxb = -(-c.max_tokens // 16)
    wsb = pk.kv_decode_workspace_size(c.B, c.hq, c.hkv, c.d, maxb, 0)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    args = (c.B, c.hq, 1 / math.sqrt(c.d), out, pk.KV_F32, lse, 0, ws, wsb)
    if fused:
        pk.contig_append_and_decode(c.ctx, dev(c.q), dev(k_new), dev(v_new), dev(c.req), dev(step),
                                    *args)
    else:
        has = np.flatnonzero(step > 0)
        pk.kv_contig_append(c.ctx, dev(k_new[has]), dev(v_new[has]), dev(c.req[has]),
                            dev((step[has] - 1).astype(np.int32)), len(has))
        pk.contig_decode_attention(c.ctx, dev(c.q), dev(c.req), dev(step), *args)
    torch.cuda.synchronize()
    assert pk.kv_contig_get_device_error(c.ctx) == 0
    rows, logical_k, logical_v = [], [], []
    for b, L in enumerate(step):
        k_ptr, v_ptr = pk.kv_contig_ptrs(c.ctx, int(c.req[b]))
        rows.append(read_linear(k_ptr, c.hkv, c.head_stride, int(L), c.d, c.bf16))
        rows.append(read_linear(v_ptr, c.hkv, c.head_stride, int(L), c.d, c.bf16))
        kb = c.K[b] if L == 0 else np.concatenate([c.K[b], k_new[b:b + 1]])
        vb = c.V[b] if L == 0 else np.concatenate([c.V[b], v_new[b:b + 1]])
        logical_k.append(kb)
        logical_v.append(vb)
    res = [host(out), host(lse)] + rows
    q = c.q
    c.close()
    return res, (logical_k, logical_v, step, q)


@pytest.mark.parametrize("hq,d,dtype", [(32, 128, "bf16"), (16, 128, "bf16"), (8, 64, "f32")])
def test_contig_fused_step_equals_append_then_decode(hq, d, dtype):
    """contig_append_and_decode is one launch on the tensor-core path (8 and 4
    query heads per kv head) and the two calls for fp32 / d64; either way the
    output, the log-sum-exp and the requests' rows equal, bit for bit,
    kv_contig_append at position seq_lens - 1 followed by
    contig_decode_attention, and the output matches the oracle on the
    appended content."""
    require_cuda()
    a, (lk, lv, step, q) = _contig_step(True, hq, d, dtype, seed=930 + hq + d)
    b, _ = _contig_step(False, hq, d, dtype, seed=930 + hq + d)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    n = int(step.max())
    kb, vb = [], []
    for k, v in zip(lk, lv):
        kp = np.zeros((4, n, d), k.dtype)
        vp = np.zeros((4, n, d), v.dtype)
        kp[:, :len(k)] = k.transpose(1, 0, 2)
        vp[:, :len(v)] = v.transpose(1, 0, 2)
        kb.append(kp)
        vb.append(vp)
    ref, _ = oracle.linear_decode(kb, vb, np.arange(len(step)), step, q, 1 / math.sqrt(d))
    assert_close_scaled(a[0], ref, 1e-5 if dtype == "f32" else 2e-3, "fused contiguous step")
    assert np.all(a[0][2] == 0)  # the request without a token: empty sequence


KV_DEVERR_UNMAPPED = 0x8  # include/paged_kv.h


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_contig_fused_step_past_the_mapped_range_appends_nothing(d, dtype):
    """Request 0 holds exactly one mapped page of tokens and its step length
    is one more: the call sets KV_DEVERR_UNMAPPED and writes nothing, so the
    request's last mapped row keeps its token (on the fused path the clamped
    length must not patch or write that row); request 1's step is unaffected
    and matches the oracle.  bf16 / d128 is the fused kernel, fp32 / d64 the
    append and decode calls."""
    require_cuda()
    ctx = pk.kv_contig_create(4, 3 * 8192, 4, d, pk.KV_BF16 if dtype == "bf16" else pk.KV_F32)
    head_stride, page, _ = pk.kv_contig_layout(ctx)
    tpp = page // (d * (2 if dtype == "bf16" else 4))  # tokens per page
    g = W.rng(960 + d)
    lens = [tpp, 37]
    K = [W.normal(g, (L, 4, d), dtype) for L in lens]
    V = [W.normal(g, (L, 4, d), dtype) for L in lens]
    for r, L in enumerate(lens):
        pk.kv_contig_reserve(ctx, r)
        pk.kv_contig_ensure(ctx, r, L)
        pk.kv_contig_append(ctx, dev(K[r]), dev(V[r]), dev(np.full(L, r, np.int32)),
                            dev(np.arange(L, dtype=np.int32)), L)
    pk.kv_contig_ensure(ctx, 1, lens[1] + 1)  # request 0 is not grown
    torch.cuda.synchronize()
    assert pk.kv_contig_get_device_error(ctx) == 0
    q = W.normal(g, (2, 16, d), dtype)
    k_new = W.normal(g, (2, 4, d), dtype)
    v_new = W.normal(g, (2, 4, d), dtype)
    step = np.array([lens[0] + 1, lens[1] + 1], np.int32)
    out = torch.empty((2, 16, d), dtype=torch.float32, device="cuda")
    maxb = -(-3 * 8192 // 16)
    wsb = pk.kv_decode_workspace_size(2, 16, 4, d, maxb, 0)
    ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
    pk.contig_append_and_decode(ctx, dev(q), dev(k_new), dev(v_new), dev(np.arange(2, dtype=np.int32)),
                                dev(step), 2, 16, 1 / math.sqrt(d), out, pk.KV_F32, None, 0, ws, wsb)
    torch.cuda.synchronize()
    assert pk.kv_contig_get_device_error(ctx) & KV_DEVERR_UNMAPPED
    bf = dtype == "bf16"
    k0, v0 = pk.kv_contig_ptrs(ctx, 0)
    np.testing.assert_array_equal(read_linear(k0, 4, head_stride, lens[0], d, bf),
                                  K[0].transpose(1, 0, 2))
    np.testing.assert_array_equal(read_linear(v0, 4, head_stride, lens[0], d, bf),
                                  V[0].transpose(1, 0, 2))
    # request 1: its step, against the oracle on its appended content
    n = lens[1] + 1
    kb = np.concatenate([K[1], k_new[1:2]]).transpose(1, 0, 2).copy()
    vb = np.concatenate([V[1], v_new[1:2]]).transpose(1, 0, 2).copy()
    ref, _ = oracle.linear_decode([kb], [vb], np.zeros(1, np.int32), np.array([n], np.int32),
                                  q[1:2], 1 / math.sqrt(d))
    assert_close_scaled(host(out)[1:2], ref, 1e-5 if dtype == "f32" else 2e-3, "request 1")
    pk.kv_contig_destroy(ctx)
