"""Chunked causal paged prefill (tcgen05) on the GPU against the CPU oracle.

bf16 inputs, fp32 output: max|err| <= 2e-3 * max|o_ref|; lse to 1e-3.
The chunk's K/V are written with kv_append first, as in a prefill step.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W
from _gpu import assert_close_scaled, bf16_to_f64, dev, host, pool_views, require_cuda

pytestmark = pytest.mark.gpu


class PrefillCase:
    def __init__(self, cached, chunk, hq, hkv, seed, extra_blocks=3, poison=True, pool=None):
        require_cuda()
        d = 128
        g = W.rng(seed)
        self.cached = np.asarray(cached, np.int32)
        self.chunk = np.asarray(chunk, np.int32)
        self.lens = (self.cached + self.chunk).astype(np.int32)
        self.B, self.hq, self.hkv, self.d = len(cached), hq, hkv, d
        need = sum(oracle.blocks_needed(int(L), 16) for L in self.lens)
        nb = need + extra_blocks
        perm = W.permutation(g, nb)
        self.maxb = max(1, max(oracle.blocks_needed(int(L), 16) for L in self.lens))
        self.tables = oracle.build_block_tables(self.lens, 16, perm, self.maxb)
        self.nb = nb
        pool_k = W.normal(g, (nb, hkv, 16, d), "bf16")
        pool_v = W.normal(g, (nb, hkv, 16, d), "bf16")
        if poison:
            # every slot at or past each sequence's length holds NaN
            used = np.zeros((nb, 16), bool)
            for b, L in enumerate(self.lens):
                j = np.arange(L)
                used[self.tables[b, j // 16], j % 16] = True
            pool_k.transpose(0, 2, 1, 3)[~used] = W.NAN_BF16
            pool_v.transpose(0, 2, 1, 3)[~used] = W.NAN_BF16
        T = int(self.chunk.sum())
        self.total_q = T
        self.k_new = W.normal(g, (T, hkv, d), "bf16")
        self.v_new = W.normal(g, (T, hkv, d), "bf16")
        self.q = W.normal(g, (T, hq, d), "bf16")
        self.cu = np.concatenate([[0], np.cumsum(self.chunk)]).astype(np.int32)
        # slots of the chunk's tokens (positions cached .. cached+T-1)
        slots = []
        for b in range(self.B):
            pos = np.arange(self.cached[b], self.lens[b])
            slots.append(self.tables[b, pos // 16].astype(np.int64) * 16 + pos % 16)
        self.slots = np.concatenate(slots) if slots else np.zeros(0, np.int64)
        # oracle pool: the same append in the oracle's byte copy
        self.ref_k, self.ref_v = pool_k.copy(), pool_v.copy()
        oracle.append(self.ref_k, self.ref_v, self.k_new, self.v_new, self.slots)
        self.pool = pk.kv_pool_create(nb, 16, hkv, d, pk.KV_BF16)
        kv, vv = pool_views(self.pool, nb, hkv, d, True)
        kv.copy_(dev(pool_k))
        vv.copy_(dev(pool_v))
        pk.kv_append(self.pool, dev(self.k_new), dev(self.v_new), dev(self.slots), T)
        torch.cuda.synchronize()

    def run(self, out_bf16=False):
        out = torch.full((self.total_q, self.hq, self.d), float("nan"), dtype=torch.float32,
                         device="cuda")
        if out_bf16:
            out = torch.zeros((self.total_q, self.hq, self.d), dtype=torch.int16, device="cuda")
        lse = torch.empty((self.total_q, self.hq), dtype=torch.float32, device="cuda")
        pk.paged_prefill_attention(self.pool, dev(self.q), dev(self.cu), self.total_q,
                                   int(self.chunk.max()), dev(self.tables), self.maxb,
                                   dev(self.lens), self.B, self.hq, 1 / math.sqrt(self.d), out,
                                   pk.KV_BF16 if out_bf16 else pk.KV_F32, lse)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(self.pool) == 0
        o = host(out, like_bf16=out_bf16)
        return (bf16_to_f64(o) if out_bf16 else o.astype(np.float64)), host(lse).astype(np.float64)

    def oracle(self, items=None):
        return oracle.paged_prefill(self.ref_k, self.ref_v, self.tables, self.lens, self.cu,
                                    self.q, 1 / math.sqrt(self.d), items=items)

    def close(self):
        pk.kv_pool_destroy(self.pool)


@pytest.mark.parametrize("cached,chunk", [
    ([0], [128]),                 # one full tile, no cache
    ([0], [200]),                 # ragged second tile
    ([300], [130]),               # cache not a multiple of the tile
    ([37, 0, 512, 5], [1, 77, 256, 129]),  # mixed, incl. a one-token chunk
])
def test_prefill_matches_oracle(cached, chunk):
    c = PrefillCase(cached, chunk, hq=4, hkv=2, seed=60 + len(chunk))
    ref, ref_lse = c.oracle()
    out, lse = c.run()
    assert_close_scaled(out, ref, 2e-3, f"prefill cached={cached} chunk={chunk}")
    np.testing.assert_allclose(lse, ref_lse, atol=1e-3)
    c.close()


def test_prefill_gqa_group_of_seven_and_bf16_output():
    c = PrefillCase([150, 1000], [300, 64], hq=14, hkv=2, seed=70)
    ref, _ = c.oracle()
    out, _ = c.run(out_bf16=True)
    scale = np.max(np.abs(ref))
    assert np.all(np.abs(out - ref) <= 2e-3 * scale + 2.0 ** -8 * np.abs(ref))
    c.close()


def test_prefill_one_token_chunk_equals_decode():
    c = PrefillCase([0, 33, 700], [1, 1, 1], hq=8, hkv=2, seed=71, poison=False)
    out, lse = c.run()
    o_dec = torch.empty((3, 8, 128), dtype=torch.float32, device="cuda")
    pk.paged_decode_attention(c.pool, dev(c.q), dev(c.tables), c.maxb, dev(c.lens), 3, 8,
                              1 / math.sqrt(128), o_dec, pk.KV_F32, None, 1, None, 0)
    torch.cuda.synchronize()
    assert_close_scaled(out, host(o_dec), 2e-3, "prefill(T=1) vs decode")
    c.close()


def test_prefill_leaves_rows_outside_chunks_untouched():
    c = PrefillCase([16], [20], hq=4, hkv=2, seed=72)
    c.total_q = 40  # q/out buffers with 20 spare rows past the only chunk
    c.q = np.concatenate([c.q, W.normal(W.rng(1), (20, 4, 128), "bf16")])
    out, _ = c.run()
    assert np.all(np.isnan(out[20:]))
    assert np.all(np.isfinite(out[:20]))
    c.close()


def test_prefill_flags_v_values_beyond_fp16():
    """The PV product runs on fp16 operands: an attended V value of 70000
    (representable in bf16, not in fp16) saturates to 65504 and sets
    KV_DEVERR_VALUE_RANGE; rows that do not attend its key stay exact, and no
    row turns non-finite (a causally masked weight of zero meets a finite
    value)."""
    c = PrefillCase([40], [100], hq=4, hkv=2, seed=73, poison=False)
    key, h, dim = 50, 0, 3                     # chunk position 10: rows 10.. attend it
    blk, off = int(c.tables[0, key // 16]), key % 16
    big = W.to_bf16_bits(np.array([70000.0], np.float32))[0]
    c.ref_v[blk, h, off, dim] = big
    _, vv = pool_views(c.pool, c.nb, c.hkv, c.d, True)
    vv[blk, h, off, dim] = int(big)            # 0x4789 < 0x8000: the same int16
    out = torch.full((c.total_q, c.hq, c.d), float("nan"), dtype=torch.float32, device="cuda")
    pk.paged_prefill_attention(c.pool, dev(c.q), dev(c.cu), c.total_q, int(c.chunk.max()),
                               dev(c.tables), c.maxb, dev(c.lens), c.B, c.hq, 1 / math.sqrt(c.d),
                               out, pk.KV_F32, None)
    torch.cuda.synchronize()
    assert pk.kv_get_device_error(c.pool) == 0x10
    out = host(out).astype(np.float64)
    assert np.all(np.isfinite(out))
    ref, _ = c.oracle()
    assert_close_scaled(out[:10], ref[:10], 2e-3, "rows before the large key")
    # rows that attend it see 65504 there: the oracle on fp32 copies of the
    # pools (bf16 widens exactly) with that one value replaced
    v32 = W.bf16_bits_to_f32(c.ref_v)
    v32[blk, h, off, dim] = 65504.0
    ref_sat, _ = oracle.paged_prefill(W.bf16_bits_to_f32(c.ref_k), v32, c.tables, c.lens, c.cu,
                                      W.bf16_bits_to_f32(c.q), 1 / math.sqrt(c.d))
    assert_close_scaled(out[10:], ref_sat[10:], 2e-3, "rows attending the saturated value")
    c.close()


@pytest.mark.slow
def test_yi34b_prefill_full_size_sampled():
    cfg = W.CONFIGS["yi34b_prefill"]
    c = PrefillCase([cfg["cached_len"]] * cfg["batch"], [cfg["chunk_len"]] * cfg["batch"],
                    hq=cfg["num_q_heads"], hkv=cfg["num_kv_heads"], seed=cfg["seed"],
                    extra_blocks=0, poison=False)
    out, lse = c.run()
    g = W.rng(5)
    rows = list(g.integers(0, c.total_q, 40)) + [0, 2047, 2048, c.total_q - 1]
    items = [(int(r), int(h)) for r, h in zip(rows, g.integers(0, c.hq, len(rows)))]
    T = cfg["chunk_len"]
    # one CTA's whole slab (two 128-row query tiles) for every query head: the
    # last 256 rows of the third sequence, ending at its final query
    items += [(2 * T + T - 256 + r, h) for r in range(256) for h in range(c.hq)]
    # every row of the first sequence's first query tile, for every head: its
    # last key tile is the one the causal boundary cuts (cached length 8192)
    items += [(r, h) for r in range(128) for h in range(c.hq)]
    items = sorted(set(items))
    ref, ref_lse = c.oracle(items)
    got = np.array([out[r, h] for r, h in items])
    assert_close_scaled(got, ref, 2e-3, "yi-34b prefill sampled")
    np.testing.assert_allclose([lse[r, h] for r, h in items], ref_lse, atol=1e-3)
    assert np.all(np.isfinite(out))
    c.close()
