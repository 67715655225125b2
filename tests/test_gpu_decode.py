"""Paged decode attention on the GPU against the CPU oracle.

Tolerances (from the attention accuracy targets): fp32 inputs max|err| <=
1e-5 * max|o_ref|; bf16 inputs max|err| <= 2e-3 * max|o_ref|, judged on fp32
output; bf16 output additionally allows its own rounding (2^-8 relative).
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

TOL = {"f32": 1e-5, "bf16": 2e-3}


class Case:
    """A pool filled with given content, block tables and queries."""

    def __init__(self, lens, tables, pool_k, pool_v, q):
        require_cuda()
        self.bf16 = pool_k.dtype == np.uint16
        self.dtype = "bf16" if self.bf16 else "f32"
        self.nb, self.hkv, _, self.d = pool_k.shape
        self.B, self.hq, _ = q.shape
        self.lens, self.tables, self.pool_k, self.pool_v, self.q = lens, tables, pool_k, pool_v, q
        self.pool = pk.kv_pool_create(self.nb, 16, self.hkv, self.d,
                                      pk.KV_BF16 if self.bf16 else pk.KV_F32)
        kv, vv = pool_views(self.pool, self.nb, self.hkv, self.d, self.bf16)
        kv.copy_(dev(pool_k))
        vv.copy_(dev(pool_v))
        self.t_tables, self.t_lens, self.t_q = dev(tables), dev(lens), dev(q)

    def run(self, splits=0, out_bf16=False, tables=None, lens=None, expect_err=0):
        maxb = self.tables.shape[1]
        out = torch.empty((self.B, self.hq, self.d),
                          dtype=torch.int16 if out_bf16 else torch.float32, device="cuda")
        lse = torch.empty((self.B, self.hq), dtype=torch.float32, device="cuda")
        wsb = pk.kv_decode_workspace_size(self.B, self.hq, self.hkv, self.d, maxb, splits)
        ws = torch.empty(max(wsb // 4, 1), dtype=torch.float32, device="cuda")
        pk.paged_decode_attention(self.pool, self.t_q, self.t_tables if tables is None else tables,
                                  maxb, self.t_lens if lens is None else lens, self.B, self.hq,
                                  1.0 / math.sqrt(self.d), out,
                                  pk.KV_BF16 if out_bf16 else pk.KV_F32, lse, splits, ws, wsb)
        torch.cuda.synchronize()
        assert pk.kv_get_device_error(self.pool) == expect_err
        o = host(out, like_bf16=out_bf16)
        return (bf16_to_f64(o) if out_bf16 else o.astype(np.float64)), host(lse).astype(np.float64)

    def oracle(self, items=None):
        return oracle.paged_decode(self.pool_k, self.pool_v, self.tables, self.lens, self.q,
                                   1.0 / math.sqrt(self.d), items=items)

    def close(self):
        pk.kv_pool_destroy(self.pool)


def random_case(lens, hq, hkv, d, dtype, seed, extra_blocks=3, poison_tail=True):
    g = W.rng(seed)
    lens = np.asarray(lens, np.int32)
    need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
    nb = need + extra_blocks
    perm = W.permutation(g, nb)
    maxb = max(1, max(oracle.blocks_needed(int(L), 16) for L in lens))
    tables = oracle.build_block_tables(lens, 16, perm, maxb)
    pool_k = W.normal(g, (nb, hkv, 16, d), dtype)
    pool_v = W.normal(g, (nb, hkv, 16, d), dtype)
    if poison_tail:
        # Unused slots of each last block and unused blocks hold NaN: masking
        # must skip them, not multiply them by zero.
        nan = W.NAN_BF16 if dtype == "bf16" else W.NAN_F32
        raw_k = pool_k.view(np.uint16 if dtype == "bf16" else np.uint32)
        raw_v = pool_v.view(np.uint16 if dtype == "bf16" else np.uint32)
        used = np.zeros((nb, 16), bool)
        for b, L in enumerate(lens):
            for j in range(L):
                used[tables[b, j // 16], j % 16] = True
        raw_k.transpose(0, 2, 1, 3)[~used] = nan
        raw_v.transpose(0, 2, 1, 3)[~used] = nan
    q = W.normal(g, (len(lens), hq, d), dtype)
    return Case(lens, tables, pool_k, pool_v, q)


# --------------------------------------------------------------------------
def test_tiny_fp32_config_all_split_plans():
    cfg = W.CONFIGS["tiny_fp32"]
    inp = W.decode_inputs("tiny_fp32", cfg["num_blocks"])
    tables = oracle.build_block_tables(inp["lens"], 16, inp["perm"], 3)
    c = Case(inp["lens"], tables, inp["pool_k"], inp["pool_v"], inp["q"])
    ref, ref_lse = c.oracle()
    for splits in (0, 1, 2, 3):
        out, lse = c.run(splits)
        assert_close_scaled(out, ref, TOL["f32"], f"splits={splits}")
        np.testing.assert_allclose(lse, ref_lse, atol=1e-5)
    c.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("g", [1, 2, 4, 8, 3, 7])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_lengths_every_group_size(dtype, g, d):
    hkv = 2
    lens = [1, 15, 16, 17, 35, 100, 257, 0, 64]
    c = random_case(lens, hq=g * hkv, hkv=hkv, d=d, dtype=dtype, seed=100 + g + d)
    ref, ref_lse = c.oracle()
    for splits in (1, 4):
        out, lse = c.run(splits)
        assert_close_scaled(out, ref, TOL[dtype], f"{dtype} g={g} d={d} splits={splits}")
        finite = np.isfinite(ref_lse)
        np.testing.assert_allclose(lse[finite], ref_lse[finite], atol=1e-5 if dtype == "f32" else 1e-3)
        assert np.all(np.isneginf(lse[~finite]))
        assert np.all(out[np.array(lens) == 0] == 0)
    c.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_length_one_context_returns_v_exactly(dtype):
    c = random_case([1, 1, 1], hq=8, hkv=2, d=128, dtype=dtype, seed=7)
    out, _ = c.run(1)
    for b in range(3):
        v = c.pool_v[c.tables[b, 0], :, 0]
        v = bf16_to_f64(v) if dtype == "bf16" else v.astype(np.float64)
        for hq in range(8):
            np.testing.assert_array_equal(out[b, hq], v[hq // 4])
    c.close()


def test_physical_placement_gives_bit_identical_output():
    c = random_case([35, 17, 300, 1, 129], hq=8, hkv=2, d=128, dtype="bf16", seed=8,
                    extra_blocks=10, poison_tail=False)
    out1, lse1 = c.run(2)
    perm = W.permutation(W.rng(55), c.nb)
    kv, vv = pool_views(c.pool, c.nb, c.hkv, c.d, True)
    k2, v2 = np.empty_like(c.pool_k), np.empty_like(c.pool_v)
    k2[perm] = c.pool_k
    v2[perm] = c.pool_v
    kv.copy_(dev(k2))
    vv.copy_(dev(v2))
    t2 = np.where(c.tables >= 0, perm[np.maximum(c.tables, 0)], -1).astype(np.int32)
    out2, lse2 = c.run(2, tables=dev(t2))
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)
    c.close()


def test_bf16_output_rounding():
    c = random_case([700, 33, 1200, 5], hq=32, hkv=8, d=128, dtype="bf16", seed=9)
    ref, _ = c.oracle()
    out, _ = c.run(0, out_bf16=True)
    scale = np.max(np.abs(ref))
    assert np.all(np.abs(out - ref) <= 2e-3 * scale + 2.0 ** -8 * np.abs(ref))
    c.close()


def test_split_plans_agree_within_fp32_rounding():
    c = random_case([4000, 2500, 17, 900], hq=32, hkv=8, d=128, dtype="bf16", seed=10)
    ref, _ = c.oracle()
    outs = [c.run(s)[0] for s in (1, 2, 7, 0)]
    for o in outs:
        assert_close_scaled(o, ref, 2e-3)
        assert_close_scaled(o, outs[0], 1e-5)
    c.close()


def test_out_of_range_block_id_is_flagged_not_faulted():
    c = random_case([40, 40], hq=4, hkv=2, d=64, dtype="f32", seed=11)
    bad = c.tables.copy()
    bad[1, 1] = c.nb + 5
    out, _ = c.run(1, tables=dev(bad), expect_err=0x1)
    ref, _ = c.oracle()
    assert_close_scaled(out[0], ref[0], 1e-5)   # the other sequence is unaffected
    assert np.all(np.isfinite(out[1]))
    c.close()


# --------------------------------------------------------------------------
# Full-size workloads in the benchmark's launch configuration (automatic
# split plan), checked on sampled (sequence, head) outputs.
# --------------------------------------------------------------------------
def _full_decode_case(name):
    lens = W.decode_lengths(name)
    need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
    nb = int(math.ceil(W.CONFIGS[name]["pool_factor"] * need))
    inp = W.decode_inputs(name, nb)
    maxb = oracle.blocks_needed(W.CONFIGS[name]["len_hi"], 16)
    tables = oracle.build_block_tables(inp["lens"], 16, inp["perm"], maxb)
    return Case(inp["lens"], tables, inp["pool_k"], inp["pool_v"], inp["q"])


def _sample_items(B, hq, n, seed):
    g = W.rng(seed)
    items = {(int(b), int(h)) for b, h in zip(g.integers(0, B, n), g.integers(0, hq, n))}
    items |= {(0, 0), (B - 1, hq - 1)}
    return sorted(items)


def test_llama3_8b_decode_full_size_sampled():
    c = _full_decode_case("llama3_8b_decode")
    out, lse = c.run(0)
    items = _sample_items(c.B, c.hq, 96, 1)
    ref, ref_lse = c.oracle(items)
    got = np.array([out[b, h] for b, h in items])
    assert_close_scaled(got, ref, TOL["bf16"], "llama3-8b sampled")
    np.testing.assert_allclose([lse[b, h] for b, h in items], ref_lse, atol=1e-3)
    assert np.all(np.isfinite(out))
    c.close()


@pytest.mark.slow
def test_yi6b_long_context_full_size_sampled():
    c = _full_decode_case("yi6b_long_decode")
    out, lse = c.run(0)
    items = _sample_items(c.B, c.hq, 24, 2)
    ref, ref_lse = c.oracle(items)
    got = np.array([out[b, h] for b, h in items])
    assert_close_scaled(got, ref, TOL["bf16"], "yi-6b sampled")
    np.testing.assert_allclose([lse[b, h] for b, h in items], ref_lse, atol=1e-3)
    assert np.all(np.isfinite(out))
    c.close()
