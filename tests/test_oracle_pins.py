"""Pins for the CPU oracle: checks against what the pages and plain maths fix.

None of these re-types the oracle's own formula.  Each checks a fact that a
plausible mistake (a wrong head mapping, a dropped normalisation, a wrong
block index or offset, an off-by-one in the causal window, a wrong lse) would
break: the pages' worked example, closed forms, invariants, special cases that
reduce to a library routine, and an exactly-summed brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import brute
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BS = W.BLOCK_SIZE


# --------------------------------------------------------------------------
# Block accounting: "PagedAttention Nedir?", section "Nasil Calisir?".
# --------------------------------------------------------------------------
def test_worked_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    assert oracle.blocks_needed(g["tokens"], g["block_size"]) == g["blocks"]
    assert oracle.unused_slots(g["tokens"], g["block_size"]) == g["unused_slots"]


def test_only_last_block_has_unused_slots():
    # "Makale Bulteni -- PagedAttention ve vLLM": internal fragmentation is
    # limited to the free slots of the last block.
    for bs in (1, 4, 16, 32):
        assert oracle.blocks_needed(0, bs) == 0
        for n in range(1, 200):
            nb = oracle.blocks_needed(n, bs)
            assert (nb - 1) * bs < n <= nb * bs
            assert 0 <= oracle.unused_slots(n, bs) < bs


def test_tiny_config_block_counts():
    # 35 and 17 tokens at 16 per block: 3 + 2 blocks, 13 + 15 unused slots.
    assert [oracle.blocks_needed(n, BS) for n in (35, 17)] == [3, 2]
    assert [oracle.unused_slots(n, BS) for n in (35, 17)] == [13, 15]


def test_block_tables_hand_out_free_blocks_in_order():
    order = np.array([7, 3, 11, 0, 5, 9], np.int32)
    t = oracle.build_block_tables([35, 17], BS, order, max_blocks=4)
    assert t.tolist() == [[7, 3, 11, -1], [0, 5, -1, -1]]
    with pytest.raises(RuntimeError):
        oracle.build_block_tables([35, 17, 80], BS, order, max_blocks=8)


# --------------------------------------------------------------------------
# Append and reassembly.
# --------------------------------------------------------------------------
def _slots_for(table, n):
    # slot = physical block * BS + offset inside the block, for logical token j
    return np.array([table[j // BS] * BS + j % BS for j in range(n)], np.int64)


SENTINEL = {"f32": W.NAN_F32, "bf16": W.NAN_BF16, "f16": W.NAN_F16}


def _widen(a, dtype):
    """Exact fp64 values of stored elements, by numpy (not the oracle)."""
    return (W.bf16_bits_to_f32(a) if dtype == "bf16" else a).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_append_then_gather_round_trip(dtype):
    g = W.rng(5)
    nb, hkv, d, n = 12, 3, 64, 41
    table = W.permutation(g, nb)[: oracle.blocks_needed(n, BS)]
    pk = W.empty_pool(nb, hkv, d, dtype, SENTINEL[dtype])
    pv = pk.copy()
    k = W.normal(g, (n, hkv, d), dtype)
    v = W.normal(g, (n, hkv, d), dtype)
    slots = _slots_for(table, n)
    oracle.append(pk, pv, k, v, slots)
    np.testing.assert_array_equal(oracle.gather_logical(pk, table, n), _widen(k, dtype))
    np.testing.assert_array_equal(oracle.gather_logical(pv, table, n), _widen(v, dtype))
    # Every slot not named by the mapping keeps its sentinel bits.
    written = np.zeros(nb * BS, bool)
    written[slots] = True
    flat = pk.reshape(nb, hkv, BS, d).transpose(0, 2, 1, 3).reshape(nb * BS, -1)
    raw = flat.view(np.uint32 if dtype == "f32" else np.uint16)
    assert np.all(raw[~written] == SENTINEL[dtype])


def test_half_precision_widening_for_every_bit_pattern():
    """IEEE 754 binary16 -> fp64 (the oracle's own decode) against numpy's
    float16 for all 65536 patterns: normals, subnormals, zeros, infinities,
    NaNs."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # a few values by their definition
    assert oracle.half_bits_to_f64(np.array([0x3C00, 0x0001, 0x7BFF, 0xC000], np.uint16)).tolist() == \
        [1.0, 2.0 ** -24, 65504.0, -2.0]


def test_append_skips_negative_slots():
    pk = W.empty_pool(2, 1, 64, "f32")
    pv = W.empty_pool(2, 1, 64, "f32")
    k = np.ones((3, 1, 64), np.float32)
    oracle.append(pk, pv, k, k, np.array([-1, 17, -5], np.int64))
    assert pk[1, 0, 1].tolist() == [1.0] * 64
    assert np.count_nonzero(pk) == 64


# --------------------------------------------------------------------------
# Attention maths.
# --------------------------------------------------------------------------
def _tiny_case(seed=11, lens=(35, 17), nb=16, hq=4, hkv=2, d=64, dtype="f32"):
    g = W.rng(seed)
    perm = W.permutation(g, nb)
    maxb = max(oracle.blocks_needed(L, BS) for L in lens)
    tables = oracle.build_block_tables(lens, BS, perm, maxb)
    pk = W.normal(g, (nb, hkv, BS, d), dtype)
    pv = W.normal(g, (nb, hkv, BS, d), dtype)
    q = W.normal(g, (len(lens), hq, d), dtype)
    return np.array(lens, np.int32), tables, pk, pv, q


def test_length_one_context_returns_v_exactly():
    lens, tables, pk, pv, q = _tiny_case(lens=(1, 1))
    out, lse = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    for b in range(2):
        for hq in range(4):
            v = pv[tables[b, 0], hq // 2, 0].astype(np.float64)
            np.testing.assert_array_equal(out[b, hq], v)
            s = 0.125 * float(np.dot(q[b, hq].astype(np.float64), pk[tables[b, 0], hq // 2, 0]))
            assert lse[b, hq] == pytest.approx(s, rel=1e-14, abs=1e-14)


def test_zero_query_gives_mean_of_own_kv_head():
    # Equal scores -> uniform weights -> the plain mean of the logical V rows of
    # the kv head this query head reads; lse = log(L).  Distinct kv heads pin
    # the grouped-query mapping hq -> hq // (Hq / Hkv).
    lens, tables, pk, pv, q = _tiny_case()
    q[:] = 0
    out, lse = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    for b, L in enumerate(lens):
        rows = [pv[tables[b, j // BS], :, j % BS] for j in range(L)]  # [L][Hkv][D]
        mean = np.mean(np.array(rows, np.float64), axis=0)
        for hq in range(4):
            np.testing.assert_allclose(out[b, hq], mean[hq // 2], rtol=0, atol=1e-15)
            assert lse[b, hq] == pytest.approx(math.log(L), abs=1e-14)
    assert not np.allclose(out[:, 0], out[:, 2])  # the two kv heads really differ


def test_dominant_score_selects_its_value():
    lens, tables, pk, pv, q = _tiny_case()
    b, hq, j = 0, 3, 22
    k = pk[tables[b, j // BS], hq // 2, j % BS].astype(np.float64)
    q[b, hq] = (400.0 * k / np.linalg.norm(k)).astype(np.float32)
    out, _ = oracle.paged_decode(pk, pv, tables, lens, q, 1.0)
    np.testing.assert_allclose(out[b, hq], pv[tables[b, j // BS], hq // 2, j % BS], atol=1e-9)


def test_physical_placement_does_not_change_the_result():
    # "PagedAttention Nedir?": the logical token order is kept while the
    # physical placement is free.  Same logical content, two placements.
    lens, tables, pk, pv, q = _tiny_case()
    out1, lse1 = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    perm = W.permutation(W.rng(99), 16)
    pk2, pv2 = np.empty_like(pk), np.empty_like(pv)
    pk2[perm] = pk
    pv2[perm] = pv
    out2, lse2 = oracle.paged_decode(pk2, pv2, perm[tables].astype(np.int32), lens, q, 0.125)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_matches_exact_brute_force(dtype):
    lens, tables, pk, pv, q = _tiny_case(seed=3, lens=(35, 17, 1, 16), nb=24, dtype=dtype)
    out, lse = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    f = lambda a: _widen(a, dtype)  # noqa: E731
    bo, bl = brute.paged_decode(f(pk), f(pv), tables, lens, f(q), 0.125, BS)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-13)


def test_matches_library_softmax_on_numpy_reassembly():
    lens, tables, pk, pv, q = _tiny_case(seed=4)
    out, lse = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    for b, L in enumerate(lens):
        j = np.arange(L)
        K = pk[tables[b, j // BS], :, j % BS].astype(np.float64)  # [L][Hkv][D]
        V = pv[tables[b, j // BS], :, j % BS].astype(np.float64)
        for hq in range(4):
            s = 0.125 * K[:, hq // 2] @ q[b, hq].astype(np.float64)
            np.testing.assert_allclose(out[b, hq], scipy.special.softmax(s) @ V[:, hq // 2],
                                       atol=1e-14)
            assert lse[b, hq] == pytest.approx(scipy.special.logsumexp(s), abs=1e-13)


def test_shift_and_linearity_in_v():
    # Weights sum to one: o(V + c) = o(V) + c and o(aV) = a o(V).
    g = W.rng(8)
    K = g.standard_normal((40, 2, 64))
    V = g.standard_normal((40, 2, 64))
    q = g.standard_normal(64)
    o, lse = oracle.attend_logical(q, K, V, 1, 0.125)
    o2, lse2 = oracle.attend_logical(q, K, V + 3.5, 1, 0.125)
    o3, _ = oracle.attend_logical(q, K, -2.0 * V, 1, 0.125)
    np.testing.assert_allclose(o2, o + 3.5, atol=1e-13)
    np.testing.assert_allclose(o3, -2.0 * o, atol=1e-13)
    assert lse2 == lse


def test_split_and_merge_by_lse_equals_whole():
    # The key range can be cut anywhere: partial results recombine through
    # their log-sum-exp weights.  A wrong lse breaks this identity.
    g = W.rng(9)
    K = g.standard_normal((300, 1, 128))
    V = g.standard_normal((300, 1, 128))
    q = 2.0 * g.standard_normal(128)
    o, lse = oracle.attend_logical(q, K, V, 0, 1 / math.sqrt(128))
    parts = [oracle.attend_logical(q, K[a:b], V[a:b], 0, 1 / math.sqrt(128))
             for a, b in ((0, 77), (77, 200), (200, 300))]
    M = max(p[1] for p in parts)
    w = np.array([math.exp(p[1] - M) for p in parts])
    merged = sum(wi * p[0] for wi, p in zip(w, parts)) / w.sum()
    np.testing.assert_allclose(merged, o, atol=1e-13)
    assert M + math.log(w.sum()) == pytest.approx(lse, abs=1e-12)


def test_empty_context_gives_zero_and_minus_infinity():
    lens, tables, pk, pv, q = _tiny_case(lens=(0, 17))
    out, lse = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


# --------------------------------------------------------------------------
# Contiguous (vAttention) layout: same maths, linear addressing.
# --------------------------------------------------------------------------
def test_linear_layout_matches_paged_layout_exactly():
    lens, tables, pk, pv, q = _tiny_case(dtype="bf16")
    max_ctx = 48
    kb, vb = [], []
    for b, L in enumerate(lens):
        k = np.zeros((2, max_ctx, 64), np.uint16)
        v = np.zeros((2, max_ctx, 64), np.uint16)
        for j in range(L):
            k[:, j] = pk[tables[b, j // BS], :, j % BS]
            v[:, j] = pv[tables[b, j // BS], :, j % BS]
        kb.append(k); vb.append(v)
    o1, l1 = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    o2, l2 = oracle.linear_decode(kb, vb, np.arange(2), lens, q, 0.125)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# --------------------------------------------------------------------------
# Chunked causal prefill.
# --------------------------------------------------------------------------
def _prefill_case(cached=(20, 0), chunk=(13, 9), hq=4, hkv=2, d=64, seed=21):
    g = W.rng(seed)
    total = [c + t for c, t in zip(cached, chunk)]
    nb = sum(oracle.blocks_needed(L, BS) for L in total) + 3
    perm = W.permutation(g, nb)
    maxb = max(oracle.blocks_needed(L, BS) for L in total)
    tables = oracle.build_block_tables(total, BS, perm, maxb)
    pk = W.normal(g, (nb, hkv, BS, d), "f32")
    pv = W.normal(g, (nb, hkv, BS, d), "f32")
    q = W.normal(g, (sum(chunk), hq, d), "f32")
    cu = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    return np.array(total, np.int32), cu, tables, pk, pv, q


def test_prefill_zero_query_is_causal_prefix_mean():
    # Query i of a chunk that follows c cached tokens sees keys 0..c+i.
    lens, cu, tables, pk, pv, q = _prefill_case()
    q[:] = 0
    out, lse = oracle.paged_prefill(pk, pv, tables, lens, cu, q, 0.125)
    for b in range(2):
        c = lens[b] - (cu[b + 1] - cu[b])
        for i in range(cu[b + 1] - cu[b]):
            rows = np.array([pv[tables[b, j // BS], :, j % BS] for j in range(c + i + 1)], np.float64)
            for hq in range(4):
                np.testing.assert_allclose(out[cu[b] + i, hq], rows[:, hq // 2].mean(0), atol=1e-15)
                assert lse[cu[b] + i, hq] == pytest.approx(math.log(c + i + 1), abs=1e-14)


def test_prefill_first_query_without_cache_returns_first_v():
    lens, cu, tables, pk, pv, q = _prefill_case()
    out, _ = oracle.paged_prefill(pk, pv, tables, lens, cu, q, 0.125)
    b = 1  # no cached tokens: query 0 attends key 0 only
    for hq in range(4):
        np.testing.assert_array_equal(out[cu[b], hq], pv[tables[b, 0], hq // 2, 0])


def test_prefill_last_query_equals_decode():
    # The last query of a chunk sees the whole sequence, like a decode query.
    lens, cu, tables, pk, pv, q = _prefill_case()
    out, lse = oracle.paged_prefill(pk, pv, tables, lens, cu, q, 0.125)
    last = q[cu[1:] - 1]
    od, ld = oracle.paged_decode(pk, pv, tables, lens, last, 0.125)
    np.testing.assert_array_equal(out[cu[1:] - 1], od)
    np.testing.assert_array_equal(lse[cu[1:] - 1], ld)


def test_sampled_items_match_full_evaluation():
    lens, tables, pk, pv, q = _tiny_case()
    out, lse = oracle.paged_decode(pk, pv, tables, lens, q, 0.125)
    items = [(1, 3), (0, 0), (1, 1)]
    o2, l2 = oracle.paged_decode(pk, pv, tables, lens, q, 0.125, items=items)
    for i, (b, h) in enumerate(items):
        np.testing.assert_array_equal(o2[i], out[b, h])
        assert l2[i] == lse[b, h]
    lens, cu, tables, pk, pv, q = _prefill_case()
    out, lse = oracle.paged_prefill(pk, pv, tables, lens, cu, q, 0.125)
    items = [(0, 0), (21, 3), (5, 2)]
    o2, l2 = oracle.paged_prefill(pk, pv, tables, lens, cu, q, 0.125, items=items)
    for i, (r, h) in enumerate(items):
        np.testing.assert_array_equal(o2[i], out[r, h])
