"""CPU tests of the C ABI: the library builds and loads, exports every entry
point the header declares, and its host-only logic (block accounting, free
list, reference counts, copy-on-write planning) is right.  No GPU needed.
"""
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_cache_196_gb300 as pk
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^(?:kv_status|const char\s*\*)\s*(\w+)\s*\(", src, flags=re.M)
    return names


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 30
    L = pk.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # and the binding forwards each of them under the same name
    assert not [n for n in names if not hasattr(pk, n)]


def test_status_strings():
    assert pk.kv_status_string(0) == "ok"
    assert "argument" in pk.kv_status_string(-1)


def test_worked_example_block_accounting():
    # "PagedAttention Nedir?", "Nasil Calisir?": 35 tokens at 16 per block
    # need 3 blocks and leave 13 slots unused.
    assert pk.kv_blocks_for_tokens(35, 16) == (3, 13)
    for n in range(0, 300, 7):
        assert pk.kv_blocks_for_tokens(n, 16) == (oracle.blocks_needed(n, 16),
                                                 oracle.unused_slots(n, 16))


def test_allocator_free_list_and_refcounts():
    a = pk.kv_allocator_create(8)
    try:
        assert pk.kv_allocator_num_free(a) == 8
        ids = np.zeros(3, np.int32)
        pk.kv_allocator_alloc(a, ids)
        assert ids.tolist() == [0, 1, 2]
        assert pk.kv_allocator_num_free(a) == 5
        pk.kv_allocator_share(a, ids[:1])
        assert pk.kv_allocator_refcount(a, 0) == 2
        pk.kv_allocator_free(a, ids)          # 0 -> 1 ref, 1 and 2 -> free
        assert pk.kv_allocator_refcount(a, 0) == 1
        assert pk.kv_allocator_num_free(a) == 7
        with pytest.raises(pk.KVError):        # double free
            pk.kv_allocator_free(a, ids[1:2])
        with pytest.raises(pk.KVError):        # sharing a free block
            pk.kv_allocator_share(a, ids[1:2])
        with pytest.raises(pk.KVError) as e:   # more than is free
            pk.kv_allocator_alloc(a, np.zeros(8, np.int32))
        assert e.value.status == -2
        assert pk.kv_allocator_num_free(a) == 7
        # freed blocks are reused after the never-used ones (FIFO)
        more = np.zeros(7, np.int32)
        pk.kv_allocator_alloc(a, more)
        assert more.tolist() == [3, 4, 5, 6, 7, 1, 2]
    finally:
        pk.kv_allocator_destroy(a)


def test_allocator_rejects_over_free_within_one_call():
    a = pk.kv_allocator_create(4)
    ids = np.zeros(1, np.int32)
    pk.kv_allocator_alloc(a, ids)
    with pytest.raises(pk.KVError):
        pk.kv_allocator_free(a, np.array([0, 0], np.int32))
    assert pk.kv_allocator_refcount(a, 0) == 1
    pk.kv_allocator_destroy(a)


def test_set_order_only_when_all_free():
    a = pk.kv_allocator_create(4)
    pk.kv_allocator_set_order(a, np.array([2, 0, 3, 1], np.int32))
    ids = np.zeros(2, np.int32)
    pk.kv_allocator_alloc(a, ids)
    assert ids.tolist() == [2, 0]
    with pytest.raises(pk.KVError) as e:
        pk.kv_allocator_set_order(a, np.array([0, 1, 2, 3], np.int32))
    assert e.value.status == -7
    with pytest.raises(pk.KVError):
        b = pk.kv_allocator_create(4)
        try:
            pk.kv_allocator_set_order(b, np.array([0, 0, 1, 2], np.int32))
        finally:
            pk.kv_allocator_destroy(b)
    pk.kv_allocator_destroy(a)


def _build_tables_with_library(lens, perm, max_blocks):
    a = pk.kv_allocator_create(len(perm))
    pk.kv_allocator_set_order(a, perm)
    tables = np.full((len(lens), max_blocks), -1, np.int32)
    slots = []
    for b, L in enumerate(lens):
        s = np.zeros(int(L), np.int64)
        nb, ncow = pk.kv_prepare_append(a, tables[b], 0, 0, int(L), s, np.zeros(0, np.int32),
                                        np.zeros(0, np.int32))
        assert ncow == 0 and nb == oracle.blocks_needed(int(L), 16)
        slots.append(s)
    free = pk.kv_allocator_num_free(a)
    pk.kv_allocator_destroy(a)
    return tables, slots, free


def test_block_tables_match_oracle_on_tiny_workload():
    cfg = W.CONFIGS["tiny_fp32"]
    lens = np.array(cfg["lens"], np.int32)
    perm = W.permutation(W.rng(cfg["seed"]), cfg["num_blocks"])
    tables, slots, free = _build_tables_with_library(lens, perm, 3)
    np.testing.assert_array_equal(tables, oracle.build_block_tables(lens, 16, perm, 3))
    assert free == 16 - 5
    # slot of logical token j = table[j // 16] * 16 + j % 16
    for b, L in enumerate(lens):
        j = np.arange(L)
        np.testing.assert_array_equal(slots[b], tables[b, j // 16].astype(np.int64) * 16 + j % 16)


def test_block_tables_match_oracle_on_llama_shaped_workload():
    lens = W.decode_lengths("llama3_8b_decode")
    need = sum(oracle.blocks_needed(int(L), 16) for L in lens)
    nb = int(np.ceil(1.2 * need))
    perm = W.permutation(W.rng(77), nb)
    tables, _, free = _build_tables_with_library(lens, perm, 256)
    np.testing.assert_array_equal(tables, oracle.build_block_tables(lens, 16, perm, 256))
    assert free == nb - need


def test_prepare_append_grows_and_copies_shared_blocks_on_write():
    a = pk.kv_allocator_create(16)
    parent = np.full(4, -1, np.int32)
    s = np.zeros(20, np.int64)
    nb, _ = pk.kv_prepare_append(a, parent, 0, 0, 20, s, np.zeros(0, np.int32), np.zeros(0, np.int32))
    assert nb == 2 and parent[:2].tolist() == [0, 1]
    # fork: the child shares both blocks
    child = parent.copy()
    pk.kv_allocator_share(a, child[:2])
    assert pk.kv_allocator_refcount(a, 1) == 2
    # the child writes position 20 (inside shared block 1): copy-on-write
    src, dst = np.zeros(2, np.int32), np.zeros(2, np.int32)
    s1 = np.zeros(1, np.int64)
    nb_c, ncow = pk.kv_prepare_append(a, child, 2, 20, 1, s1, src, dst)
    assert (nb_c, ncow) == (2, 1)
    assert src[0] == 1 and dst[0] == child[1] and child[1] not in (0, 1)
    assert s1[0] == child[1] * 16 + 4
    assert pk.kv_allocator_refcount(a, 1) == 1 and pk.kv_allocator_refcount(a, child[1]) == 1
    assert child[0] == 0 and pk.kv_allocator_refcount(a, 0) == 2  # untouched block still shared
    # the parent now owns block 1 alone: appending needs no copy
    nb_p, ncow = pk.kv_prepare_append(a, parent, 2, 20, 13, np.zeros(13, np.int64), src, dst)
    assert (nb_p, ncow) == (3, 0)
    pk.kv_allocator_destroy(a)


def test_prepare_append_failure_changes_nothing():
    a = pk.kv_allocator_create(3)
    row = np.full(8, -1, np.int32)
    with pytest.raises(pk.KVError) as e:
        pk.kv_prepare_append(a, row, 0, 0, 64, np.zeros(64, np.int64), np.zeros(0, np.int32),
                             np.zeros(0, np.int32))
    assert e.value.status == -2
    assert row.tolist() == [-1] * 8 and pk.kv_allocator_num_free(a) == 3
    with pytest.raises(pk.KVError) as e:  # table row too short
        pk.kv_prepare_append(a, row[:1], 0, 0, 20, np.zeros(20, np.int64), np.zeros(0, np.int32),
                             np.zeros(0, np.int32))
    assert e.value.status == -1
    # a shared block with no room to report the copy is an argument error
    nb, _ = pk.kv_prepare_append(a, row, 0, 0, 5, np.zeros(5, np.int64), np.zeros(0, np.int32),
                                 np.zeros(0, np.int32))
    pk.kv_allocator_share(a, row[:1])
    with pytest.raises(pk.KVError):
        pk.kv_prepare_append(a, row, nb, 5, 1, np.zeros(1, np.int64), np.zeros(0, np.int32),
                             np.zeros(0, np.int32))
    assert pk.kv_allocator_refcount(a, row[0]) == 2
    pk.kv_allocator_destroy(a)


def test_split_plan_and_workspace():
    pb, ms = pk.kv_decode_split_plan(64, 8, 256, 4)
    assert pb * ms >= 256 and pb % 4 == 0 and ms == -(-256 // pb)
    assert pk.kv_decode_workspace_size(64, 32, 8, 128, 256, 1) == 0
    ws = pk.kv_decode_workspace_size(64, 32, 8, 128, 256, 4)
    assert ws == 64 * 32 * ms * 129 * 4


def _shared_layout(n_blocks=64):
    """Two sequences sharing a 40-token prefix (3 blocks, the last partly used),
    plus one private sequence."""
    a = pk.kv_allocator_create(n_blocks)
    none = np.zeros(0, np.int32)
    tables = np.full((3, 8), -1, np.int32)
    nb = np.zeros(3, np.int32)
    nb[0], _ = pk.kv_prepare_append(a, tables[0], 0, 0, 40, np.zeros(40, np.int64), none, none)
    tables[1, :3] = tables[0, :3]
    pk.kv_allocator_share(a, tables[1, :3])
    nb[1] = 3
    nb[2], _ = pk.kv_prepare_append(a, tables[2], 0, 0, 20, np.zeros(20, np.int64), none, none)
    return a, tables, nb


def test_batched_planner_matches_sequential_planner():
    a1, t1, nb1 = _shared_layout()
    a2, t2, nb2 = _shared_layout()
    lens = np.array([40, 40, 20], np.int64)
    n_new = np.array([1, 30, 5], np.int32)
    # sequential
    slots_seq, pairs_seq = [], []
    cs, cd = np.zeros(4, np.int32), np.zeros(4, np.int32)
    for b in range(3):
        s = np.zeros(n_new[b], np.int64)
        nb1[b], nc = pk.kv_prepare_append(a1, t1[b], int(nb1[b]), int(lens[b]), int(n_new[b]), s,
                                          cs, cd)
        slots_seq.append(s)
        pairs_seq += list(zip(cs[:nc], cd[:nc]))
    # batched
    slots = np.zeros(int(n_new.sum()), np.int64)
    src, dst = np.zeros(8, np.int32), np.zeros(8, np.int32)
    nc = pk.kv_prepare_append_batch(a2, t2, nb2, lens, n_new, slots, src, dst)
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(nb1, nb2)
    np.testing.assert_array_equal(slots, np.concatenate(slots_seq))
    assert list(zip(src[:nc], dst[:nc])) == pairs_seq
    # the shared, partly used block 2 was copied once, for the first writer
    # (sequence 0); the second writer (sequence 1) then found it private
    assert nc == 1 and pairs_seq[0] == (t1[1, 2], t1[0, 2])


def test_batched_planner_changes_nothing_on_failure():
    a, t, nb = _shared_layout(n_blocks=7)  # 5 used, 2 free
    before = (t.copy(), nb.copy(), pk.kv_allocator_num_free(a))
    lens = np.array([40, 40, 20], np.int64)
    n_new = np.array([1, 60, 1], np.int32)  # needs more blocks than are free
    with pytest.raises(pk.KVError) as e:
        pk.kv_prepare_append_batch(a, t, nb, lens, n_new, np.zeros(62, np.int64),
                                   np.zeros(8, np.int32), np.zeros(8, np.int32))
    assert e.value.status == -2
    np.testing.assert_array_equal(t, before[0])
    np.testing.assert_array_equal(nb, before[1])
    assert pk.kv_allocator_num_free(a) == before[2]
    for blk in t[0, :3]:
        assert pk.kv_allocator_refcount(a, int(blk)) == 2


def _parse_schedule(s):
    C, P, most, W, deep, B, hkv = (int(x) for x in s[:7])
    cta = s[8:8 + C + 1]
    off = (8 + C + 1 + 3) // 4 * 4
    pcs = s[off:off + 4 * P].reshape(P, 4)
    pieces = [dict(b=int(x[0]), h=int(x[1]) & 0xffff, split=int(x[1]) >> 16, blk0=int(x[2]),
                   n=int(x[3]) & 0xffff, ns=int(x[3]) >> 16) for x in pcs]
    return dict(C=C, P=P, most=most, W=W, deep=deep, B=B, hkv=hkv, cta=cta, pieces=pieces)


@pytest.mark.parametrize("case", ["llama", "yi", "ragged", "one_long", "all_empty"])
def test_decode_schedule_covers_every_block_once_in_equal_runs(case):
    """The balanced schedule cuts the blocks of all (sequence, kv head) pairs,
    laid end to end, into runs of equal length: every block of every pair in
    exactly one piece, each pair's pieces numbered 0..n-1 in block order, every
    CTA but the last holding exactly W blocks."""
    g = W.rng(4040)
    hkv, max_blocks = 8, 256
    if case == "llama":
        lens = W.decode_lengths("llama3_8b_decode") + 1
    elif case == "yi":
        lens, hkv, max_blocks = W.decode_lengths("yi6b_long_decode"), 4, 12288
    elif case == "ragged":
        lens = np.concatenate([[0, 1, 15, 16, 17, 4096, 0], g.integers(1, 4096, 40)])
    elif case == "one_long":
        lens, hkv, max_blocks = np.array([196608]), 1, 12288
    else:
        lens = np.zeros(5, np.int64)
    lens = np.asarray(lens, np.int32)
    s = _parse_schedule(pk.kv_decode_schedule(lens, hkv, max_blocks, num_sms=152))
    nb = -(-lens.astype(np.int64) // 16)
    T = int(nb.sum()) * hkv
    assert s["B"] == len(lens) and s["hkv"] == hkv
    C, Wd = s["C"], s["W"]
    assert C == max(1, -(-T // Wd))
    # one wave: five CTAs per SM, or 2.4 with the deep ring (runs >= 256 blocks)
    assert s["deep"] == (Wd >= 256)
    assert C <= (364 if s["deep"] else 760)
    if case == "llama":
        assert not s["deep"] and Wd == -(-T // 760)
    if case == "yi":
        assert s["deep"] and Wd == -(-T // 364)
    # per-pair coverage
    seen = {}
    per_cta = np.zeros(C, np.int64)
    cta = s["cta"]
    assert cta[0] == 0 and cta[-1] == s["P"] and np.all(np.diff(cta) >= 0)
    for c in range(C):
        last = -1
        for i in range(cta[c], cta[c + 1]):
            q = s["pieces"][i]
            key = (q["b"], q["h"])
            gpos = (q["b"] * hkv + q["h"]) * 10**6 + q["blk0"]
            assert gpos >= last  # pieces of a CTA in end-to-end order
            last = gpos
            seen.setdefault(key, []).append(q)
            per_cta[c] += q["n"]
    assert sorted(seen) == [(b, h) for b in range(len(lens)) for h in range(hkv)]
    most = 1
    for (b, h), qs in seen.items():
        qs.sort(key=lambda q: q["split"])
        ns = qs[0]["ns"]
        most = max(most, ns)
        assert ns <= 32 and [q["split"] for q in qs] == list(range(ns))
        assert all(q["ns"] == ns for q in qs)
        pos = 0
        for q in qs:
            assert q["blk0"] == pos and 0 <= q["n"] <= Wd
            pos += q["n"]
        assert pos == nb[b]
        if nb[b] == 0:
            assert ns == 1 and qs[0]["n"] == 0
    assert s["most"] == most
    # equal runs
    assert np.all(per_cta[:-1] == Wd) and 0 <= per_cta[-1] <= Wd and per_cta.sum() == T


def test_decode_schedule_workspace_and_limits():
    lens = np.full(3, 4096, np.int32)
    s = pk.kv_decode_schedule(lens, 8, 256, num_sms=152)
    most, slots = int(s[2]), int(s[7])
    assert slots == most  # partial results per (sequence, query head): one per piece
    assert pk.kv_decode_schedule_workspace_size(s, 32, 128) == (
        0 if slots == 1 else 3 * 32 * slots * (128 + 1) * 4)
    # a sequence that would need more than 32 pieces of at most 1024 blocks
    with pytest.raises(pk.KVError) as e:
        pk.kv_decode_schedule(np.array([33 * 1024 * 16], np.int32), 1, 33 * 1024, num_sms=152)
    assert e.value.status == -3


def test_pool_calls_reject_a_null_pool():
    for call in (lambda: pk.kv_pool_set_launch_overlap(0, True),
                 lambda: pk.kv_pool_allocator(0)):
        with pytest.raises(pk.KVError) as e:
            call()
        assert e.value.status == -1


@pytest.mark.parametrize("case", ["llama", "yi", "ragged"])
def test_decode_schedule_whole_pieces(case):
    """KV_SCHED_WHOLE_PIECES: every pair cut into near-equal pieces (lengths
    differ by at most one block), one piece per CTA, CTAs longest first."""
    g = W.rng(4041)
    hkv, max_blocks = 8, 256
    if case == "llama":
        lens = W.decode_lengths("llama3_8b_decode") + 1
    elif case == "yi":
        lens, hkv, max_blocks = W.decode_lengths("yi6b_long_decode"), 4, 12288
    else:
        lens = np.concatenate([[0, 1, 15, 16, 17, 4096, 0], g.integers(1, 4096, 40)])
    lens = np.asarray(lens, np.int32)
    s = _parse_schedule(pk.kv_decode_schedule(lens, hkv, max_blocks, num_sms=152,
                                              flags=pk.KV_SCHED_WHOLE_PIECES))
    nb = -(-lens.astype(np.int64) // 16)
    assert s["C"] == s["P"] and list(s["cta"]) == list(range(s["C"] + 1))
    n = [q["n"] for q in s["pieces"]]
    assert n == sorted(n, reverse=True) and max(n) == s["W"]
    seen = {}
    for q in s["pieces"]:
        seen.setdefault((q["b"], q["h"]), []).append(q)
    assert len(seen) == len(lens) * hkv
    for (b, h), qs in seen.items():
        qs.sort(key=lambda q: q["split"])
        ns = qs[0]["ns"]
        assert [q["split"] for q in qs] == list(range(ns)) and ns <= 32
        pos = 0
        for q in qs:
            assert q["blk0"] == pos
            pos += q["n"]
        assert pos == nb[b]
        assert max(q["n"] for q in qs) - min(q["n"] for q in qs) <= 1
    assert s["most"] == max(q["ns"] for q in s["pieces"])


def test_decode_schedule_arguments():
    lens = np.array([4096, 100, 17], np.int32)
    # a forced CTA count must fit one wave: 5 per SM (4 stages) or 3 per SM (8 stages)
    s = _parse_schedule(pk.kv_decode_schedule(lens, 8, 256, num_sms=4, num_ctas=20, ring_stages=4))
    assert s["C"] <= 20 and s["deep"] == 0
    s = _parse_schedule(pk.kv_decode_schedule(lens, 8, 256, num_sms=4, num_ctas=12, ring_stages=8))
    assert s["C"] <= 12 and s["deep"] == 1
    for kw in (dict(num_ctas=21, ring_stages=4), dict(num_ctas=13, ring_stages=8),
               dict(ring_stages=6), dict(flags=2), dict(num_ctas=-1)):
        with pytest.raises(pk.KVError) as e:
            pk.kv_decode_schedule(lens, 8, 256, num_sms=4, **kw)
        assert e.value.status == -1, kw
    # lengths past the table width are clamped to it (the device flags them)
    s = _parse_schedule(pk.kv_decode_schedule(np.array([10**6], np.int32), 1, 64, num_sms=4))
    assert sum(q["n"] for q in s["pieces"]) == 64


def test_cascade_order_places_one_block_suffixes_after_the_first_40_percent():
    """kv_cascade_order: sequences with more than 16 own tokens longest first
    (ties in batch order), those with at most 16 as one run, longest first,
    after the first 40% (rounded) of the others; a permutation of the batch."""
    g = W.rng(4043)
    lens = np.concatenate([g.integers(17, 1025, 40), g.integers(1, 17, 25), [16, 17, 0, 17]])
    lens = g.permutation(lens).astype(np.int32)
    order = np.zeros(len(lens), np.int32)
    pk.kv_cascade_order(lens, order)
    assert sorted(order) == list(range(len(lens)))
    longs = [b for b in sorted(range(len(lens)), key=lambda b: (-int(lens[b]), b)) if lens[b] > 16]
    shorts = [b for b in sorted(range(len(lens)), key=lambda b: (-int(lens[b]), b)) if lens[b] <= 16]
    head = (2 * len(longs) + 2) // 5
    assert list(order) == longs[:head] + shorts + longs[head:]
    # all long or all short: plain longest first
    for sel in (lens[lens > 16], lens[lens <= 16]):
        o = np.zeros(len(sel), np.int32)
        pk.kv_cascade_order(sel.astype(np.int32), o)
        assert list(o) == sorted(range(len(sel)), key=lambda b: (-int(sel[b]), b))
    pk.kv_cascade_order(np.zeros(0, np.int32), np.zeros(0, np.int32))  # empty batch
