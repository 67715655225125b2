"""CPU oracle for the paged KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product package never imports it,
and it imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain fp64 C).  This module only moves
numpy arrays in and out of it.  ``brute.py`` holds a second, pure-Python
statement used to pin the C code on tiny inputs.

Element arrays: fp32 data is ``np.float32``; bfloat16 data is ``np.uint16``
holding the bf16 bit pattern; IEEE half precision is ``np.float16``.  The
dtype code is taken from the array.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    """Load (building if needed) the oracle shared library.

    ORACLE_LIB, if set, names another build of oracle.c to load instead; the
    mutation tests use it to check that the pins catch planted mistakes."""
    global _lib
    if _lib is None:
        path = os.environ.get("ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.oracle_blocks_needed.restype = i64
        L.oracle_blocks_needed.argtypes = [i64, i64]
        L.oracle_unused_slots.restype = i64
        L.oracle_unused_slots.argtypes = [i64, i64]
        L.oracle_build_block_tables.restype = i32
        L.oracle_build_block_tables.argtypes = [i32, vp, i32, vp, i64, i32, vp]
        L.oracle_append.restype = None
        L.oracle_append.argtypes = [vp, vp, i64, i32, i32, i32, i32, vp, vp, vp, i64]
        L.oracle_gather_logical.restype = None
        L.oracle_gather_logical.argtypes = [vp, i32, i32, i32, i32, vp, i64, vp]
        L.oracle_paged_decode.restype = None
        L.oracle_paged_decode.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, i32, vp, i32,
                                          i32, dbl, i64, vp, vp, vp, vp]
        L.oracle_linear_decode.restype = None
        L.oracle_linear_decode.argtypes = [vp, vp, i32, i32, i64, i32, vp, vp, i32, vp, i32, i32,
                                           dbl, i64, vp, vp, vp, vp]
        L.oracle_paged_prefill.restype = None
        L.oracle_paged_prefill.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp, vp, i32, vp,
                                           i32, i32, dbl, i64, vp, vp, vp, vp]
        L.oracle_attend_logical.restype = None
        L.oracle_attend_logical.argtypes = [vp, vp, vp, i64, i32, i32, i32, dbl, vp, vp]
        L.oracle_num_threads.restype = i32
        L.oracle_half_to_double.restype = None
        L.oracle_half_to_double.argtypes = [vp, i64, vp]
        _lib = L
    return _lib


def _code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float16:
        return 2
    raise TypeError(f"oracle takes float32, uint16 (bf16 bits) or float16 arrays, got {a.dtype}")


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().oracle_num_threads()


def blocks_needed(n_tokens: int, block_size: int) -> int:
    return lib().oracle_blocks_needed(n_tokens, block_size)


def unused_slots(n_tokens: int, block_size: int) -> int:
    return lib().oracle_unused_slots(n_tokens, block_size)


def build_block_tables(lens, block_size: int, free_order, max_blocks: int) -> np.ndarray:
    """Tables [B][max_blocks] filled by handing out ``free_order`` in sequence order."""
    lens = _c(lens, np.int32)
    free_order = _c(free_order, np.int32)
    tables = np.empty((len(lens), max_blocks), np.int32)
    rc = lib().oracle_build_block_tables(len(lens), _p(lens), block_size, _p(free_order),
                                         len(free_order), max_blocks, _p(tables))
    if rc != 0:
        raise RuntimeError("oracle: pool exhausted or table row too short")
    return tables


def append(pool_k: np.ndarray, pool_v: np.ndarray, k_new, v_new, slot_mapping) -> None:
    """In-place append into pools shaped [NB][Hkv][BS][D]."""
    nb, hkv, bs, d = pool_k.shape
    assert pool_k.flags.c_contiguous and pool_v.flags.c_contiguous
    k_new = _c(k_new, pool_k.dtype)
    v_new = _c(v_new, pool_k.dtype)
    slots = _c(slot_mapping, np.int64)
    lib().oracle_append(_p(pool_k), _p(pool_v), nb, hkv, bs, d, pool_k.itemsize, _p(k_new),
                        _p(v_new), _p(slots), len(slots))


def gather_logical(pool: np.ndarray, table, length: int) -> np.ndarray:
    """Logical [length][Hkv][D] fp64 view of one sequence."""
    nb, hkv, bs, d = pool.shape
    table = _c(table, np.int32)
    out = np.empty((length, hkv, d), np.float64)
    lib().oracle_gather_logical(_p(pool), _code(pool), hkv, bs, d, _p(table), length, _p(out))
    return out


def paged_decode(pool_k, pool_v, tables, lens, q, scale, items=None):
    """Decode attention.  q [B][Hq][D].  Returns (out fp64, lse fp64).

    items=None -> out [B][Hq][D], lse [B][Hq]; else items is a list of (b, hq)
    and out is [n][D], lse [n].
    """
    nb, hkv, bs, d = pool_k.shape
    B, hq, _ = q.shape
    tables = _c(tables, np.int32)
    lens = _c(lens, np.int32)
    q = np.ascontiguousarray(q)
    if items is None:
        out = np.empty((B, hq, d)); lse = np.empty((B, hq))
        ib = ih = None; n = -1
    else:
        it = np.asarray(items, np.int32).reshape(-1, 2)
        ib = _c(it[:, 0], np.int32); ih = _c(it[:, 1], np.int32); n = len(it)
        out = np.empty((n, d)); lse = np.empty((n,))
    lib().oracle_paged_decode(_p(pool_k), _p(pool_v), _code(pool_k), hkv, bs, d, _p(tables),
                              tables.shape[1], _p(lens), B, _p(q), _code(q), hq, float(scale), n,
                              None if ib is None else _p(ib), None if ih is None else _p(ih),
                              _p(out), _p(lse))
    return out, lse


def linear_decode(k_bases, v_bases, req_ids, lens, q, scale, items=None):
    """Decode over per-request linear buffers [Hkv][max_ctx][D] (one array per
    request, all of the same shape)."""
    hkv, max_ctx, d = k_bases[0].shape
    if any(a.shape != k_bases[0].shape for a in list(k_bases) + list(v_bases)):
        raise ValueError("all request buffers must share one [Hkv][max_ctx][D] shape")
    B, hq, _ = q.shape
    kb = (ctypes.c_void_p * len(k_bases))(*[a.ctypes.data for a in k_bases])
    vb = (ctypes.c_void_p * len(v_bases))(*[a.ctypes.data for a in v_bases])
    req_ids = _c(req_ids, np.int32)
    lens = _c(lens, np.int32)
    q = np.ascontiguousarray(q)
    if items is None:
        out = np.empty((B, hq, d)); lse = np.empty((B, hq)); ib = ih = None; n = -1
    else:
        it = np.asarray(items, np.int32).reshape(-1, 2)
        ib = _c(it[:, 0], np.int32); ih = _c(it[:, 1], np.int32); n = len(it)
        out = np.empty((n, d)); lse = np.empty((n,))
    lib().oracle_linear_decode(kb, vb, _code(k_bases[0]), hkv, max_ctx, d, _p(req_ids), _p(lens),
                               B, _p(q), _code(q), hq, float(scale), n,
                               None if ib is None else _p(ib), None if ih is None else _p(ih),
                               _p(out), _p(lse))
    return out, lse


def paged_prefill(pool_k, pool_v, tables, seq_lens, cu_q, q, scale, items=None):
    """Causal chunked prefill.  q [sumT][Hq][D].  items: list of (row, hq)."""
    nb, hkv, bs, d = pool_k.shape
    rows, hq, _ = q.shape
    tables = _c(tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    cu_q = _c(cu_q, np.int32)
    q = np.ascontiguousarray(q)
    if items is None:
        out = np.empty((rows, hq, d)); lse = np.empty((rows, hq)); ir = ih = None; n = -1
    else:
        it = np.asarray(items, np.int32).reshape(-1, 2)
        ir = _c(it[:, 0], np.int32); ih = _c(it[:, 1], np.int32); n = len(it)
        out = np.empty((n, d)); lse = np.empty((n,))
    lib().oracle_paged_prefill(_p(pool_k), _p(pool_v), _code(pool_k), hkv, bs, d, _p(tables),
                               tables.shape[1], _p(seq_lens), _p(cu_q), len(seq_lens), _p(q),
                               _code(q), hq, float(scale), n,
                               None if ir is None else _p(ir), None if ih is None else _p(ih),
                               _p(out), _p(lse))
    return out, lse


def attend_logical(q, K, V, h, scale):
    """Attention of one fp64 query [D] over explicit fp64 K, V [n][Hkv][D], kv head h."""
    q = _c(q, np.float64); K = _c(K, np.float64); V = _c(V, np.float64)
    n, hkv, d = K.shape
    o = np.empty(d); lse = np.empty(1)
    lib().oracle_attend_logical(_p(q), _p(K), _p(V), n, hkv, h, d, float(scale), _p(o), _p(lse))
    return o, float(lse[0])


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64, for comparisons."""
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def half_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """The oracle's own exact widening of binary16 bit patterns (uint16) to fp64."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    lib().oracle_half_to_double(_p(bits), bits.size, _p(out))
    return out
