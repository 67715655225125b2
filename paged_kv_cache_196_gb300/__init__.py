"""Python binding of libpagedkv.so (the GB300 paged KV-cache library).

Argument marshalling only: every function below has the name of a C entry
point declared in ``include/paged_kv.h`` and forwards to it through ctypes.
Tensors are passed as raw device (or host) pointers; streams default to the
current PyTorch stream.  All compute runs in the library's CUDA kernels; there
is no fallback path -- if the library cannot be built or loaded, importing the
binding's functions raises.

Non-zero statuses raise ``KVError``.
"""
import ctypes
import os

from . import build as _build

__all__ = [
    "KVError", "lib", "KV_F32", "KV_BF16", "KV_F16", "kv_status_string", "kv_last_cuda_error", "kv_blocks_for_tokens",
    "kv_allocator_create", "kv_allocator_destroy", "kv_allocator_set_order",
    "kv_allocator_alloc", "kv_allocator_share", "kv_allocator_free", "kv_allocator_refcount",
    "kv_allocator_num_free", "kv_prepare_append", "kv_prepare_append_batch",
    "kv_prefix_cache_create", "kv_prefix_cache_destroy", "kv_prefix_cache_match",
    "kv_prefix_cache_insert", "kv_prefix_cache_evict", "kv_prefix_cache_stats", "kv_pool_create", "kv_pool_destroy",
    "kv_pool_ptrs", "kv_pool_allocator", "kv_alloc_blocks", "kv_share_blocks", "kv_free_blocks",
    "kv_cow_if_shared", "kv_append", "kv_copy_blocks", "kv_swap_out",
    "kv_swap_in", "kv_swap_bytes",
    "kv_decode_workspace_size", "kv_decode_split_plan", "kv_decode_plan", "paged_decode_attention",
    "paged_append_and_decode", "kv_decode_order",
    "paged_decode_attention_noalloc", "kv_cascade_plan", "kv_cascade_order", "kv_cascade_workspace_size",
    "paged_decode_attention_cascade", "paged_prefill_attention", "kv_get_device_error", "kv_contig_create", "kv_contig_destroy",
    "kv_contig_layout", "kv_contig_reserve", "kv_contig_ensure", "kv_contig_release",
    "kv_contig_ptrs", "kv_contig_stats", "kv_contig_page_pool", "kv_contig_page_stats", "kv_contig_append", "contig_decode_attention",
    "contig_append_and_decode", "kv_contig_get_device_error", "kv_debug_set_wait_limit_ns", "kv_debug_fail_page_create",
    "KV_WAIT_LIMIT_DEFAULT_NS",
]

KV_F32 = 0
KV_BF16 = 1
KV_F16 = 2
KV_WAIT_LIMIT_DEFAULT_NS = 2000000000

STATUS = {0: "KV_OK", -1: "KV_ERR_ARG", -2: "KV_ERR_OOM", -3: "KV_ERR_UNSUPPORTED",
          -4: "KV_ERR_CUDA", -5: "KV_ERR_DEVICE_BOUNDS", -6: "KV_ERR_TIMEOUT", -7: "KV_ERR_STATE"}


class KVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)} ({kv_status_string(status)})"
        if status in (-2, -4):
            msg += f" [{kv_last_cuda_error()}]"
        super().__init__(msg)


_lib = None
_i32, _i64, _f32, _vp, _sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
_P = ctypes.POINTER

# name -> argtypes (every function returns kv_status unless listed in _RESTYPE)
_SIGS = {
    "kv_status_string": [_i32],
    "kv_last_cuda_error": [],
    "kv_blocks_for_tokens": [_i64, _i32, _P(_i64), _P(_i64)],
    "kv_allocator_create": [_i32, _P(_vp)],
    "kv_allocator_destroy": [_vp],
    "kv_allocator_set_order": [_vp, _vp, _i32],
    "kv_allocator_alloc": [_vp, _i32, _vp],
    "kv_allocator_share": [_vp, _i32, _vp],
    "kv_allocator_free": [_vp, _i32, _vp],
    "kv_allocator_refcount": [_vp, ctypes.c_int32, _P(_i32)],
    "kv_allocator_num_free": [_vp, _P(_i32)],
    "kv_prepare_append": [_vp, _i32, _vp, _i32, _P(_i32), _i64, _i32, _vp, _vp, _vp, _P(_i32)],
    "kv_prepare_append_batch": [_vp, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _P(_i32)],
    "kv_prefix_cache_create": [_vp, _i32, _i32, _P(_vp)],
    "kv_prefix_cache_destroy": [_vp],
    "kv_prefix_cache_match": [_vp, _vp, _i64, _vp, _i32, _P(_i32)],
    "kv_prefix_cache_insert": [_vp, _vp, _i64, _vp, _i32, _P(_i32)],
    "kv_prefix_cache_evict": [_vp, _i32, _P(_i32)],
    "kv_prefix_cache_stats": [_vp, _P(_i32), _P(_i64), _P(_i64)],
    "kv_pool_create": [_i32, _i32, _i32, _i32, _i32, _P(_vp)],
    "kv_pool_destroy": [_vp],
    "kv_pool_ptrs": [_vp, _P(_vp), _P(_vp)],
    "kv_pool_allocator": [_vp, _P(_vp)],
    "kv_pool_set_launch_overlap": [_vp, _i32],
    "kv_alloc_blocks": [_vp, _i32, _vp],
    "kv_share_blocks": [_vp, _i32, _vp],
    "kv_free_blocks": [_vp, _i32, _vp],
    "kv_cow_if_shared": [_vp, _P(_i32), _P(_i32), _vp],
    "kv_append": [_vp, _vp, _vp, _vp, _i32, _vp],
    "kv_copy_blocks": [_vp, _vp, _vp, _i32, _vp],
    "kv_swap_out": [_vp, _vp, _i32, _vp, _vp],
    "kv_swap_in": [_vp, _vp, _i32, _vp, _vp],
    "kv_swap_bytes": [_vp, _i32, _P(_sz)],
    "kv_decode_workspace_size": [_i32, _i32, _i32, _i32, _i32, _i32, _P(_sz)],
    "kv_decode_split_plan": [_i32, _i32, _i32, _i32, _P(_i32), _P(_i32)],
    "kv_decode_plan": [_vp, _i32, _i32, _i32, _P(_i32)],
    "paged_decode_attention": [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _i32, _vp, _i32,
                               _vp, _sz, _vp],
    "paged_append_and_decode": [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _f32,
                                _vp, _i32, _vp, _i32, _vp, _sz, _vp],
    "kv_decode_order": [_vp, _i32, _vp],
    "kv_decode_schedule_capacity": [_i32, _i32, _i32, _i32, _P(_sz)],
    "kv_decode_schedule": [_vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _sz, _P(_sz)],
    "kv_decode_schedule_workspace_size": [_vp, _i32, _i32, _P(_sz)],
    "paged_decode_attention_scheduled": [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _f32,
                                         _vp, _vp, _vp, _i32, _vp, _vp, _sz, _vp],
    "paged_decode_attention_noalloc": [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _i32,
                                       _vp, _i32, _vp],
    "kv_cascade_plan": [_i32, _i32, _i32, _i32, _P(_i32)],
    "kv_cascade_order": [_vp, _i32, _vp],
    "kv_cascade_workspace_size": [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _P(_sz)],
    "paged_decode_attention_cascade": [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _f32, _vp, _i32,
                                       _i32, _vp, _i32, _i32, _vp, _i32, _vp, _i32, _vp, _vp,
                                       _sz, _vp],
    "paged_prefill_attention": [_vp, _vp, _vp, _i32, _i32, _vp, _i32, _vp, _i32, _i32, _f32, _vp,
                                _i32, _vp, _vp],
    "kv_get_device_error": [_vp, _P(_i32), _vp],
    "kv_contig_create": [_i32, _i32, _i32, _i32, _i32, _P(_vp)],
    "kv_contig_destroy": [_vp],
    "kv_contig_layout": [_vp, _P(_i64), _P(_i64), _P(_i64)],
    "kv_contig_reserve": [_vp, _i32],
    "kv_contig_ensure": [_vp, _i32, _i64],
    "kv_contig_release": [_vp, _i32],
    "kv_contig_ptrs": [_vp, _i32, _P(_vp), _P(_vp)],
    "kv_contig_page_pool": [_vp, _i32, _i32],
    "kv_contig_page_stats": [_vp, _P(_i32), _P(_i64), _P(_i64), _P(ctypes.c_double),
                             _P(ctypes.c_double)],
    "kv_contig_stats": [_vp, _i32, _P(_i64), _P(_i64)],
    "kv_contig_append": [_vp, _vp, _vp, _vp, _vp, _i32, _vp],
    "contig_decode_attention": [_vp, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _i32, _vp, _i32, _vp,
                                _sz, _vp],
    "contig_append_and_decode": [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _f32, _vp, _i32, _vp,
                                 _i32, _vp, _sz, _vp],
    "kv_contig_get_device_error": [_vp, _P(_i32), _vp],
    "kv_contig_set_launch_overlap": [_vp, _i32],
    "kv_debug_set_wait_limit_ns": [ctypes.c_uint64],
    "kv_debug_fail_page_create": [_i32],
}
_RESTYPE = {"kv_status_string": ctypes.c_char_p, "kv_last_cuda_error": ctypes.c_char_p}


def lib_path() -> str:
    return _build.LIB


def lib(build: bool = True):
    """The loaded library (built first if missing or stale and ``build``)."""
    global _lib
    if _lib is None:
        path = _build.build() if build else _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libpagedkv.so not found at {path}; run paged_kv_cache_196_gb300/build.py")
        L = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _RESTYPE.get(name, ctypes.c_int)
        _lib = L
    return _lib


def _ptr(x):
    """Raw address of a tensor / numpy array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


_torch = None


def _stream(s):
    """A stream argument as the raw handle: None = torch's current stream."""
    global _torch
    if s is None:
        if _torch is None:
            import torch
            _torch = torch
        return _torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str):
    if st != 0:
        raise KVError(st, where)


def kv_status_string(status: int) -> str:
    return lib().kv_status_string(status).decode()


def kv_last_cuda_error() -> str:
    return lib().kv_last_cuda_error().decode()


def kv_blocks_for_tokens(n_tokens: int, block_size: int = 16):
    b, u = _i64(), _i64()
    _check(lib().kv_blocks_for_tokens(n_tokens, block_size, ctypes.byref(b), ctypes.byref(u)),
           "kv_blocks_for_tokens")
    return b.value, u.value


# ---------------------------------------------------------------- allocator
def kv_allocator_create(num_blocks: int) -> int:
    h = _vp()
    _check(lib().kv_allocator_create(num_blocks, ctypes.byref(h)), "kv_allocator_create")
    return h.value


def kv_allocator_destroy(a: int):
    _check(lib().kv_allocator_destroy(a), "kv_allocator_destroy")


def kv_allocator_set_order(a: int, order):
    """order: int32 numpy array (host)."""
    _check(lib().kv_allocator_set_order(a, _ptr(order), len(order)), "kv_allocator_set_order")


def kv_allocator_alloc(a: int, ids_out):
    """Fills ids_out (int32 numpy array) with len(ids_out) fresh blocks."""
    _check(lib().kv_allocator_alloc(a, len(ids_out), _ptr(ids_out)), "kv_allocator_alloc")


def kv_allocator_share(a: int, ids):
    _check(lib().kv_allocator_share(a, len(ids), _ptr(ids)), "kv_allocator_share")


def kv_allocator_free(a: int, ids):
    _check(lib().kv_allocator_free(a, len(ids), _ptr(ids)), "kv_allocator_free")


def kv_allocator_refcount(a: int, block_id: int) -> int:
    r = _i32()
    _check(lib().kv_allocator_refcount(a, block_id, ctypes.byref(r)), "kv_allocator_refcount")
    return r.value


def kv_allocator_num_free(a: int) -> int:
    r = _i32()
    _check(lib().kv_allocator_num_free(a, ctypes.byref(r)), "kv_allocator_num_free")
    return r.value


def kv_prepare_append(a: int, table_row, num_blocks: int, cur_len: int, n_new: int, slots_out,
                      cow_src, cow_dst, block_size: int = 16):
    """Host step of an append.  table_row (int32), slots_out (int64), cow_src/cow_dst
    (int32, capacity = their length) are numpy arrays updated in place.
    Returns (num_blocks, n_cow)."""
    nb = _i32(num_blocks)
    ncow = _i32(len(cow_src))
    _check(lib().kv_prepare_append(a, block_size, _ptr(table_row), len(table_row),
                                   ctypes.byref(nb), cur_len, n_new, _ptr(slots_out),
                                   _ptr(cow_src), _ptr(cow_dst), ctypes.byref(ncow)),
           "kv_prepare_append")
    return nb.value, ncow.value


def kv_prepare_append_batch(a: int, tables, num_blocks, cur_lens, n_new, slots_out, cow_src,
                            cow_dst, block_size: int = 16) -> int:
    """Batched host step.  tables int32 [B][max_blocks], num_blocks int32 [B] (updated in
    place), cur_lens int64 [B], n_new int32 [B], slots_out int64 [sum n_new], cow_src /
    cow_dst int32 (capacity = their length).  Returns the number of copy pairs."""
    ncow = _i32(len(cow_src))
    _check(lib().kv_prepare_append_batch(a, block_size, tables.shape[0], _ptr(tables),
                                         tables.shape[1], _ptr(num_blocks), _ptr(cur_lens),
                                         _ptr(n_new), _ptr(slots_out), _ptr(cow_src),
                                         _ptr(cow_dst), ctypes.byref(ncow)),
           "kv_prepare_append_batch")
    return ncow.value


# ---------------------------------------------------------------- prefix cache
def kv_prefix_cache_create(a: int, capacity_blocks: int, block_size: int = 16) -> int:
    h = _vp()
    _check(lib().kv_prefix_cache_create(a, block_size, capacity_blocks, ctypes.byref(h)),
           "kv_prefix_cache_create")
    return h.value


def kv_prefix_cache_destroy(c: int):
    _check(lib().kv_prefix_cache_destroy(c), "kv_prefix_cache_destroy")


def kv_prefix_cache_match(c: int, tokens, blocks_out) -> int:
    """tokens int32 numpy; blocks_out int32 numpy (capacity = its length)."""
    n = _i32()
    _check(lib().kv_prefix_cache_match(c, _ptr(tokens), len(tokens), _ptr(blocks_out),
                                       len(blocks_out), ctypes.byref(n)), "kv_prefix_cache_match")
    return n.value


def kv_prefix_cache_insert(c: int, tokens, blocks) -> int:
    n = _i32()
    _check(lib().kv_prefix_cache_insert(c, _ptr(tokens), len(tokens), _ptr(blocks), len(blocks),
                                        ctypes.byref(n)), "kv_prefix_cache_insert")
    return n.value


def kv_prefix_cache_evict(c: int, n_blocks: int) -> int:
    n = _i32()
    _check(lib().kv_prefix_cache_evict(c, n_blocks, ctypes.byref(n)), "kv_prefix_cache_evict")
    return n.value


def kv_prefix_cache_stats(c: int):
    cb, lk, ht = _i32(), _i64(), _i64()
    _check(lib().kv_prefix_cache_stats(c, ctypes.byref(cb), ctypes.byref(lk), ctypes.byref(ht)),
           "kv_prefix_cache_stats")
    return cb.value, lk.value, ht.value


# ---------------------------------------------------------------- pool
def kv_pool_create(num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                   dtype: int) -> int:
    h = _vp()
    _check(lib().kv_pool_create(num_blocks, block_size, num_kv_heads, head_dim, dtype,
                                ctypes.byref(h)), "kv_pool_create")
    return h.value


def kv_pool_destroy(p: int):
    _check(lib().kv_pool_destroy(p), "kv_pool_destroy")


def kv_pool_ptrs(p: int):
    k, v = _vp(), _vp()
    _check(lib().kv_pool_ptrs(p, ctypes.byref(k), ctypes.byref(v)), "kv_pool_ptrs")
    return k.value, v.value


def kv_pool_set_launch_overlap(p: int, enable: bool):
    """Let this pool's tensor-core decode launches overlap the previous kernel
    in their stream (each waits for it before touching memory)."""
    _check(lib().kv_pool_set_launch_overlap(p, 1 if enable else 0), "kv_pool_set_launch_overlap")


def kv_pool_allocator(p: int) -> int:
    a = _vp()
    _check(lib().kv_pool_allocator(p, ctypes.byref(a)), "kv_pool_allocator")
    return a.value


def kv_alloc_blocks(p: int, ids_out):
    """Fills ids_out (int32 numpy array) with len(ids_out) fresh blocks of the pool."""
    _check(lib().kv_alloc_blocks(p, len(ids_out), _ptr(ids_out)), "kv_alloc_blocks")


def kv_share_blocks(p: int, ids):
    """ids: int32 numpy array."""
    _check(lib().kv_share_blocks(p, len(ids), _ptr(ids)), "kv_share_blocks")


def kv_free_blocks(p: int, ids):
    """ids: int32 numpy array."""
    _check(lib().kv_free_blocks(p, len(ids), _ptr(ids)), "kv_free_blocks")


def kv_cow_if_shared(p: int, block_id: int, stream=None):
    """Returns (block id to write into, copied?)."""
    bid = _i32(block_id)
    copied = _i32()
    _check(lib().kv_cow_if_shared(p, ctypes.byref(bid), ctypes.byref(copied), _stream(stream)),
           "kv_cow_if_shared")
    return bid.value, bool(copied.value)


def kv_append(p: int, k_new, v_new, slot_mapping, num_tokens: int, stream=None):
    _check(lib().kv_append(p, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), num_tokens,
                           _stream(stream)), "kv_append")


def kv_copy_blocks(p: int, src, dst, n: int, stream=None):
    _check(lib().kv_copy_blocks(p, _ptr(src), _ptr(dst), n, _stream(stream)), "kv_copy_blocks")


def kv_swap_out(p: int, block_ids, n: int, host_buf, stream=None):
    _check(lib().kv_swap_out(p, _ptr(block_ids), n, _ptr(host_buf), _stream(stream)), "kv_swap_out")


def kv_swap_in(p: int, block_ids, n: int, host_buf, stream=None):
    _check(lib().kv_swap_in(p, _ptr(block_ids), n, _ptr(host_buf), _stream(stream)), "kv_swap_in")


def kv_swap_bytes(p: int, n: int) -> int:
    r = _sz()
    _check(lib().kv_swap_bytes(p, n, ctypes.byref(r)), "kv_swap_bytes")
    return r.value


def kv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_blocks,
                             num_splits=0) -> int:
    r = _sz()
    _check(lib().kv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_blocks,
                                          num_splits, ctypes.byref(r)), "kv_decode_workspace_size")
    return r.value


def kv_decode_split_plan(batch, num_kv_heads, max_blocks, num_splits=0):
    pb, ms = _i32(), _i32()
    _check(lib().kv_decode_split_plan(batch, num_kv_heads, max_blocks, num_splits,
                                      ctypes.byref(pb), ctypes.byref(ms)), "kv_decode_split_plan")
    return pb.value, ms.value


def kv_decode_plan(host_seq_lens, num_kv_heads: int, max_blocks: int) -> int:
    """num_splits for a decode over sequences of these (host, int32) lengths."""
    import numpy as _np
    lens = _np.ascontiguousarray(host_seq_lens, dtype=_np.int32)
    r = _i32()
    _check(lib().kv_decode_plan(_ptr(lens), len(lens), num_kv_heads, max_blocks, ctypes.byref(r)),
           "kv_decode_plan")
    return r.value


def paged_decode_attention(p: int, q, block_tables, max_blocks: int, seq_lens, batch: int,
                           num_q_heads: int, scale: float, out, out_dtype: int, lse_out=None,
                           num_splits: int = 0, workspace=None, workspace_bytes: int = 0,
                           stream=None):
    _check(lib().paged_decode_attention(p, _ptr(q), _ptr(block_tables), max_blocks, _ptr(seq_lens),
                                        batch, num_q_heads, scale, _ptr(out), out_dtype,
                                        _ptr(lse_out), num_splits, _ptr(workspace),
                                        workspace_bytes, _stream(stream)),
           "paged_decode_attention")


def kv_decode_order(host_seq_lens, order_out):
    """host_seq_lens, order_out: int32 numpy arrays of the batch size (host)."""
    _check(lib().kv_decode_order(_ptr(host_seq_lens), len(host_seq_lens), _ptr(order_out)),
           "kv_decode_order")


def paged_append_and_decode(p: int, q, k_new, v_new, slot_mapping, block_tables, max_blocks: int,
                            seq_lens, batch: int, num_q_heads: int, scale: float, out,
                            out_dtype: int, lse_out=None, num_splits: int = 0, workspace=None,
                            workspace_bytes: int = 0, stream=None, seq_order=None):
    """kv_append of one token per sequence, then paged_decode_attention (one
    fused launch where supported); seq_order: device int32 permutation of the
    batch or None.  See the C header."""
    _check(lib().paged_append_and_decode(p, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                         _ptr(block_tables), max_blocks, _ptr(seq_lens),
                                         _ptr(seq_order), batch,
                                         num_q_heads, scale, _ptr(out), out_dtype, _ptr(lse_out),
                                         num_splits, _ptr(workspace), workspace_bytes,
                                         _stream(stream)), "paged_append_and_decode")


def kv_decode_schedule_capacity(batch: int, num_kv_heads: int, max_blocks: int,
                                num_sms: int = 0) -> int:
    """int32 words a kv_decode_schedule of this batch shape may need."""
    r = _sz()
    _check(lib().kv_decode_schedule_capacity(batch, num_kv_heads, max_blocks, num_sms,
                                             ctypes.byref(r)), "kv_decode_schedule_capacity")
    return r.value


KV_SCHED_WHOLE_PIECES = 1


def kv_decode_schedule(host_seq_lens, num_kv_heads: int, max_blocks: int, num_sms: int = 0,
                       num_ctas: int = 0, ring_stages: int = 0, flags: int = 0, out=None):
    """Balanced decode schedule for these host int32 lengths: an int32 numpy
    array (header, first piece of each CTA, pieces) to copy to the device for
    paged_decode_attention_scheduled.  num_sms = 0: the current device's;
    num_ctas / ring_stages = 0: the library's rule.  With `out` (a contiguous
    int32 host array) the schedule is written there and a view of its used
    part is returned."""
    import numpy as _np
    lens = _np.ascontiguousarray(host_seq_lens, dtype=_np.int32)
    if out is None:
        cap = kv_decode_schedule_capacity(len(lens), num_kv_heads, max_blocks, num_sms)
        buf = _np.zeros(cap, _np.int32)
    else:
        buf = out
    used = _sz()
    _check(lib().kv_decode_schedule(_ptr(lens), len(lens), num_kv_heads, max_blocks, num_sms,
                                    num_ctas, ring_stages, flags, _ptr(buf), len(buf),
                                    ctypes.byref(used)),
           "kv_decode_schedule")
    return buf[:used.value].copy() if out is None else buf[:used.value]


def kv_decode_schedule_workspace_size(host_schedule, num_q_heads: int, head_dim: int) -> int:
    r = _sz()
    _check(lib().kv_decode_schedule_workspace_size(_ptr(host_schedule), num_q_heads, head_dim,
                                                   ctypes.byref(r)),
           "kv_decode_schedule_workspace_size")
    return r.value


def paged_decode_attention_scheduled(p: int, q, block_tables, max_blocks: int, seq_lens,
                                     batch: int, num_q_heads: int, scale: float, host_schedule,
                                     schedule, out, out_dtype: int, lse_out=None, workspace=None,
                                     workspace_bytes: int = 0, stream=None, k_new=None, v_new=None,
                                     slot_mapping=None):
    """Decode (with the step's append when k_new is given) on a balanced
    schedule: host_schedule is kv_decode_schedule's array, schedule its device
    copy.  See the C header."""
    _check(lib().paged_decode_attention_scheduled(p, _ptr(q), _ptr(k_new), _ptr(v_new),
                                                  _ptr(slot_mapping), _ptr(block_tables),
                                                  max_blocks, _ptr(seq_lens), batch, num_q_heads,
                                                  scale, _ptr(host_schedule), _ptr(schedule),
                                                  _ptr(out), out_dtype, _ptr(lse_out),
                                                  _ptr(workspace), workspace_bytes,
                                                  _stream(stream)),
           "paged_decode_attention_scheduled")


def paged_decode_attention_noalloc(p: int, q, block_tables, max_blocks: int, seq_lens,
                                   batch: int, num_q_heads: int, scale: float, out,
                                   out_dtype: int, lse_out=None, num_splits: int = 0,
                                   stream=None):
    """paged_decode_attention with the split scratch in the library's fixed
    device array (for callers that cannot allocate); see the C header."""
    _check(lib().paged_decode_attention_noalloc(p, _ptr(q), _ptr(block_tables), max_blocks,
                                                _ptr(seq_lens), batch, num_q_heads, scale,
                                                _ptr(out), out_dtype, _ptr(lse_out), num_splits,
                                                _stream(stream)),
           "paged_decode_attention_noalloc")


def kv_cascade_order(host_suffix_lens, order_out):
    """host_suffix_lens, order_out: int32 numpy arrays of the batch size (host)."""
    _check(lib().kv_cascade_order(_ptr(host_suffix_lens), len(host_suffix_lens), _ptr(order_out)),
           "kv_cascade_order")


def kv_cascade_plan(num_groups: int, num_kv_heads: int, max_prefix_blocks: int,
                    requested: int = 0) -> int:
    r = _i32()
    _check(lib().kv_cascade_plan(num_groups, num_kv_heads, max_prefix_blocks, requested,
                                 ctypes.byref(r)), "kv_cascade_plan")
    return r.value


def kv_cascade_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_blocks, num_splits,
                              prefix_splits) -> int:
    r = _sz()
    _check(lib().kv_cascade_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_blocks,
                                           num_splits, prefix_splits, ctypes.byref(r)),
           "kv_cascade_workspace_size")
    return r.value


def paged_decode_attention_cascade(p: int, q, block_tables, max_blocks: int, seq_lens, batch: int,
                                   num_q_heads: int, scale: float, group_seqs, num_groups: int,
                                   group_size: int, shared_tokens, max_prefix_blocks: int,
                                   prefix_splits: int, out, out_dtype: int, lse_out=None,
                                   num_splits: int = 0, workspace=None, workspace_bytes: int = 0,
                                   stream=None, seq_order=None):
    """Decode with each group's shared prefix blocks read once; see the C header."""
    _check(lib().paged_decode_attention_cascade(
        p, _ptr(q), _ptr(block_tables), max_blocks, _ptr(seq_lens), batch, num_q_heads, scale,
        _ptr(group_seqs), num_groups, group_size, _ptr(shared_tokens), max_prefix_blocks,
        prefix_splits, _ptr(out), out_dtype, _ptr(lse_out), num_splits, _ptr(seq_order),
        _ptr(workspace), workspace_bytes, _stream(stream)), "paged_decode_attention_cascade")


def paged_prefill_attention(p: int, q, cu_q, total_q: int, max_q_len: int, block_tables,
                            max_blocks: int, seq_lens, batch: int, num_q_heads: int, scale: float,
                            out, out_dtype: int, lse_out=None, stream=None):
    _check(lib().paged_prefill_attention(p, _ptr(q), _ptr(cu_q), total_q, max_q_len,
                                         _ptr(block_tables), max_blocks, _ptr(seq_lens), batch,
                                         num_q_heads, scale, _ptr(out), out_dtype, _ptr(lse_out),
                                         _stream(stream)),
           "paged_prefill_attention")


def kv_get_device_error(p: int, stream=None) -> int:
    """Returns the device error bits (and clears them); never raises on set bits."""
    code = _i32()
    st = lib().kv_get_device_error(p, ctypes.byref(code), _stream(stream))
    if st not in (0, -3, -5, -6):
        raise KVError(st, "kv_get_device_error")
    return code.value


# ---------------------------------------------------------------- contiguous path
def kv_contig_create(max_requests, max_tokens, num_kv_heads, head_dim, dtype) -> int:
    h = _vp()
    _check(lib().kv_contig_create(max_requests, max_tokens, num_kv_heads, head_dim, dtype,
                                  ctypes.byref(h)), "kv_contig_create")
    return h.value


def kv_contig_destroy(c: int):
    _check(lib().kv_contig_destroy(c), "kv_contig_destroy")


def kv_contig_layout(c: int):
    hs, pg, rb = _i64(), _i64(), _i64()
    _check(lib().kv_contig_layout(c, ctypes.byref(hs), ctypes.byref(pg), ctypes.byref(rb)),
           "kv_contig_layout")
    return hs.value, pg.value, rb.value


def kv_contig_reserve(c: int, req: int):
    _check(lib().kv_contig_reserve(c, req), "kv_contig_reserve")


def kv_contig_ensure(c: int, req: int, n_tokens: int):
    _check(lib().kv_contig_ensure(c, req, n_tokens), "kv_contig_ensure")


def kv_contig_release(c: int, req: int):
    _check(lib().kv_contig_release(c, req), "kv_contig_release")


def kv_contig_ptrs(c: int, req: int):
    k, v = _vp(), _vp()
    _check(lib().kv_contig_ptrs(c, req, ctypes.byref(k), ctypes.byref(v)), "kv_contig_ptrs")
    return k.value, v.value


def kv_contig_page_pool(c: int, low: int, high: int):
    _check(lib().kv_contig_page_pool(c, low, high), "kv_contig_page_pool")


def kv_contig_page_stats(c: int):
    sp, cr, ru = _i32(), _i64(), _i64()
    mu, uu = ctypes.c_double(), ctypes.c_double()
    _check(lib().kv_contig_page_stats(c, ctypes.byref(sp), ctypes.byref(cr), ctypes.byref(ru),
                                      ctypes.byref(mu), ctypes.byref(uu)), "kv_contig_page_stats")
    return dict(spare=sp.value, created=cr.value, reused=ru.value, map_us=mu.value, unmap_us=uu.value)


def kv_contig_stats(c: int, req: int):
    t, b = _i64(), _i64()
    _check(lib().kv_contig_stats(c, req, ctypes.byref(t), ctypes.byref(b)), "kv_contig_stats")
    return t.value, b.value


def kv_contig_append(c: int, k_new, v_new, req_ids, positions, num_tokens: int, stream=None):
    _check(lib().kv_contig_append(c, _ptr(k_new), _ptr(v_new), _ptr(req_ids), _ptr(positions),
                                  num_tokens, _stream(stream)), "kv_contig_append")


def contig_decode_attention(c: int, q, req_ids, seq_lens, batch: int, num_q_heads: int,
                            scale: float, out, out_dtype: int, lse_out=None, num_splits: int = 0,
                            workspace=None, workspace_bytes: int = 0, stream=None):
    _check(lib().contig_decode_attention(c, _ptr(q), _ptr(req_ids), _ptr(seq_lens), batch,
                                         num_q_heads, scale, _ptr(out), out_dtype, _ptr(lse_out),
                                         num_splits, _ptr(workspace), workspace_bytes,
                                         _stream(stream)),
           "contig_decode_attention")


def contig_append_and_decode(c: int, q, k_new, v_new, req_ids, seq_lens, batch: int,
                             num_q_heads: int, scale: float, out, out_dtype: int, lse_out=None,
                             num_splits: int = 0, workspace=None, workspace_bytes: int = 0,
                             stream=None):
    """Each sequence's new token at position seq_lens[b] - 1 of its request,
    then contig_decode_attention (one fused launch where supported).  See the
    C header."""
    _check(lib().contig_append_and_decode(c, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(req_ids),
                                          _ptr(seq_lens), batch, num_q_heads, scale, _ptr(out),
                                          out_dtype, _ptr(lse_out), num_splits, _ptr(workspace),
                                          workspace_bytes, _stream(stream)),
           "contig_append_and_decode")


def kv_contig_set_launch_overlap(c: int, enable: bool):
    """Let this context's appends and decodes overlap the previous kernel in
    their stream (each waits for it before touching memory)."""
    _check(lib().kv_contig_set_launch_overlap(c, 1 if enable else 0), "kv_contig_set_launch_overlap")


def kv_contig_get_device_error(c: int, stream=None) -> int:
    code = _i32()
    st = lib().kv_contig_get_device_error(c, ctypes.byref(code), _stream(stream))
    if st not in (0, -5, -6):
        raise KVError(st, "kv_contig_get_device_error")
    return code.value


# ---------------------------------------------------------------- test hooks
def kv_debug_set_wait_limit_ns(ns: int):
    """Time limit of the kernels' pipeline waits on the current device (tests
    only; KV_WAIT_LIMIT_DEFAULT_NS restores the default)."""
    _check(lib().kv_debug_set_wait_limit_ns(int(ns)), "kv_debug_set_wait_limit_ns")


def kv_debug_fail_page_create(after: int):
    """The contiguous path's page creation after `after` more successful ones
    fails once (tests only; negative cancels)."""
    _check(lib().kv_debug_fail_page_create(int(after)), "kv_debug_fail_page_create")
