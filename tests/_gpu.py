"""Helpers for the GPU tests: device copies of numpy arrays, torch views of
library-owned device memory, tolerance checks.  No arithmetic of the method.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_196_gb300 as pk


def require_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    pk.lib()  # build / load; raises if the library is missing


def dev(a: np.ndarray) -> torch.Tensor:
    """Device copy of a numpy array; bf16 bit patterns (uint16) travel as int16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor, like_bf16=False) -> np.ndarray:
    a = t.detach().cpu().numpy()
    return a.view(np.uint16) if like_bf16 else a


class _Raw:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


def view(ptr: int, shape, bf16: bool, typestr=None) -> torch.Tensor:
    """A torch tensor aliasing library-owned device memory (no copy)."""
    return torch.as_tensor(_Raw(ptr, shape, typestr or ("<i2" if bf16 else "<f4")), device="cuda")


_cudart = None


def _rt():
    global _cudart
    if _cudart is None:
        import ctypes
        import glob
        cands = ["libcudart.so", "libcudart.so.13", "libcudart.so.12"]
        cands += sorted(glob.glob("/usr/local/cuda*/lib64/libcudart.so*"))
        for c in cands:
            try:
                _cudart = ctypes.CDLL(c)
                break
            except OSError:
                continue
        if _cudart is None:
            raise RuntimeError("libcudart not found")
        _cudart.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
    return _cudart


def read_linear(ptr: int, heads: int, stride_tokens: int, n_tokens: int, d: int, bf16: bool):
    """Copies rows 0..n_tokens-1 of every head of a [heads][stride][d] device
    region (any device address, e.g. virtual-memory-mapped) to a numpy array."""
    dt = np.uint16 if bf16 else np.float32
    e = 2 if bf16 else 4
    out = np.empty((heads, n_tokens, d), dt)
    torch.cuda.synchronize()
    for h in range(heads):
        if n_tokens:
            rc = _rt().cudaMemcpy(out[h].ctypes.data, ptr + h * stride_tokens * d * e,
                                  n_tokens * d * e, 2)  # device to host
            assert rc == 0, f"cudaMemcpy failed: {rc}"
    return out


def pool_views(pool, num_blocks, hkv, d, bf16):
    kp, vp = pk.kv_pool_ptrs(pool)
    shape = (num_blocks, hkv, 16, d)
    return view(kp, shape, bf16), view(vp, shape, bf16)


def assert_close_scaled(out, ref, rel, what=""):
    """max |out - ref| <= rel * max |ref| (the attention tolerance)."""
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(out - ref))) if ref.size else 0.0
    assert err <= rel * scale, f"{what}: max|err| {err:.3e} > {rel:g} * {scale:.3e}"
    return err / scale if scale else 0.0


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
