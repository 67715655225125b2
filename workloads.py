"""Seeded synthetic inputs for the paged KV-cache hot path.

This module is shared by the tests (which feed the same arrays to the CUDA
library and to the CPU oracle) and by ``bench.py``.  It holds NO arithmetic of
the method: it only draws random numbers (lengths, permutations, N(0,1)
values rounded once to bfloat16) and describes the five workload shapes.
Block tables, slot mappings and pool sizes are computed by the callers, each
side with its own code.

The shapes stand in for the workloads the vAttention and PagedAttention
evaluations use (Llama-3-8B / Yi-6B / Yi-34B head layouts, contexts up to
192K tokens); no model weights or traces are involved.

bfloat16 data is carried as ``np.uint16`` bit patterns; fp32 as ``np.float32``;
IEEE half precision as ``np.float16``.
"""
import numpy as np

BLOCK_SIZE = 16  # tokens per KV block, the size the PagedAttention pages use

# One entry per workload; ``seed`` = 1960 + index.
CONFIGS = {
    # 2 sequences (35 and 17 tokens), pool of 16 physical blocks assigned by a
    # seeded permutation, 4 query heads / 2 kv heads, head_dim 64, fp32.
    "tiny_fp32": dict(index=1, seed=1961, batch=2, lens=(35, 17), num_blocks=16,
                      num_q_heads=4, num_kv_heads=2, head_dim=64, dtype="f32"),
    # Llama-3-8B-shaped decode: 64 sequences, lengths uniform in [512, 4096],
    # 32 q heads / 8 kv heads, head_dim 128, pool 1.2x the blocks needed, shuffled.
    "llama3_8b_decode": dict(index=2, seed=1962, batch=64, len_lo=512, len_hi=4096,
                             len_dist="uniform", pool_factor=1.2, num_q_heads=32,
                             num_kv_heads=8, head_dim=128, dtype="bf16"),
    # Yi-6B-shaped long-context decode: 8 sequences, lengths log-uniform in
    # [32768, 196608], 32 q heads / 4 kv heads, head_dim 128; split-KV; the same
    # inputs also go through the contiguous (virtual-memory-backed) path.
    "yi6b_long_decode": dict(index=3, seed=1963, batch=8, len_lo=32768, len_hi=196608,
                             len_dist="log_uniform", pool_factor=1.2, num_q_heads=32,
                             num_kv_heads=4, head_dim=128, dtype="bf16"),
    # Append + one decode step with a shared prefix: 256 sequences with cached
    # lengths uniform in [128, 2048]; groups of 16 share a 1024-token prefix as
    # the same physical blocks; one new token per sequence.
    "shared_prefix_step": dict(index=4, seed=1964, batch=256, len_lo=128, len_hi=2048,
                               len_dist="uniform", group_size=16, prefix_len=1024,
                               pool_factor=1.2, num_q_heads=32, num_kv_heads=8,
                               head_dim=128, dtype="bf16"),
    # Yi-34B-shaped chunked causal prefill: 4 sequences with 8192 cached tokens
    # in shuffled blocks plus a new 2048-token chunk; 56 q heads / 8 kv heads.
    "yi34b_prefill": dict(index=5, seed=1965, batch=4, cached_len=8192, chunk_len=2048,
                          pool_factor=1.0, num_q_heads=56, num_kv_heads=8, head_dim=128,
                          dtype="bf16"),
}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(g: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0, 1) samples drawn in fp32; bf16 and f16 data are rounded once from
    them (round to nearest, ties to even)."""
    x = g.standard_normal(size=shape, dtype=np.float32)
    if dtype == "bf16":
        return to_bf16_bits(x)
    if dtype == "f16":
        return x.astype(np.float16)
    return x


def lengths(g: np.random.Generator, cfg: dict) -> np.ndarray:
    """Context lengths of a workload, int32."""
    if "lens" in cfg:
        return np.asarray(cfg["lens"], np.int32)
    if "cached_len" in cfg:
        return np.full(cfg["batch"], cfg["cached_len"] + cfg["chunk_len"], np.int32)
    lo, hi, B = cfg["len_lo"], cfg["len_hi"], cfg["batch"]
    if cfg["len_dist"] == "uniform":
        return g.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    u = g.uniform(np.log(lo), np.log(hi), size=B)
    return np.floor(np.exp(u)).astype(np.int32)


def permutation(g: np.random.Generator, n: int) -> np.ndarray:
    """A seeded random order of physical block ids 0..n-1 (int32)."""
    return g.permutation(n).astype(np.int32)


def empty_pool(num_blocks: int, num_kv_heads: int, head_dim: int, dtype: str,
               fill=None) -> np.ndarray:
    """Pool array [num_blocks][Hkv][BLOCK_SIZE][D]; optionally filled with a bit pattern."""
    shape = (num_blocks, num_kv_heads, BLOCK_SIZE, head_dim)
    if dtype == "bf16":
        return np.full(shape, 0 if fill is None else fill, np.uint16)
    if dtype == "f16":
        return np.full(shape, 0 if fill is None else fill, np.uint16).view(np.float16)
    a = np.zeros(shape, np.float32)
    if fill is not None:
        a.view(np.uint32)[...] = fill
    return a


NAN_BF16 = 0x7FC1      # quiet-NaN bit patterns used as "never written" sentinels
NAN_F16 = 0x7E01
NAN_F32 = 0x7FC00001


def decode_inputs(name: str, num_blocks: int, seed_offset: int = 0, dtype=None) -> dict:
    """Random draws for a paged-decode workload, in a fixed order.

    Returns lens [B], perm [num_blocks], pool_k / pool_v [NB][Hkv][16][D], q [B][Hq][D].
    The caller sizes the pool (``num_blocks``) and builds the block tables.
    ``dtype`` overrides the workload's storage type (the same draws, rounded
    to that type).
    """
    cfg = CONFIGS[name]
    dt = dtype or cfg["dtype"]
    g = rng(cfg["seed"] + seed_offset)
    lens = lengths(g, cfg)
    perm = permutation(g, num_blocks)
    shape = (num_blocks, cfg["num_kv_heads"], BLOCK_SIZE, cfg["head_dim"])
    pool_k = normal(g, shape, dt)
    pool_v = normal(g, shape, dt)
    q = normal(g, (len(lens), cfg["num_q_heads"], cfg["head_dim"]), dt)
    return dict(lens=lens, perm=perm, pool_k=pool_k, pool_v=pool_v, q=q)


def decode_lengths(name: str, seed_offset: int = 0) -> np.ndarray:
    """The lengths ``decode_inputs`` would draw (they are drawn first)."""
    cfg = CONFIGS[name]
    return lengths(rng(cfg["seed"] + seed_offset), cfg)


def shared_prefix_inputs(name: str = "shared_prefix_step", seed_offset: int = 0,
                         batch=None, dtype=None) -> dict:
    """Logical content of the shared-prefix step.

    lens [B] = cached lengths before the step; prefix_k/v [groups][prefix_len][Hkv][D];
    suffix_k/v: list of [max(L - prefix_len, 0)][Hkv][D] per sequence;
    new_k/new_v [B][Hkv][D] (the token appended this step); q [B][Hq][D].
    Sequence b belongs to group b // group_size and its first min(L, prefix_len)
    tokens are that group's prefix.  ``dtype`` overrides the storage type.
    """
    cfg = dict(CONFIGS[name])
    if batch is not None:
        cfg["batch"] = batch
    if dtype is not None:
        cfg["dtype"] = dtype
    g = rng(cfg["seed"] + seed_offset)
    lens = lengths(g, cfg)
    B, P, Hkv, D, dt = cfg["batch"], cfg["prefix_len"], cfg["num_kv_heads"], cfg["head_dim"], cfg["dtype"]
    groups = -(-B // cfg["group_size"])
    prefix_k = normal(g, (groups, P, Hkv, D), dt)
    prefix_v = normal(g, (groups, P, Hkv, D), dt)
    suffix_k, suffix_v = [], []
    for L in lens:
        n = max(int(L) - P, 0)
        suffix_k.append(normal(g, (n, Hkv, D), dt))
        suffix_v.append(normal(g, (n, Hkv, D), dt))
    new_k = normal(g, (B, Hkv, D), dt)
    new_v = normal(g, (B, Hkv, D), dt)
    q = normal(g, (B, cfg["num_q_heads"], D), dt)
    return dict(lens=lens, prefix_k=prefix_k, prefix_v=prefix_v, suffix_k=suffix_k,
                suffix_v=suffix_v, new_k=new_k, new_v=new_v, q=q, group_size=cfg["group_size"],
                prefix_len=P, dtype=dt)


def prefill_inputs(name: str, num_blocks: int, batch=None, cached_len=None, chunk_len=None,
                   seed_offset: int = 0, dtype=None) -> dict:
    """Random draws for the chunked-prefill workload.

    Returns cached_lens [B], chunk_lens [B], perm [num_blocks], pool_k / pool_v
    (cached tokens' content; every slot drawn), k_new / v_new [sum T][Hkv][D]
    and q [sum T][Hq][D].  ``dtype`` overrides the storage type.
    """
    cfg = dict(CONFIGS[name])
    for k, v in (("batch", batch), ("cached_len", cached_len), ("chunk_len", chunk_len),
                 ("dtype", dtype)):
        if v is not None:
            cfg[k] = v
    g = rng(cfg["seed"] + seed_offset)
    B = cfg["batch"]
    cached = np.full(B, cfg["cached_len"], np.int32)
    chunk = np.full(B, cfg["chunk_len"], np.int32)
    perm = permutation(g, num_blocks)
    shape = (num_blocks, cfg["num_kv_heads"], BLOCK_SIZE, cfg["head_dim"])
    pool_k = normal(g, shape, cfg["dtype"])
    pool_v = normal(g, shape, cfg["dtype"])
    T = int(chunk.sum())
    k_new = normal(g, (T, cfg["num_kv_heads"], cfg["head_dim"]), cfg["dtype"])
    v_new = normal(g, (T, cfg["num_kv_heads"], cfg["head_dim"]), cfg["dtype"])
    q = normal(g, (T, cfg["num_q_heads"], cfg["head_dim"]), cfg["dtype"])
    return dict(cached_lens=cached, chunk_lens=chunk, perm=perm, pool_k=pool_k, pool_v=pool_v,
                k_new=k_new, v_new=v_new, q=q)
