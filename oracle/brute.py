"""Pure-Python brute-force statement of paged attention -- TEST INFRASTRUCTURE ONLY.

A second, independent restatement used to pin the C oracle on tiny inputs.
It never touches the C code: it walks the block table token by token with
Python integers, builds the explicit score list, and sums with ``math.fsum``
(exactly rounded sums) so that its own rounding error is negligible.

Source: "PagedAttention Nedir?" (bitcanli.com), sections "PagedAttention
Nedir?" (blocks found through a mapping table, logical order preserved) and
"Nasil Calisir?" step 4 (attention reads K/V from the blocks' locations).
"""
import math


def _row(pool, block, head, offset):
    return [float(x) for x in pool[block][head][offset]]


def attention(q, keys, values, scale):
    """softmax(scale * q.k_j) weighted sum of values, with exact summation."""
    if not keys:
        return [0.0] * len(q), -math.inf
    scores = [scale * math.fsum(a * b for a, b in zip(q, k)) for k in keys]
    m = max(scores)
    w = [math.exp(s - m) for s in scores]
    l = math.fsum(w)
    out = [math.fsum(wj * v[d] for wj, v in zip(w, values)) / l for d in range(len(q))]
    return out, m + math.log(l)


def paged_decode(pool_k, pool_v, tables, lens, q, scale, block_size):
    """pool_* indexable as [block][head][offset][dim] (any nested sequence / array).

    q indexable as [b][hq][dim].  Returns nested lists out[b][hq][dim], lse[b][hq].
    """
    num_kv_heads = len(pool_k[0])
    out, lse = [], []
    for b, L in enumerate(lens):
        num_q_heads = len(q[b])
        group = num_q_heads // num_kv_heads
        ob, lb = [], []
        for hq in range(num_q_heads):
            h = hq // group
            keys, vals = [], []
            for j in range(int(L)):
                blk = int(tables[b][j // block_size])
                keys.append(_row(pool_k, blk, h, j % block_size))
                vals.append(_row(pool_v, blk, h, j % block_size))
            o, s = attention([float(x) for x in q[b][hq]], keys, vals, scale)
            ob.append(o)
            lb.append(s)
        out.append(ob)
        lse.append(lb)
    return out, lse
