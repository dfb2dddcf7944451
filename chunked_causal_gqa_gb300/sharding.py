"""Head sharding of one layer's prefill attention across ranks.

The operation needs no exchange between kv heads: kv head j and the query
heads j*group .. (j+1)*group-1 that read it (contiguous GQA groups, gnosis
"Prefill attention -> GPU: handoff", section "GPU design", GQA bullet) form an
independent problem.  A rank that owns kv heads [a, b) computes the output
columns of query heads [a*group, b*group) from its own slices of q and the
cache; the outputs concatenate along the head axis.
"""
from __future__ import annotations


def kv_head_range(num_kv_heads: int, world: int, rank: int) -> tuple:
    """Contiguous, balanced [start, stop) of kv heads owned by `rank`."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    base, extra = divmod(num_kv_heads, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard(q, k_cache, v_cache, world: int, rank: int):
    """This rank's (q [T, Hs, D], k [Hkv_s, L, D], v) slices and its query-head range."""
    H, Hkv = q.shape[1], k_cache.shape[0]
    if H % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    g = H // Hkv
    a, b = kv_head_range(Hkv, world, rank)
    return (q[:, a * g:b * g], k_cache[a:b], v_cache[a:b]), (a * g, b * g)
