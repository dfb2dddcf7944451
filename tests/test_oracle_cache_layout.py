"""The oracle's cache-layout entry (strided q/out rows, a cache allocated for
more positions than L, a circular cache for sliding-window layers) against
the contiguous entry, which the pins in test_oracle_pins.py fix.

The layouts follow the gnosis page "Prefill attention -> GPU: handoff"
(section "GPU design", "Layout": batch_q rows of qkv_dim elements, kv head kh
at kh * max_seq_len * head_dim) and the TensorSharp2 Gemma-4 prefill design
(section 4, R4: sliding-window layers write position pos at index
pos % capacity).  Every expected value here comes from the contiguous oracle
on arrays that numpy slicing, or a plain in-order replay of the ring writes,
extracts from the caller-layout buffers -- index arithmetic that is not the
oracle's own.
"""
import numpy as np
import pytest

import oracle


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _strided_case(rng, T, sp, H, Hkv, D, pad, extra_rows):
    """Caller-layout buffers with garbage in every element the call must not read."""
    L = sp + T
    qkv_dim = H * D + pad
    cap = L + extra_rows
    q_buf = _rand(rng, T, qkv_dim) * 1e3            # padding: large garbage
    k_buf = _rand(rng, Hkv, cap, D) * 1e3
    v_buf = _rand(rng, Hkv, cap, D) * 1e3
    q = q_buf[:, :H * D].reshape(T, H, D) / 1e3     # the heads, scaled back to N(0,1)
    q_buf[:, :H * D] = q.reshape(T, H * D)
    k = _rand(rng, Hkv, L, D)
    v = _rand(rng, Hkv, L, D)
    k_buf[:, :L] = k
    v_buf[:, :L] = v
    return q_buf, k_buf, v_buf, q, k, v, qkv_dim, cap


@pytest.mark.parametrize("T,sp,H,Hkv,D,window,pad,extra", [
    (7, 0, 4, 2, 8, 0, 8, 0),
    (9, 13, 8, 2, 16, 0, 24, 37),
    (6, 20, 4, 1, 4, 5, 4, 3),
    (1, 30, 2, 2, 8, 0, 0, 64),
])
def test_strided_rows_and_capacity_match_contiguous(T, sp, H, Hkv, D, window, pad, extra):
    rng = np.random.default_rng(1000 + T + sp)
    q_buf, k_buf, v_buf, q, k, v, qkv_dim, cap = _strided_case(rng, T, sp, H, Hkv, D, pad,
                                                               extra)
    out_init = _rand(rng, T * qkv_dim)
    got = oracle.prefill_attention_cache(q_buf, k_buf, v_buf, T, sp, H, Hkv, D, window=window,
                                         qkv_dim=qkv_dim, max_seq_len=cap, out_init=out_init,
                                         threads=2).reshape(T, qkv_dim)
    want = oracle.prefill_attention(q, k, v, window=window, threads=2)
    assert np.array_equal(got[:, :H * D].reshape(T, H, D), want)
    # elements outside the heads keep what the caller had there
    assert np.array_equal(got[:, H * D:], out_init.reshape(T, qkv_dim)[:, H * D:])


def _ring_fill(k_full, cap):
    """Replay the cache writes of positions 0 .. L-1 in order into a ring of cap rows."""
    Hkv, L, D = k_full.shape
    ring = np.full((Hkv, cap, D), np.nan)
    for j in range(L):
        ring[:, j % cap] = k_full[:, j]
    return ring


@pytest.mark.parametrize("T,sp,H,Hkv,D,window,cap", [
    (6, 40, 4, 2, 8, 8, 13),      # cap = window + T - 1: the least that works, wrapped
    (6, 40, 4, 2, 8, 8, 16),
    (3, 100, 2, 1, 4, 1, 3),      # window 1: each row sees only itself
    (5, 2, 4, 2, 8, 6, 16),       # L <= cap: no wrap yet
    (12, 77, 8, 2, 8, 10, 32),
])
def test_ring_cache_matches_linear(T, sp, H, Hkv, D, window, cap):
    rng = np.random.default_rng(2000 + cap + sp)
    L = sp + T
    q = _rand(rng, T, H, D)
    k = _rand(rng, Hkv, L, D)
    v = _rand(rng, Hkv, L, D)
    kr, vr = _ring_fill(k, cap), _ring_fill(v, cap)
    # slots never written (L < cap) stay NaN: the oracle must never read them
    got = oracle.prefill_attention_cache(q, kr, vr, T, sp, H, Hkv, D, window=window,
                                         max_seq_len=cap, ring=True, threads=2)
    want = oracle.prefill_attention(q, k, v, window=window, threads=2)
    assert np.array_equal(got.reshape(T, H, D), want)


def test_ring_multi_chunk_prefill_past_the_window():
    """Chunked prefill through a circular cache equals one-shot attention.

    Each chunk first writes its own keys at pos % cap, then attends; the ring
    holds window + chunk - 1 rows, the least that keeps every visible key.
    """
    rng = np.random.default_rng(3000)
    H, Hkv, D, window, chunk = 4, 2, 8, 9, 5
    total = 41
    cap = window + chunk - 1
    q = _rand(rng, total, H, D)
    k = _rand(rng, Hkv, total, D)
    v = _rand(rng, Hkv, total, D)
    want = oracle.prefill_attention(q, k, v, window=window, threads=2)
    kr = np.full((Hkv, cap, D), np.nan)
    vr = np.full((Hkv, cap, D), np.nan)
    for sp in range(0, total, chunk):
        T = min(chunk, total - sp)
        for j in range(sp, sp + T):
            kr[:, j % cap] = k[:, j]
            vr[:, j % cap] = v[:, j]
        got = oracle.prefill_attention_cache(q[sp:sp + T], kr, vr, T, sp, H, Hkv, D,
                                             window=window, max_seq_len=cap, ring=True,
                                             threads=2)
        assert np.array_equal(got.reshape(T, H, D), want[sp:sp + T])


@pytest.mark.parametrize("plant", ["ring_offset", "qkv_stride", "kv_stride"])
def test_layout_plants_are_caught(plant):
    rng = np.random.default_rng(4000)
    T, sp, H, Hkv, D, window, cap = 6, 40, 4, 2, 8, 8, 16
    L = sp + T
    q_buf, k_buf, v_buf, q, k, v, qkv_dim, _ = _strided_case(rng, T, sp, H, Hkv, D, 8, 0)
    want = oracle.prefill_attention(q, k, v, window=window, threads=1)
    if plant == "ring_offset":
        kr, vr = _ring_fill(k, cap), _ring_fill(v, cap)
        got = oracle.prefill_attention_cache(q, kr, vr, T, sp, H, Hkv, D, window=window,
                                             max_seq_len=cap, ring=True, threads=1,
                                             plant=plant).reshape(T, H, D)
    else:
        got = oracle.prefill_attention_cache(q_buf, k_buf, v_buf, T, sp, H, Hkv, D,
                                             window=window, qkv_dim=qkv_dim, max_seq_len=L,
                                             threads=1, plant=plant)
        got = got.reshape(T, qkv_dim)[:, :H * D].reshape(T, H, D)
    assert not np.allclose(got, want, atol=1e-6, equal_nan=False)


def test_cache_layout_arguments_are_checked():
    rng = np.random.default_rng(5)
    T, sp, H, Hkv, D = 4, 10, 2, 1, 4
    q = _rand(rng, T, H, D)
    k = _rand(rng, Hkv, 32, D)
    with pytest.raises(ValueError):     # circular cache needs a window
        oracle.prefill_attention_cache(q, k, k, T, sp, H, Hkv, D, window=0, max_seq_len=8,
                                       ring=True)
    with pytest.raises(ValueError):     # ring smaller than window + T - 1
        oracle.prefill_attention_cache(q, k, k, T, sp, H, Hkv, D, window=6, max_seq_len=8,
                                       ring=True)
    with pytest.raises(ValueError):     # linear cache shorter than L
        oracle.prefill_attention_cache(q, k, k, T, sp, H, Hkv, D, max_seq_len=13)
    with pytest.raises(ValueError):     # rows shorter than the heads
        oracle.prefill_attention_cache(q, k, k, T, sp, H, Hkv, D, qkv_dim=H * D - 1,
                                       max_seq_len=14)
