"""pfa_prefill_attention_cache on the GPU against the oracle's cache-layout
entry: strided q / out rows, caches allocated for more positions than L, and
circular (ring) caches of sliding-window layers, for bf16 head_dim 128 and
512 and for fp32.

The inputs are the exact buffers the kernels read, with garbage in every
element the call must ignore (q row padding, cache rows past L); elements of
out outside the heads must come back unchanged.
"""
import numpy as np
import pytest
import torch

import chunked_causal_gqa_gb300 as pkg
import oracle
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

_TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


def _buffers(T, sp, H, Hkv, D, dtype, pad, cap, ring, seed):
    """(q_buf [T, qkv_dim], k_buf, v_buf [Hkv, cap, D], qkv_dim) on the host."""
    L = sp + T
    q, k, v = W.make_random(T, sp, H, Hkv, D, dtype, seed=seed, q_std=1.0, kv_std=0.5)
    g = torch.Generator().manual_seed(seed + 99)
    qkv_dim = H * D + pad
    q_buf = (torch.randn(T, qkv_dim, generator=g) * 100).to(_TORCH[dtype])
    q_buf[:, :H * D] = q.reshape(T, H * D)
    k_buf = (torch.randn(Hkv, cap, D, generator=g) * 100).to(_TORCH[dtype])
    v_buf = (torch.randn(Hkv, cap, D, generator=g) * 100).to(_TORCH[dtype])
    if ring:
        # the cache writes of positions 0 .. L-1, in order: the last min(L, cap)
        # positions are the ones left in the ring
        j = torch.arange(max(0, L - cap), L)
        k_buf[:, j % cap] = k[:, j]
        v_buf[:, j % cap] = v[:, j]
    else:
        k_buf[:, :L] = k
        v_buf[:, :L] = v
    return q_buf, k_buf, v_buf, qkv_dim


def _run_case(T, sp, H, Hkv, D, window, dtype, pad, cap, ring, workspace="auto", seed=0):
    q_buf, k_buf, v_buf, qkv_dim = _buffers(T, sp, H, Hkv, D, dtype, pad, cap, ring, seed)
    d = G.dev()
    qd, kd, vd = q_buf.to(d), k_buf.to(d), v_buf.to(d)
    sentinel = torch.full((T, qkv_dim), 7.0, dtype=_TORCH[dtype], device=d)
    q_view = qd[:, :H * D].view(T, H, D)
    out_view = sentinel[:, :H * D].view(T, H, D)
    pkg.prefill_attention_cache(q_view, kd, vd, out_view, start_pos=sp, window=window,
                                ring=ring, workspace=workspace)
    assert pkg.last_device_error() == 0
    got = G.to_np(sentinel)
    want = oracle.prefill_attention_cache(q_buf, k_buf, v_buf, T, sp, H, Hkv, D, window=window,
                                          qkv_dim=qkv_dim, max_seq_len=cap, ring=ring,
                                          out_init=np.full(T * qkv_dim, 7.0)).reshape(T, qkv_dim)
    G.check(got[:, :H * D], want[:, :H * D], dtype,
            f"T{T} sp{sp} H{H}/{Hkv} D{D} w{window} {dtype} pad{pad} cap{cap} ring{ring}")
    assert np.all(got[:, H * D:] == 7.0), "elements outside the heads were written"


# (T, start_pos, H, Hkv, D, window, dtype, pad, rows past L, ring)
LINEAR = [
    (300, 200, 32, 8, 128, 0, "bf16", 64, 300, False),
    (257, 0, 8, 2, 128, 0, "bf16", 8, 1000, False),
    (200, 500, 8, 2, 128, 129, "bf16", 128, 77, False),
    (130, 100, 8, 2, 512, 0, "bf16", 512, 200, False),
    (130, 100, 8, 2, 512, 0, "bf16", 8, 200, False),      # rows 16 B (not 32 B) aligned
    (77, 30, 8, 2, 64, 0, "f32", 4, 50, False),
    (40, 10, 4, 1, 128, 7, "f32", 128, 1, False),
]


@pytest.mark.parametrize("case", LINEAR,
                         ids=lambda c: "T%d_sp%d_H%d_Hkv%d_D%d_w%d_%s_pad%d_extra%d_%s" % c)
def test_strided_rows_and_capacity(case):
    T, sp, H, Hkv, D, window, dtype, pad, extra, ring = case
    _run_case(T, sp, H, Hkv, D, window, dtype, pad, sp + T + extra, ring, seed=T + sp)


# (T, start_pos, H, Hkv, D, window, dtype, pad, capacity, ring)
RING = [
    (200, 3000, 32, 8, 128, 256, "bf16", 0, 512, True),     # wrapped; 455 <= 512
    (300, 5000, 8, 2, 128, 1024, "bf16", 0, 1408, True),    # Gemma-like window, wrapped
    (100, 50, 8, 2, 128, 64, "bf16", 0, 256, True),         # L <= capacity: not wrapped
    (128, 9000, 8, 2, 512, 1024, "bf16", 512, 1152, True),  # head_dim 512, wrapped
    (60, 700, 8, 2, 64, 40, "f32", 4, 99, True),            # fp32: any capacity >= w + T - 1
    (60, 700, 8, 2, 128, 40, "f32", 4, 99, True),           # fp32 head_dim 128 (paired CTAs)
    (1, 12345, 8, 2, 128, 128, "bf16", 0, 128, True),       # one token, ring of one tile
]


@pytest.mark.parametrize("case", RING,
                         ids=lambda c: "T%d_sp%d_H%d_Hkv%d_D%d_w%d_%s_pad%d_cap%d_%s" % c)
@pytest.mark.parametrize("workspace", ["auto", None])
def test_ring_cache(case, workspace):
    T, sp, H, Hkv, D, window, dtype, pad, cap, ring = case
    _run_case(T, sp, H, Hkv, D, window, dtype, pad, cap, ring, workspace=workspace,
              seed=cap + T)


@pytest.mark.parametrize("D", [128, 512])
def test_ring_chunked_prefill_past_the_window(D):
    """A prompt prefilled chunk by chunk through a ring cache equals one-shot
    attention: each chunk writes its keys at pos % capacity, then attends."""
    H, Hkv, window, chunk, total = 8, 2, 256, 256, 1500
    cap = 512                                   # >= window + chunk - 1, multiple of 128
    q, k, v = W.make_random(total, 0, H, Hkv, D, "bf16", seed=D, q_std=1.0, kv_std=0.5)
    want = oracle.prefill_attention(q, k, v, window=window)
    d = G.dev()
    kr = torch.zeros(Hkv, cap, D, dtype=torch.bfloat16, device=d)
    vr = torch.zeros_like(kr)
    kd, vd, qd = k.to(d), v.to(d), q.to(d)
    for sp in range(0, total, chunk):
        T = min(chunk, total - sp)
        j = torch.arange(sp, sp + T, device=d)
        kr[:, j % cap] = kd[:, j]
        vr[:, j % cap] = vd[:, j]
        got = pkg.prefill_attention_cache(qd[sp:sp + T], kr, vr, start_pos=sp, window=window,
                                          ring=True)
        assert pkg.last_device_error() == 0
        G.check(G.to_np(got), want[sp:sp + T], "bf16", f"chunk at {sp}")


def test_cache_layout_errors():
    d = G.dev()
    H, Hkv, D, T, sp = 8, 2, 128, 64, 1000
    q = torch.zeros(T, H, D, dtype=torch.bfloat16, device=d)
    k = torch.zeros(Hkv, 512, D, dtype=torch.bfloat16, device=d)

    def status(**kw):
        kk = kw.pop("k", k)
        args = dict(start_pos=sp, window=256, ring=True)
        args.update(kw)
        try:
            pkg.prefill_attention_cache(q, kk, kk.clone(), **args)
        except pkg.PfaError as e:
            return e.name
        return "PFA_OK"

    assert status() == "PFA_OK"
    assert status(window=0) == "PFA_ERR_SHAPE"             # ring needs a window
    assert status(window=500) == "PFA_ERR_SHAPE"           # 500 + 63 > 512 rows
    k300 = torch.zeros(Hkv, 300, D, dtype=torch.bfloat16, device=d)
    assert status(k=k300, window=200) == "PFA_ERR_SHAPE"   # wrapped bf16 ring of 300 rows
    assert status(ring=False) == "PFA_ERR_SHAPE"           # linear cache shorter than L
    buf = torch.zeros(T, H * D + 4, dtype=torch.bfloat16, device=d)
    qs = buf[:, :H * D].view(T, H, D)                     # rows of 2056 bytes
    with pytest.raises(pkg.PfaError) as e:
        pkg.prefill_attention_cache(qs, k, k.clone(), start_pos=sp, window=256, ring=True)
    assert e.value.name == "PFA_ERR_ALIGNMENT"
    torch.cuda.synchronize()
    assert pkg.last_device_error() == 0


def test_ring_cache_with_the_tail_split():
    """The tail-split schedule reading a wrapped circular cache."""
    T, sp, H, Hkv, D, window, cap = 1280, 60000, 32, 8, 128, 1024, 2304
    assert pkg.schedule(T, sp, H, Hkv, D, window)[0] == "tail"
    _run_case(T, sp, H, Hkv, D, window, "bf16", 0, cap, True, workspace="auto", seed=1234)
