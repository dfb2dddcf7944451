"""A seeded sweep of random shapes through every entry point, against the
fp64 oracle: contiguous calls with and without a workspace, caller layouts
(strided rows, cache capacity, circular caches) and device-side lengths,
bf16 head_dim 128 / 512 and fp32 head_dim 128 / others.  The hand-picked
cases elsewhere cover the named corner cases; this catches combinations
nobody picked."""
import numpy as np
import pytest
import torch

import chunked_causal_gqa_gb300 as pkg
import oracle
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

_TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


def _draw_case(rng):
    dtype = "bf16" if rng.random() < 0.7 else "f32"
    if dtype == "bf16":
        D = 128 if rng.random() < 0.75 else 512
    else:
        D = 128 if rng.random() < 0.6 else int(rng.choice([32, 64, 96, 256]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 2, 3, 4, 8]))
    H = Hkv * group
    T = int(rng.choice([1, 2, 17, 64, 127, 129, 300, 700]))
    sp = int(rng.choice([0, 1, 50, 128, 1000, 4000]))
    window = int(rng.choice([0, 0, 1, 64, 200, 1024]))
    entry = str(rng.choice(["plain", "ws", "cache", "ring", "graph"]))
    if entry == "ring" and window == 0:
        window = 256
    return dict(dtype=dtype, D=D, H=H, Hkv=Hkv, T=T, sp=sp, window=window, entry=entry,
                seed=int(rng.integers(0, 100000)))


CASES = [_draw_case(np.random.default_rng(9000 + i)) for i in range(100)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "{entry}_{dtype}_D{D}_H{H}_Hkv{Hkv}_T{T}_sp{sp}_w{window}".format(**c))
def test_random_shape(case):
    dtype, D, H, Hkv, T, sp, w, entry = (case[k] for k in
                                         ("dtype", "D", "H", "Hkv", "T", "sp", "window", "entry"))
    seed = case["seed"]
    q, k, v = W.make_random(T, sp, H, Hkv, D, dtype, seed=seed, q_std=1.0, kv_std=0.5)
    L = sp + T
    d = G.dev()
    tol = "f32" if dtype == "f32" else "bf16"
    if entry in ("plain", "ws"):
        got = G.run(q, k, v, window=w, workspace=None if entry == "plain" else "auto")
        G.check(G.to_np(got), oracle.prefill_attention(q, k, v, window=w), tol, str(case))
        return
    if entry == "graph":
        cap = L + 37
        kc = torch.zeros(Hkv, cap, D, dtype=_TORCH[dtype])
        vc = torch.zeros_like(kc)
        kc[:, :L] = k
        vc[:, :L] = v
        max_T = T + 5
        qb = torch.zeros(max_T, H, D, dtype=_TORCH[dtype])
        qb[:T] = q
        out = torch.full((max_T, H, D), 3.0, dtype=_TORCH[dtype], device=d)
        lens = torch.tensor([T, sp], dtype=torch.int64, device=d)
        pkg.prefill_attention_graph(qb.to(d), kc.to(d), vc.to(d), out, lens, window=w)
        assert pkg.last_device_error() == 0
        o = G.to_np(out)
        G.check(o[:T], oracle.prefill_attention(q, k, v, window=w), tol, str(case))
        assert np.all(o[T:] == 3.0)
        return
    # caller layouts: padded q/out rows, capacity past L, or a circular cache
    pad = 8 if dtype == "bf16" else 4
    qkv_dim = H * D + pad
    qb = torch.randn(T, qkv_dim).to(_TORCH[dtype])
    qb[:, :H * D] = q.reshape(T, H * D)
    if entry == "ring":
        need = min(L, w + T - 1)
        cap = max(128, ((need + 127) // 128) * 128) if dtype == "bf16" else need
        kc = torch.randn(Hkv, cap, D).to(_TORCH[dtype])
        vc = torch.randn(Hkv, cap, D).to(_TORCH[dtype])
        j = torch.arange(max(0, L - cap), L)
        kc[:, j % cap] = k[:, j]
        vc[:, j % cap] = v[:, j]
    else:
        cap = L + 100
        kc = torch.randn(Hkv, cap, D).to(_TORCH[dtype])
        vc = torch.randn(Hkv, cap, D).to(_TORCH[dtype])
        kc[:, :L] = k
        vc[:, :L] = v
    ob = torch.full((T, qkv_dim), 5.0, dtype=_TORCH[dtype], device=d)
    qd = qb.to(d)
    pkg.prefill_attention_cache(qd[:, :H * D].view(T, H, D), kc.to(d), vc.to(d),
                                ob[:, :H * D].view(T, H, D), start_pos=sp, window=w,
                                ring=(entry == "ring"))
    assert pkg.last_device_error() == 0
    o = G.to_np(ob)
    want = oracle.prefill_attention(q, k, v, window=w)
    G.check(o[:, :H * D].reshape(T, H, D), want, tol, str(case))
    assert np.all(o[:, H * D:] == 5.0)
