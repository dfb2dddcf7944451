"""Full-output fp64 oracle results of the named workloads, cached on disk.

The large configurations (the 64k and 128k chunks, the head_dim-512 layers)
take the oracle tens of seconds on a many-core host.  Their whole output is
computed once per input recipe and kept under oracle/_build/cache/ (ignored by
git), keyed by the workload's shape, window, scale and seeds and by the hash
of the oracle's C source, so a change to any of them recomputes it.  Only the
oracle writes these files; nothing from the CUDA path is ever stored.
"""
from __future__ import annotations

import hashlib
import os

import numpy as np

import oracle
from chunked_causal_gqa_gb300 import workloads as W

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CACHE_DIR = os.path.join(_ROOT, "oracle", "_build", "cache")
_memo: dict = {}


def _key(wl) -> str:
    h = hashlib.sha256()
    with open(os.path.join(_ROOT, "oracle", "pfa_oracle.c"), "rb") as f:
        h.update(f.read())
    h.update(repr((wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.T, wl.start_pos, wl.window,
                   wl.dtype, wl.q_std, wl.kv_std, tuple(wl.seeds), wl.scale)).encode())
    return h.hexdigest()[:20]


def full_output(wl, inputs=None) -> np.ndarray:
    """The oracle's [T][H][D] float64 output for workload `wl` (inputs from
    workloads.make_inputs, or the same tensors passed in)."""
    key = _key(wl)
    if key in _memo:
        return _memo[key]
    path = os.path.join(CACHE_DIR, f"{wl.name}-{key}.npy")
    want = None
    if os.path.isfile(path):
        try:
            want = np.load(path)
            if want.shape != (wl.T, wl.num_heads, wl.head_dim):
                want = None
        except (OSError, ValueError):
            want = None
    if want is None:
        q, k, v = inputs if inputs is not None else W.make_inputs(wl)
        want = oracle.prefill_attention(q, k, v, window=wl.window, scale=wl.scale)
        os.makedirs(CACHE_DIR, exist_ok=True)
        tmp = f"{path}.tmp{os.getpid()}.npy"
        np.save(tmp, want)
        os.replace(tmp, path)
    _memo.clear()          # keep one large result in memory at a time
    _memo[key] = want
    return want
