"""fp64 CPU oracle for chunked causal GQA prefill attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path
(``chunked_causal_gqa_gb300``) never imports this package, and this package
imports nothing from it.

The arithmetic lives in ``pfa_oracle.c`` (plain C, double precision), which
restates the per-(token, head) loop of the gnosis page "Prefill attention ->
GPU: handoff" (sections "What already shipped" and "GPU design": GQA mapping
kv_h = h / (H / Hkv), scale 1/sqrt(head_dim) applied before the row max,
keys j <= start_pos + t, softmax, weighted sum of V) plus the sliding-window
band (j > pos - window) of the TensorSharp2 Gemma-4 prefill design (section 5,
Option A, "causal(+windowed)" masks).  This module only compiles that file
with gcc, widens inputs to float64 and passes host arrays through ctypes.

Parity status: pinned (brute force in exact/high-precision arithmetic on
tiny inputs, closed forms, a hand-derived worked example under
tests/golden/, invariants and planted controls; see tests/test_oracle_*.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pfa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpfa_oracle.so")
_lock = threading.Lock()
_lib = None

# Planted-mistake codes understood by pfa_oracle_prefill_attention_planted.
PLANTS = {
    "mask_strict": 1,
    "window_wide": 2,
    "kv_head_modulo": 3,
    "no_scale": 4,
    "no_max_shift": 5,
    "kv_stride": 6,
    "window_narrow": 7,
    "ring_offset": 8,
    "qkv_stride": 9,
}


def build(force: bool = False) -> str:
    """Compile pfa_oracle.c into a shared library with gcc; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.pfa_oracle_prefill_attention.argtypes = [
            dp, dp, dp, dp, i64, i64, i32, i32, i32, i32, ctypes.c_double, i32]
        lib.pfa_oracle_prefill_attention.restype = i32
        lib.pfa_oracle_prefill_attention_planted.argtypes = [
            dp, dp, dp, dp, i64, i64, i32, i32, i32, i32, ctypes.c_double, i32, i32]
        lib.pfa_oracle_prefill_attention_planted.restype = i32
        lib.pfa_oracle_prefill_attention_rows.argtypes = [
            dp, dp, dp, i64, i64, i32, i32, i32, i32, ctypes.c_double,
            ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32), i64, dp, i32]
        lib.pfa_oracle_prefill_attention_rows.restype = i32
        lib.pfa_oracle_prefill_attention_cache.argtypes = [
            dp, dp, dp, dp, i64, i64, i32, i32, i32, i32, ctypes.c_double, i64, i64, i32, i32,
            i32]
        lib.pfa_oracle_prefill_attention_cache.restype = i32
        _lib = lib
        return lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(a) -> np.ndarray:
    """Host float64 copy of an array-like (numpy array or CPU torch tensor)."""
    if hasattr(a, "detach"):  # torch tensor: widen on the host
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(q, k, v):
    if q.ndim != 3 or k.ndim != 3 or v.ndim != 3 or k.shape != v.shape:
        raise ValueError("q must be [T][H][D]; k, v must be [Hkv][L][D] of equal shape")
    T, H, D = q.shape
    Hkv, L, Dk = k.shape
    if Dk != D:
        raise ValueError("head_dim mismatch")
    start_pos = L - T
    if start_pos < 0:
        raise ValueError("cache holds fewer than T positions")
    return T, H, D, Hkv, L, start_pos


def prefill_attention(q, k, v, window: int = 0, scale: float | None = None,
                      threads: int | None = None, plant: str | None = None) -> np.ndarray:
    """fp64 attention output [T][H][D] for q [T][H][D], k/v [Hkv][L][D].

    start_pos is L - T.  ``scale`` defaults to 1/sqrt(head_dim) evaluated in
    float32 (the value the configurations pass to the GPU call).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D, Hkv, L, start_pos = _shapes(q, k, v)
    if scale is None:
        scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    out = np.empty((T, H, D), dtype=np.float64)
    lib = _load()
    n = threads or default_threads()
    if plant is None:
        rc = lib.pfa_oracle_prefill_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), T, start_pos,
                                              H, Hkv, D, int(window), float(scale), n)
    else:
        rc = lib.pfa_oracle_prefill_attention_planted(_ptr(q), _ptr(k), _ptr(v), _ptr(out), T,
                                                      start_pos, H, Hkv, D, int(window),
                                                      float(scale), n, PLANTS[plant])
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out


def prefill_attention_rows(q, k, v, rows, window: int = 0, scale: float | None = None,
                           threads: int | None = None) -> np.ndarray:
    """fp64 attention of selected (t, h) rows only; returns [len(rows)][D]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D, Hkv, L, start_pos = _shapes(q, k, v)
    if scale is None:
        scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    rt = np.ascontiguousarray(rows[:, 0], dtype=np.int64)
    rh = np.ascontiguousarray(rows[:, 1], dtype=np.int32)
    out = np.empty((len(rows), D), dtype=np.float64)
    lib = _load()
    rc = lib.pfa_oracle_prefill_attention_rows(
        _ptr(q), _ptr(k), _ptr(v), T, start_pos, H, Hkv, D, int(window), float(scale),
        rt.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        rh.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(rows), _ptr(out),
        threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out


def prefill_attention_cache(q_buf, k_buf, v_buf, T: int, start_pos: int, H: int, Hkv: int,
                            D: int, window: int = 0, scale: float | None = None,
                            qkv_dim: int | None = None, max_seq_len: int | None = None,
                            ring: bool = False, out_init=None, threads: int | None = None,
                            plant: str | None = None) -> np.ndarray:
    """fp64 attention over caller-layout buffers (flat arrays).

    q_buf holds token t's head h at [t*qkv_dim + h*D, +D); k_buf/v_buf hold
    key j of kv head kh at [kh*max_seq_len*D + row(j)*D, +D) with row(j) = j,
    or j % max_seq_len for a circular cache (``ring``).  Returns a flat
    float64 array of T*qkv_dim elements: the head elements of each row are
    the attention output, the others are copied from ``out_init`` (NaN when
    it is None).
    """
    qkv_dim = H * D if qkv_dim is None else int(qkv_dim)
    max_seq_len = start_pos + T if max_seq_len is None else int(max_seq_len)
    q, k, v = _f64(q_buf).reshape(-1), _f64(k_buf).reshape(-1), _f64(v_buf).reshape(-1)
    if T > 0 and q.size < (T - 1) * qkv_dim + H * D:
        raise ValueError("q buffer too small for T rows of qkv_dim")
    if k.size < Hkv * max_seq_len * D or v.size != k.size:
        raise ValueError("k/v buffers too small for num_kv_heads * max_seq_len rows")
    if scale is None:
        scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    if out_init is None:
        out = np.full(T * qkv_dim, np.nan, dtype=np.float64)
    else:
        out = _f64(out_init).reshape(-1).copy()
        if out.size != T * qkv_dim:
            raise ValueError("out_init must hold T * qkv_dim elements")
    lib = _load()
    rc = lib.pfa_oracle_prefill_attention_cache(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), T, start_pos, H, Hkv, D, int(window),
        float(scale), qkv_dim, max_seq_len, 1 if ring else 0, threads or default_threads(),
        PLANTS[plant] if plant else 0)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out
