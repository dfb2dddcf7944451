"""Helpers for the GPU parity tests (call the CUDA path through the C ABI and
compare with the fp64 oracle)."""
from __future__ import annotations

import hashlib
import json
import os

import numpy as np
import torch

import chunked_causal_gqa_gb300 as pkg

# bf16 bar: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| element-wise (allclose form);
# fp32 bar: max |gpu - oracle| <= 1e-4.
BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
F32_ATOL = 1e-4


def dev():
    return torch.device("cuda", 0)


def run(q, k, v, window=0, scale=None, out=None, workspace="auto"):
    d = dev()
    o = pkg.prefill_attention(q.to(d), k.to(d), v.to(d), window=window, scale=scale, out=out,
                              workspace=workspace)
    status = pkg.last_device_error()
    assert status == 0, f"device error status {status}"
    return o


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def strict_report(got: np.ndarray, want: np.ndarray) -> dict:
    """The bf16 bar read strictly: |err| <= 2e-2 and |err| <= 1e-2 |oracle| must
    each hold.  Reported beside the allclose form the tests assert; the
    relative part cannot hold where the oracle's value is near zero (an
    output that cancels), so its violations are counted, not asserted."""
    err = np.abs(got - want)
    ref = np.abs(want)
    rel_bad = err > BF16_RTOL * ref
    return {"elements": int(err.size), "max_abs_err": float(err.max()),
            "abs_violations": int(np.count_nonzero(err > BF16_ATOL)),
            "rel_violations": int(np.count_nonzero(rel_bad)),
            "rel_violations_where_abs_ref_ge_0.1":
                int(np.count_nonzero(rel_bad & (ref >= 0.1)))}


def report(what: str, rec: dict) -> None:
    """Append one JSON line to the file named by $PFA_TOL_REPORT, if set."""
    path = os.environ.get("PFA_TOL_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": what, **rec}) + "\n")


def check(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    assert got.shape == want.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    if dtype == "f32":
        assert err.max() <= F32_ATOL, f"{what}: max |err| {err.max():.3e} > {F32_ATOL}"
    else:
        bound = BF16_ATOL + BF16_RTOL * np.abs(want)
        bad = err > bound
        if bad.any():
            idx = np.argwhere(bad)[:5].tolist()
            raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance, "
                                 f"max |err| {err.max():.3e}, first at {idx}")
    return float(err.max())


def digest(t: torch.Tensor) -> str:
    return hashlib.sha256(t.detach().contiguous().cpu().view(torch.uint8).numpy()
                          .tobytes()).hexdigest()


def sample_rows(T: int, H: int, n_random: int, seed: int):
    rng = np.random.default_rng(seed)
    ts = {0, 1, 31, 32, 33, 63, 64, 127, 128, 129, T // 2, T - 2, T - 1}
    ts |= set(rng.integers(0, T, n_random).tolist())
    hs = {0, 1, 3, 4, H - 1}
    rows = []
    for t in sorted(x for x in ts if 0 <= x < T):
        for h in sorted(x for x in hs if 0 <= x < H):
            rows.append((t, h))
        rows.append((t, int(rng.integers(0, H))))
    return rows
