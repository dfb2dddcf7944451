"""Closed forms of the operation, run through the CUDA path (C ABI).

The gnosis page "Prefill attention -> GPU: handoff" ("GPU design", step 3)
defines each output row as the softmax-weighted sum of the visible V rows.
Two inputs make that sum known without running any attention code:

* constant V (every element c): the weights sum to one, so every output is c;
* q = 0: every visible score is 0, the weights are uniform, and each output
  row is the plain mean of the V rows its token sees (keys max(0, pos-window+1)
  .. pos, or 0 .. pos without a window).

Bounds.  fp32 inputs: within 1e-4 (the page's parity bar).  bf16 inputs: the
kernels round each probability p to bf16 before the P V product and sum the
row's normaliser l from the unrounded p, so with constant V the result is
c * sum(bf16(p)) / sum(p), then rounded to bf16.  Each bf16 rounding moves a
value by at most 2^-8 of itself, so |out - c| <= (2^-8 + 2^-8 + 2^-16) |c|
< 2^-7 |c|.  With q = 0 every p is exactly 1 and only the fp32 sum of V and
the final bf16 rounding remain: |out - mean| <= 2^-8 |mean| + 2^-12 (the
second term a generous allowance for fp32 accumulation over <= 8192 rows of
magnitude < 4).
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

BF16_CONST_REL = 2.0 ** -7
BF16_MEAN_REL, BF16_MEAN_ABS = 2.0 ** -8, 2.0 ** -12

# (H, Hkv, D, T, start_pos, window, dtype): both bf16 kernels, both fp32
# kernels (three bf16 products on the tensor cores for head_dim 128, the CUDA
# cores otherwise), windows, a long plain launch and shapes that take the
# workspace schedules.
CASES = [
    (32, 8, 128, 300, 200, 0, "bf16"),
    (8, 2, 128, 200, 9000, 0, "bf16"),      # long instance (71 key tiles per pair)
    (8, 2, 128, 300, 500, 129, "bf16"),     # window crossing key tiles
    (8, 2, 128, 300, 20000, 0, "bf16"),     # workspace schedule
    (32, 8, 128, 1280, 2000, 0, "bf16"),    # tail split of the last pairs
    (8, 2, 512, 200, 100, 0, "bf16"),
    (8, 2, 512, 300, 700, 256, "bf16"),
    (8, 2, 128, 300, 200, 0, "f32"),        # three bf16 products
    (8, 2, 128, 200, 500, 65, "f32"),
    (8, 2, 64, 150, 40, 0, "f32"),          # CUDA-core kernel
    (4, 2, 512, 40, 30, 7, "f32"),
]


def _ids(c):
    return "H%d_Hkv%d_D%d_T%d_sp%d_w%d_%s" % c


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_constant_v_returns_the_constant(case):
    H, Hkv, D, T, sp, w, dt = case
    q, k, _ = W.make_random(T, sp, H, Hkv, D, dt, seed=sum(case[:6]) + 5, kv_std=1.0)
    c = -1.25                                     # exact in bf16 and fp32
    v = torch.full_like(k, c)
    got = G.to_np(G.run(q, k, v, window=w))
    assert np.all(np.isfinite(got))
    err = np.abs(got - c)
    if dt == "f32":
        assert err.max() <= G.F32_ATOL, f"max |out - c| = {err.max():.3e}"
    else:
        assert err.max() <= BF16_CONST_REL * abs(c), f"max |out - c| = {err.max():.3e}"
    G.report("constant V " + _ids(case), {"max_abs_err": float(err.max()),
                                          "exact_fraction": float(np.mean(err == 0))})
    # the oracle agrees with the closed form (a check of the comparison itself)
    rows = [(0, 0), (T - 1, H - 1), (T // 2, 1)]
    want = oracle.prefill_attention_rows(q, k, v, rows, window=w)
    assert np.abs(want - c).max() <= 1e-12


def _visible_means(v64: np.ndarray, T: int, sp: int, H: int, Hkv: int, w: int) -> np.ndarray:
    """out[t, h] = mean of V[h // (H/Hkv), lo(t) .. pos(t)] by prefix sums (fp64)."""
    g = H // Hkv
    csum = np.concatenate([np.zeros((Hkv, 1, v64.shape[2])), np.cumsum(v64, axis=1)], axis=1)
    out = np.empty((T, H, v64.shape[2]))
    for t in range(T):
        pos = sp + t
        lo = max(0, pos - w + 1) if w > 0 else 0
        m = (csum[:, pos + 1] - csum[:, lo]) / (pos + 1 - lo)   # [Hkv][D]
        out[t] = np.repeat(m, g, axis=0)
    return out


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_zero_queries_return_the_mean_of_the_visible_values(case):
    H, Hkv, D, T, sp, w, dt = case
    _, k, v = W.make_random(T, sp, H, Hkv, D, dt, seed=sum(case[:6]) + 9, kv_std=0.5)
    q = torch.zeros(T, H, D, dtype=k.dtype)
    got = G.to_np(G.run(q, k, v, window=w))
    want = _visible_means(v.double().numpy(), T, sp, H, Hkv, w)
    err = np.abs(got - want)
    if dt == "f32":
        assert err.max() <= G.F32_ATOL, f"max |out - mean| = {err.max():.3e}"
    else:
        bound = BF16_MEAN_REL * np.abs(want) + BF16_MEAN_ABS
        assert np.all(err <= bound), f"max |out - mean| = {err.max():.3e}"
    G.report("q=0 " + _ids(case), {"max_abs_err": float(err.max())})
    # the oracle reaches the same closed form
    rows = [(0, 0), (T - 1, H - 1), (T // 3, H // 2)]
    o = oracle.prefill_attention_rows(q, k, v, rows, window=w)
    assert np.abs(o - want[[t for t, _ in rows], [h for _, h in rows]]).max() <= 1e-12
