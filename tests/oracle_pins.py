"""Pins for the fp64 oracle that do not come from the oracle itself.

Shared by the oracle tests (which require every pin to hold) and the
planted-control tests (which require each planted mistake to break at least
one pin).  Every pin is fixed by the pages' definition or by mathematics:

* hand-derived worked examples in tests/golden/log_weight_cases.txt;
* an independent brute-force formulation in 40-digit mpmath arithmetic
  (full score matrix, explicit boolean mask, masked softmax) on tiny inputs;
* closed forms: window 1 returns V at the row's own position; the first row
  of a prompt returns V[0]; constant V rows return the constant; q = 0 gives
  the mean of the visible V rows; one overwhelmingly large score selects its
  V row (which also needs the max shift to avoid overflow).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import mpmath
import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "log_weight_cases.txt")


def _value(tok: str) -> float:
    if tok.startswith("ln(") and tok.endswith(")"):
        return math.log(float(Fraction(tok[3:-1])))
    return float(Fraction(tok))


def load_golden():
    cases, cur, key = [], None, None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "case":
                cur = {"name": parts[1]}
            elif parts[0] == "end":
                cases.append(cur)
                cur = None
            elif parts[0] in ("H", "Hkv", "D", "T", "start_pos", "window"):
                cur[parts[0]] = int(parts[1])
            elif parts[0] == "scale":
                cur["scale"] = float(Fraction(parts[1]))
            else:
                cur[parts[0]] = [_value(t) for t in parts[1:]]
    out = []
    for c in cases:
        T, H, D, Hkv = c["T"], c["H"], c["D"], c["Hkv"]
        L = c["start_pos"] + T
        out.append(dict(
            name=c["name"], window=c["window"], scale=c["scale"],
            q=np.array(c["q"], dtype=np.float64).reshape(T, H, D),
            k=np.array(c["k"], dtype=np.float64).reshape(Hkv, L, D),
            v=np.array(c["v"], dtype=np.float64).reshape(Hkv, L, D),
            out=np.array(c["out"], dtype=np.float64).reshape(T, H, D)))
    return out


def brute_force_mp(q, k, v, window, scale, dps=40):
    """Independent formulation: per query head, the full T x L score matrix,
    an explicit boolean visibility mask, and a masked softmax, in mpmath."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    T, H, D = q.shape
    Hkv, L, _ = k.shape
    sp = L - T
    group = H // Hkv
    with mpmath.workdps(dps):
        out = np.zeros((T, H, D), dtype=np.float64)
        for h in range(H):
            kv = h // group
            Km = [[mpmath.mpf(float(x)) for x in k[kv, j]] for j in range(L)]
            Vm = [[mpmath.mpf(float(x)) for x in v[kv, j]] for j in range(L)]
            for t in range(T):
                qrow = [mpmath.mpf(float(x)) for x in q[t, h]]
                pos = sp + t
                mask = [(j <= pos) and (window <= 0 or j > pos - window) for j in range(L)]
                scores = [mpmath.mpf(scale) * mpmath.fsum(a * b for a, b in zip(qrow, Km[j]))
                          for j in range(L)]
                vis = [scores[j] for j in range(L) if mask[j]]
                mx = max(vis)
                wts = [mpmath.exp(scores[j] - mx) if mask[j] else mpmath.mpf(0) for j in range(L)]
                Z = mpmath.fsum(wts)
                for d in range(D):
                    out[t, h, d] = float(mpmath.fsum(wts[j] * Vm[j][d] for j in range(L)) / Z)
    return out


def tiny_cases():
    """Seeded tiny inputs spanning head counts, windows and chunk offsets."""
    rng = np.random.default_rng(12345)
    specs = [
        # H, Hkv, D, T, start_pos, window
        (1, 1, 1, 4, 0, 0),
        (2, 1, 4, 5, 3, 0),
        (4, 2, 8, 6, 5, 0),
        (4, 2, 4, 6, 5, 3),
        (8, 2, 4, 3, 4, 2),
        (8, 8, 1, 5, 2, 7),
        (4, 1, 8, 6, 0, 1),
        (8, 4, 4, 4, 5, 3),
    ]
    cases = []
    for (H, Hkv, D, T, sp, w) in specs:
        L = sp + T
        q = rng.standard_normal((T, H, D))
        k = rng.standard_normal((Hkv, L, D))
        v = rng.standard_normal((Hkv, L, D))
        cases.append(dict(name=f"H{H}_Hkv{Hkv}_D{D}_T{T}_sp{sp}_w{w}", q=q, k=k, v=v,
                          window=w, scale=1.0 / math.sqrt(D)))
    return cases


def pin_failures(fn):
    """Run every pin against fn(q, k, v, window, scale) -> out[T][H][D].

    Returns the names of the pins that fail (empty list = all hold)."""
    bad = []

    def check(name, got, want, tol):
        got = np.asarray(got, dtype=np.float64)
        if got.shape != want.shape or not np.all(np.isfinite(got)):
            bad.append(name)
            return
        if np.max(np.abs(got - want)) > tol:
            bad.append(name)

    for c in load_golden():
        check("golden:" + c["name"], fn(c["q"], c["k"], c["v"], c["window"], c["scale"]),
              c["out"], 1e-13)

    for c in tiny_cases():
        check("brute:" + c["name"], fn(c["q"], c["k"], c["v"], c["window"], c["scale"]),
              brute_force_mp(c["q"], c["k"], c["v"], c["window"], c["scale"]), 1e-12)

    rng = np.random.default_rng(777)
    # window 1: out[t, h] = V[h / group, pos] exactly
    H, Hkv, D, T, sp = 6, 3, 5, 7, 4
    q = rng.standard_normal((T, H, D)); k = rng.standard_normal((Hkv, sp + T, D))
    v = rng.standard_normal((Hkv, sp + T, D))
    want = np.stack([np.stack([v[h // (H // Hkv), sp + t] for h in range(H)]) for t in range(T)])
    check("closed:window1", fn(q, k, v, 1, 0.3), want, 0.0)

    # first row of a prompt (t = 0 at start_pos = 0) sees only key 0
    T = 5
    q = rng.standard_normal((T, H, D)); k = rng.standard_normal((Hkv, T, D))
    v = rng.standard_normal((Hkv, T, D))
    got = np.asarray(fn(q, k, v, 0, 0.7))
    want0 = np.stack([v[h // (H // Hkv), 0] for h in range(H)])
    if not np.array_equal(got[0], want0):
        bad.append("closed:first_row_v0")

    # constant V rows: output is the constant
    T, sp = 6, 9
    q = rng.standard_normal((T, H, D)) * 3; k = rng.standard_normal((Hkv, sp + T, D))
    c = rng.standard_normal((Hkv, 1, D))
    v = np.broadcast_to(c, (Hkv, sp + T, D)).copy()
    want = np.stack([np.stack([c[h // (H // Hkv), 0] for h in range(H)]) for t in range(T)])
    check("closed:constant_v", fn(q, k, v, 0, 0.5), want, 1e-14)
    check("closed:constant_v_window", fn(q, k, v, 4, 0.5), want, 1e-14)

    # q = 0: uniform weights, out = mean of the visible V rows
    q = np.zeros((T, H, D)); v = rng.standard_normal((Hkv, sp + T, D))
    for w in (0, 4):
        want = np.zeros((T, H, D))
        for t in range(T):
            pos = sp + t
            lo = max(0, pos - w + 1) if w > 0 else 0
            for h in range(H):
                want[t, h] = v[h // (H // Hkv), lo:pos + 1].mean(axis=0)
        check(f"closed:zero_q_mean_w{w}", fn(q, k, v, w, 0.5), want, 1e-13)

    # one overwhelming score (about 1000 above the rest): out = V of that key.
    # Without the max shift exp(1000) overflows.
    H, Hkv, D, T, sp = 4, 2, 3, 3, 5
    L = sp + T
    q = np.zeros((T, H, D)); q[:, :, 0] = 1.0
    k = rng.standard_normal((Hkv, L, D)) * 0.01
    v = rng.standard_normal((Hkv, L, D))
    hot = 2
    k[:, hot, 0] = 1000.0
    want = np.zeros((T, H, D))
    for t in range(T):
        for h in range(H):
            want[t, h] = v[h // (H // Hkv), hot]
    check("closed:dominant_key", fn(q, k, v, 0, 1.0), want, 1e-12)
    return bad
