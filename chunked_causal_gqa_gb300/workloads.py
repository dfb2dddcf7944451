"""Seeded synthetic inputs for chunked causal GQA prefill attention.

This module holds the workload shapes and the seeded generators that both the
CUDA path's tests/benchmark and the CPU oracle consume.  It contains none of
the attention arithmetic: it only draws N(0, 1) numbers from a seeded CPU
``torch.Generator``, multiplies them by an exact power-of-two factor and rounds
them to the storage dtype (round-to-nearest-even for bf16).

Shapes follow the workloads the pages describe: a Mistral-7B layer
(32 query heads, 8 kv heads, head_dim 128) prefilled with a 1358-token prompt
(gnosis "Prefill attention -> GPU: handoff", section "Diagnosis"); steady-state
2048-token chunks deep into a long prompt (TensorSharp2 Gemma-4 prefill design,
section 2, a late chunk at start_pos ~60k, and its 64k/128k rows); and the
Gemma-style head_dim-512 layers with a sliding window (same page, section 2,
the head_dim-512 flash kernel, and section 4 R4 for the window layers).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    T: int
    start_pos: int
    window: int
    dtype: str                  # "f32" or "bf16"
    q_std: float
    kv_std: float
    seeds: tuple                # (q, k, v)
    description: str

    @property
    def L(self) -> int:
        return self.start_pos + self.T

    @property
    def scale(self) -> float:
        """1/sqrt(head_dim) evaluated in float32, as the configurations pass it."""
        return float(torch.tensor(1.0, dtype=torch.float32)
                     / torch.sqrt(torch.tensor(float(self.head_dim), dtype=torch.float32)))

    def visible_keys(self) -> int:
        """Sum over query tokens of the number of visible keys (per head)."""
        total = 0
        w = self.window
        sp = self.start_pos
        if w <= 0:
            # sum_{t=0}^{T-1} (sp + t + 1)
            return self.T * (sp + 1) + self.T * (self.T - 1) // 2
        for t in range(self.T):
            pos = sp + t
            total += min(pos + 1, w)
        return total

    def causal_flops(self) -> float:
        """2 flops per multiply-add, QK^T and PV: 4 * D * H * sum_t n_t."""
        return 4.0 * self.head_dim * self.num_heads * self.visible_keys()

    def algorithmic_bytes(self) -> float:
        """Q + O once, plus each kv head's visible K and V rows once."""
        es = 4 if self.dtype == "f32" else 2
        qo = 2 * self.T * self.num_heads * self.head_dim * es
        if self.window <= 0:
            keys = self.L
        else:
            keys = min(self.L, self.window + self.T - 1)
        kv = 2 * self.num_kv_heads * keys * self.head_dim * es
        return float(qo + kv)


WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", 8, 2, 128, 128, 0, 0, "f32", 1.0, 1.0, (1000, 1001, 1002),
        "tiny fp32 causal GQA layer: H=8, Hkv=2, D=128, T=128 at start_pos=0"),
    "mistral_1358": Workload(
        "mistral_1358", 32, 8, 128, 1358, 0, 0, "bf16", 0.5, 0.5, (2000, 2001, 2002),
        "Mistral-7B-shaped layer, 1358-token prompt, bf16: H=32, Hkv=8, D=128, T=1358 at start_pos=0"),
    "chunk_64k": Workload(
        "chunk_64k", 32, 8, 128, 2048, 61440, 0, "bf16", 1.0, 0.5, (3000, 3001, 3002),
        "2048-token chunk at start_pos=61440 (L=63488), bf16: H=32, Hkv=8, D=128"),
    "gemma_d512_window": Workload(
        "gemma_d512_window", 8, 2, 512, 2048, 6144, 1024, "bf16", 1.0, 1.0, (4000, 4001, 4002),
        "head_dim-512 sliding-window layer (window 1024), bf16: H=8, Hkv=2, T=2048 at start_pos=6144"),
    "gemma_d512_global": Workload(
        "gemma_d512_global", 8, 2, 512, 2048, 6144, 0, "bf16", 1.0, 1.0, (4000, 4001, 4002),
        "head_dim-512 global causal layer, bf16: H=8, Hkv=2, T=2048 at start_pos=6144"),
    "chunk_64k_t128": Workload(
        "chunk_64k_t128", 32, 8, 128, 128, 63360, 0, "bf16", 1.0, 0.5, (3100, 3101, 3102),
        "128-token chunk at start_pos=63360 (L=63488), bf16: H=32, Hkv=8, D=128 "
        "(fewer query-tile pairs than SMs)"),
    "chunk_128k": Workload(
        "chunk_128k", 32, 8, 128, 2048, 129024, 0, "bf16", 1.0, 0.5, (5000, 5001, 5002),
        "2048-token chunk at start_pos=129024 (L=131072), bf16: H=32, Hkv=8, D=128"),
    "f32_chunk_16k": Workload(
        "f32_chunk_16k", 32, 8, 128, 2048, 14336, 0, "f32", 1.0, 0.5, (6000, 6001, 6002),
        "fp32 2048-token chunk at start_pos=14336 (L=16384): H=32, Hkv=8, D=128 "
        "(the fp32 tensor-core path at a size where it is not launch-bound)"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def draw(shape, seed: int, std: float, dtype: str) -> torch.Tensor:
    """Seeded N(0, std^2) CPU tensor of `shape`, rounded to `dtype`.

    std must be a power of two so that the scaling is exact in float32.
    """
    m, e = math.frexp(std)
    if m != 0.5:
        raise ValueError("std must be a power of two")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch_dtype(dtype)).contiguous()


def make_inputs(w: Workload, T: int | None = None, start_pos: int | None = None):
    """(q [T][H][D], k [Hkv][L][D], v [Hkv][L][D]) as CPU tensors of w.dtype.

    T / start_pos override the workload's chunk (for reduced-size cases with
    the same value distribution).
    """
    T = w.T if T is None else T
    sp = w.start_pos if start_pos is None else start_pos
    L = sp + T
    q = draw((T, w.num_heads, w.head_dim), w.seeds[0], w.q_std, w.dtype)
    k = draw((w.num_kv_heads, L, w.head_dim), w.seeds[1], w.kv_std, w.dtype)
    v = draw((w.num_kv_heads, L, w.head_dim), w.seeds[2], w.kv_std, w.dtype)
    return q, k, v


def make_random(T, start_pos, H, Hkv, D, dtype="bf16", seed=0, q_std=1.0, kv_std=1.0):
    """Seeded inputs of an arbitrary shape (test cases)."""
    L = start_pos + T
    q = draw((T, H, D), seed * 3 + 11, q_std, dtype)
    k = draw((Hkv, L, D), seed * 3 + 12, kv_std, dtype)
    v = draw((Hkv, L, D), seed * 3 + 13, kv_std, dtype)
    return q, k, v
