"""pfa_prefill_attention_graph: the chunk's {T, start_pos} are read on the
device, so one CUDA graph captured around the call replays for a whole
chunked prefill (the replay requirement of the TensorSharp2 Gemma-4 prefill
design, section 4 R5: same pointers and shapes, contents refreshed in place).

Each replay's output rows are compared with the fp64 oracle's one-shot
attention over the whole prompt; rows past the run-time T must stay as they
were.
"""
import numpy as np
import pytest
import torch

import chunked_causal_gqa_gb300 as pkg
import oracle
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

SENTINEL = 3.0


def _chunks(total, max_T):
    sizes = [max_T, 100, 1, max_T, 37, 200, max_T]
    out, sp, i = [], 0, 0
    while sp < total:
        T = min(sizes[i % len(sizes)], total - sp)
        out.append((sp, T))
        sp += T
        i += 1
    return out


def _prefill(D, ring, capture_mode, dtype="bf16"):
    H, Hkv, max_T = 8, 2, 256
    if ring:
        window, cap, total = 512, 1024, 2600       # ring wraps twice; cap >= window + max_T - 1
    else:
        window, cap, total = 0, 2048, 1700
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q_all, k_all, v_all = W.make_random(total, 0, H, Hkv, D, dtype, seed=D + 7 * ring,
                                        q_std=1.0, kv_std=0.5)
    want = oracle.prefill_attention(q_all, k_all, v_all, window=window)
    d = G.dev()
    qbuf = torch.zeros(max_T, H, D, dtype=tdt, device=d)
    kc = torch.zeros(Hkv, cap, D, dtype=tdt, device=d)    # never-written rows are finite
    vc = torch.zeros_like(kc)
    out = torch.full((max_T, H, D), SENTINEL, dtype=tdt, device=d)
    lens = torch.tensor([1, 0], dtype=torch.int64, device=d)
    qd, kd, vd = q_all.to(d), k_all.to(d), v_all.to(d)

    def call():
        pkg.prefill_attention_graph(qbuf, kc, vc, out, lens, window=window, ring=ring)

    call()                                  # per-device set-up happens outside the capture
    torch.cuda.synchronize()
    assert pkg.last_device_error() == 0
    graph = None
    if capture_mode is not None:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode=capture_mode):
            call()
    for sp, T in _chunks(total, max_T):
        j = torch.arange(sp, sp + T, device=d)
        rows = j % cap if ring else j
        kc[:, rows] = kd[:, j]
        vc[:, rows] = vd[:, j]
        qbuf[:T] = qd[sp:sp + T]
        lens.copy_(torch.tensor([T, sp], dtype=torch.int64))
        out.fill_(SENTINEL)
        if graph is not None:
            graph.replay()
        else:
            call()
        assert pkg.last_device_error() == 0
        got = G.to_np(out)
        G.check(got[:T], want[sp:sp + T], dtype, f"chunk at {sp} (T={T})")
        assert np.all(got[T:] == SENTINEL), "rows past the run-time T were written"


@pytest.mark.parametrize("D", [128, 512])
@pytest.mark.parametrize("ring", [False, True])
def test_graph_replay_chunked_prefill(D, ring):
    _prefill(D, ring, "global")


def test_graph_replay_relaxed_capture():
    _prefill(128, False, "relaxed")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("ring", [False, True])
def test_graph_entry_fp32_without_capture(D, ring):
    # head_dim 64: the CUDA-core kernel; 128: the paired tensor-core kernel
    _prefill(D, ring, None, dtype="f32")


def test_graph_lengths_are_checked_on_the_device():
    d = G.dev()
    H, Hkv, D, max_T, cap = 8, 2, 128, 64, 512
    q = torch.randn(max_T, H, D, device=d).to(torch.bfloat16)
    kc = torch.zeros(Hkv, cap, D, dtype=torch.bfloat16, device=d)
    out = torch.full((max_T, H, D), SENTINEL, dtype=torch.bfloat16, device=d)
    for bad in ([max_T + 1, 0], [10, cap - 5], [-1, 0], [5, -2]):
        lens = torch.tensor(bad, dtype=torch.int64, device=d)
        pkg.prefill_attention_graph(q, kc, kc.clone(), out, lens)   # enqueues; the kernel checks
        assert pkg.last_device_error() == -11, bad                  # PFA_ERR_LENGTHS
        assert torch.all(out.float() == SENTINEL)
    lens = torch.tensor([0, 100], dtype=torch.int64, device=d)      # empty chunk
    pkg.prefill_attention_graph(q, kc, kc.clone(), out, lens)
    assert pkg.last_device_error() == 0
    assert torch.all(out.float() == SENTINEL)
    assert pkg.last_device_error() == 0                              # the word was cleared
