"""The allocation-free entry point, pfa_prefill_attention_noalloc.

It exists for callers that cannot allocate device memory around the call
(graph capture, foreign allocators, host integrations without a device
allocator): it runs the balanced schedule in the library's own static device
scratch instead of a caller workspace.  These tests call it through the C ABI
and compare it with the allocating entry point (pfa_prefill_attention_ws with
a torch-allocated workspace), twice in a row on the same shared scratch:
both entries run the same schedule, so the outputs must be bit-identical, and
both must be within the bf16 bar of the fp64 oracle.  A shape needing more
than the static scratch must be refused.
"""
import ctypes

import pytest
import torch

import chunked_causal_gqa_gb300 as pkg
import oracle
from chunked_causal_gqa_gb300 import _binding
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20   # PFA_NOALLOC_SCRATCH_BYTES in include/pfa.h
PFA_BF16 = 1


def _call_noalloc(lib, q, k, v, out, start_pos, window, scale):
    T, H, D = q.shape
    Hkv = k.shape[0]
    return lib.pfa_prefill_attention_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), T, start_pos, H, Hkv, D,
        window, float(scale), PFA_BF16, torch.cuda.current_stream().cuda_stream)


# Shapes that use the balanced schedule (short chunks deep into the cache).
CASES = [
    # (H, Hkv, D, T, start_pos, window)
    (32, 8, 128, 128, 30000, 0),
    (8, 2, 128, 300, 20000, 0),
    (8, 2, 128, 200, 8000, 2048),   # sliding window
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "H%d_Hkv%d_D%d_T%d_sp%d_w%d" % c)
def test_noalloc_matches_the_workspace_entry_on_two_calls_in_a_row(case):
    H, Hkv, D, T, sp, w = case
    lib = _binding.load()
    d = G.dev()
    q, k, v = (x.to(d) for x in W.make_random(T, sp, H, Hkv, D, "bf16", seed=61, kv_std=0.5))
    scale = float(torch.tensor(D ** -0.5, dtype=torch.float32))
    need = pkg.workspace_bytes(T, sp, H, Hkv, D, w)
    assert 0 < need <= SCRATCH_BYTES          # the shape runs in the static scratch
    ref = pkg.prefill_attention(q, k, v, window=w, scale=scale)   # caller workspace
    assert pkg.last_device_error() == 0
    want = oracle.prefill_attention(q.cpu(), k.cpu(), v.cpu(), window=w, scale=scale)
    G.check(G.to_np(ref), want, "bf16", "workspace entry vs oracle")
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        assert _call_noalloc(lib, q, k, v, out, sp, w, scale) == 0
        assert pkg.last_device_error() == 0
        assert torch.equal(out, ref), "noalloc and workspace entries differ in some bits"
        G.check(G.to_np(out), want, "bf16", "noalloc vs oracle")


def test_noalloc_refuses_a_shape_beyond_its_scratch():
    lib = _binding.load()
    d = G.dev()
    # 1k-token chunks at start_pos 120000: their balanced schedule needs a
    # little more than 32 MiB on a 152-SM GB300
    candidates = [(32, 4, 1024, 120000), (32, 8, 1024, 120000), (64, 8, 512, 120000)]
    for H, Hkv, T, sp in candidates:
        if pkg.workspace_bytes(T, sp, H, Hkv, 128, 0) > SCRATCH_BYTES:
            break
    else:
        pytest.fail("no candidate shape needs more than the static scratch on this device")
    L = sp + T
    q = torch.empty(T, H, 128, dtype=torch.bfloat16, device=d)   # refused before any launch
    k = torch.empty(Hkv, L, 128, dtype=torch.bfloat16, device=d)
    v = torch.empty_like(k)
    out = torch.empty_like(q)
    assert _call_noalloc(lib, q, k, v, out, sp, 0, 128 ** -0.5) == -10     # PFA_ERR_SCRATCH
    assert lib.pfa_status_string(-10).decode().startswith("PFA_ERR_SCRATCH")
