"""pfa_prefill_attention_host: host buffers in, host buffer out, through the C
ABI (directly and through prefill_attention on CPU tensors).  The result is
within the oracle's bar, the same on every run, and bit-identical to the
device entry wherever every group of kv heads runs the plain schedule; the
call orders itself after the work already on its stream."""
import ctypes

import pytest
import torch

import chunked_causal_gqa_gb300 as pkg
import oracle
from chunked_causal_gqa_gb300 import _binding
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

# (H, Hkv, D, T, start_pos, window, dtype).  The kv heads go to one group
# when the call moves less than 4 MiB, two below 128 MiB, else four (at most
# Hkv); each group has its own copies, kernel and (bf16) the workspace
# schedule pfa_prefill_attention_ws picks for its heads alone.
CASES = [
    (6, 2, 128, 150, 20, 0, "bf16"),       # 1 group, group size 3
    (4, 1, 128, 77, 9, 0, "bf16"),         # 1 group, one kv head
    (8, 2, 512, 200, 100, 0, "bf16"),      # 4.3 MB: 2 groups of 1 kv head, head_dim 512
    (8, 2, 128, 129, 0, 0, "f32"),         # 1 group, fp32 head_dim 128 (bf16x3 tensor-core kernel)
    (8, 4, 64, 70, 30, 20, "f32"),         # 1 group, fp32 head_dim 64 (CUDA cores)
    (32, 8, 128, 300, 3000, 0, "bf16"),    # 18 MB: 2 groups of 4 kv heads
    (10, 5, 128, 130, 3000, 64, "bf16"),   # 8 MB: 2 uneven groups (2 + 3), window
    (8, 2, 512, 100, 4000, 0, "bf16"),     # 17 MB: 2 groups, head_dim 512
    (8, 8, 128, 64, 70000, 0, "bf16"),     # 287 MB: 4 groups, pairs past 64 key tiles
    (5, 5, 128, 32, 110000, 0, "bf16"),    # 282 MB: 4 uneven groups (1 + 1 + 1 + 2)
    (32, 8, 128, 128, 20000, 0, "bf16"),   # 84 MB: 2 groups, each on the balanced schedule
    (32, 4, 512, 640, 4000, 0, "bf16"),    # 80 MB: 2 groups, each on the head_dim-512 tail split
]


def _groups(case):
    """(H, Hkv) of each group, as the library splits the kv heads."""
    H, Hkv, D, T, sp, w, dt = case
    es = 2 if dt == "bf16" else 4
    moved = 2 * T * H * D * es + 2 * Hkv * (sp + T) * D * es
    G = min(Hkv, 1 if moved < 4 << 20 else (2 if moved < 128 << 20 else 4))
    bounds = [g * Hkv // G for g in range(G + 1)]
    return [((b - a) * (H // Hkv), b - a) for a, b in zip(bounds, bounds[1:])]


def _inputs(case, pinned):
    H, Hkv, D, T, sp, w, dt = case
    q, k, v = W.make_random(T, sp, H, Hkv, D, dt, seed=sum(case[:6]), q_std=1.0, kv_std=0.5)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    return q, k, v


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "H%d_Hkv%d_D%d_T%d_sp%d_w%d_%s" % c)
def test_host_entry_matches_device_entry_and_oracle(case, pinned):
    H, Hkv, D, T, sp, w, dt = case
    q, k, v = _inputs(case, pinned)
    got = pkg.prefill_attention(q, k, v, window=w)
    assert got.device.type == "cpu" and got.is_pinned() == pinned
    assert pkg.last_device_error() == 0
    G.check(G.to_np(got), oracle.prefill_attention(q, k, v, window=w), dt, str(case))
    again = pkg.prefill_attention(q, k, v, window=w)
    assert G.digest(again) == G.digest(got)
    plain = all(pkg.schedule(T, sp, h, hkv, D, w, q.dtype)[0] == "plain"
                for h, hkv in _groups(case))
    if plain or dt != "bf16":
        on_device = G.run(q, k, v, window=w, workspace=None)
        assert G.digest(got) == G.digest(on_device.cpu())


def _buffer_bytes(lib, T, sp, H, Hkv, D, dt):
    n = ctypes.c_size_t(0)
    assert lib.pfa_host_buffer_bytes(T, sp, H, Hkv, D, 0, dt, ctypes.byref(n)) == 0
    return n.value


def test_host_entry_c_abi_orders_after_its_stream():
    """Two calls queued back to back on a side stream into one device buffer,
    behind work that scribbles over the buffer: once the stream is
    synchronised, each output equals the one a lone call gives (and the
    oracle's within the bar)."""
    lib = _binding.load()
    H, Hkv, D, T, sp = 16, 4, 128, 200, 3000      # 13 MB: 2 groups
    scale = 1.0 / D ** 0.5
    cases = [W.make_random(T, sp, H, Hkv, D, "bf16", seed=s, q_std=1.0, kv_std=0.5)
             for s in (71, 72)]
    cases = [tuple(x.pin_memory() for x in c) for c in cases]
    outs = [torch.empty((T, H, D), dtype=torch.bfloat16, pin_memory=True) for _ in cases]
    n = _buffer_bytes(lib, T, sp, H, Hkv, D, _binding.PFA_BF16)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        buf.fill_(0xFF)
    for (q, k, v), o in zip(cases, outs):
        rc = lib.pfa_prefill_attention_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                            T, sp, H, Hkv, D, 0, scale, _binding.PFA_BF16,
                                            buf.data_ptr(), n, s.cuda_stream)
        assert rc == 0
    s.synchronize()
    assert lib.pfa_last_device_error(s.cuda_stream) == 0
    for (q, k, v), o in zip(cases, outs):
        assert G.digest(o) == G.digest(pkg.prefill_attention(q, k, v, scale=scale))
        G.check(G.to_np(o), oracle.prefill_attention(q, k, v, scale=scale), "bf16")


def test_host_entry_rejects_bad_device_buffers():
    lib = _binding.load()
    H, Hkv, D, T, sp = 8, 2, 128, 64, 10
    q, k, v = _inputs((H, Hkv, D, T, sp, 0, "bf16"), True)
    o = torch.empty_like(q)
    n = _buffer_bytes(lib, T, sp, H, Hkv, D, _binding.PFA_BF16)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    host_buf = torch.empty(n, dtype=torch.uint8, pin_memory=True)

    def call(ptr, nbytes):
        return lib.pfa_prefill_attention_host(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                              o.data_ptr(), T, sp, H, Hkv, D, 0, 0.1,
                                              _binding.PFA_BF16, ptr, nbytes, None)

    assert call(buf.data_ptr(), n - 256) == -2            # too small
    assert call(buf.data_ptr() + 128, n) == -4            # not 256-byte aligned
    assert call(host_buf.data_ptr(), n) == -5             # not device memory
    torch.cuda.synchronize()
    assert call(buf.data_ptr(), n) == 0
    torch.cuda.synchronize()
    assert pkg.last_device_error() == 0


def test_host_entry_concurrent_callers():
    """Two threads, each with its own stream and device buffer, call the C
    entry back to back: every output equals the one a lone call gives."""
    import threading
    lib = _binding.load()
    H, Hkv, D, T, sp = 16, 4, 128, 150, 2000
    scale = 1.0 / D ** 0.5
    n = _buffer_bytes(lib, T, sp, H, Hkv, D, _binding.PFA_BF16)
    inputs = [tuple(x.pin_memory() for x in W.make_random(T, sp, H, Hkv, D, "bf16", seed=s,
                                                          q_std=1.0, kv_std=0.5))
              for s in (81, 82, 83, 84)]
    want = [G.digest(pkg.prefill_attention(q, k, v, scale=scale)) for q, k, v in inputs]
    errors = []

    def worker(idx):
        try:
            s = torch.cuda.Stream()
            buf = torch.empty(n, dtype=torch.uint8, device="cuda")
            outs = []
            for rep in range(6):
                q, k, v = inputs[(idx + rep) % len(inputs)]
                o = torch.empty((T, H, D), dtype=torch.bfloat16, pin_memory=True)
                rc = lib.pfa_prefill_attention_host(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                    o.data_ptr(), T, sp, H, Hkv, D, 0, scale,
                                                    _binding.PFA_BF16, buf.data_ptr(), n,
                                                    s.cuda_stream)
                if rc != 0:
                    errors.append((idx, rep, rc))
                    return
                outs.append(((idx + rep) % len(inputs), o))
            s.synchronize()
            for which, o in outs:
                if G.digest(o) != want[which]:
                    errors.append((idx, which, "mismatch"))
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append((idx, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert pkg.last_device_error() == 0


def test_host_entry_groups_take_the_head_dim_512_tail_split():
    """The case above exercises the tail split inside the host entry."""
    H, Hkv, D, T, sp, w = 32, 4, 512, 640, 4000, 0
    assert [pkg.schedule(T, sp, h, hkv, D, w)[0] for h, hkv in _groups((H, Hkv, D, T, sp, w, "bf16"))] \
        == ["tail", "tail"]
