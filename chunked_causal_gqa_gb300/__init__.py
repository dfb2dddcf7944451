"""GB300-native chunked causal GQA prefill attention.

A chunk of T query tokens at absolute positions start_pos .. start_pos+T-1
attends to the L = start_pos + T keys of a KV cache: query head h reads kv
head h / (num_heads / num_kv_heads), scores are scaled, key j is masked unless
j <= start_pos + t (and, with a sliding window, j > start_pos + t - window),
and a row softmax weights the sum of V (gnosis "Prefill attention -> GPU:
handoff", section "GPU design").

The computation runs in libpfa.so, a C-ABI library of hand-written sm_103a
kernels (include/pfa.h).  This package is its thin Python binding: it checks
tensors, passes pointers and the current CUDA stream, and copies host tensors
to and from the device when it is handed CPU tensors.
"""
from __future__ import annotations

import functools
import math
import threading

import torch

from . import _binding
from ._binding import PFA_BF16, PFA_F32, PfaError

__all__ = ["prefill_attention", "prefill_attention_cache", "prefill_attention_graph",
           "workspace_bytes", "schedule", "release_host_buffers",
           "last_device_error", "status_string", "version", "debug_configure", "PfaError",
           "PFA_F32", "PFA_BF16"]

_DTYPES = {torch.float32: PFA_F32, torch.bfloat16: PFA_BF16}


@functools.lru_cache(maxsize=None)
def _default_scale(head_dim: int) -> float:
    """1/sqrt(head_dim) rounded to float32 (the configurations' scale)."""
    return float(torch.tensor(1.0 / math.sqrt(head_dim), dtype=torch.float32))


def _stream_handle(device: torch.device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def workspace_bytes(T: int, start_pos: int, num_heads: int, num_kv_heads: int, head_dim: int,
                    window: int = 0, dtype: torch.dtype = torch.bfloat16) -> int:
    """Workspace bytes the balanced schedule needs on the current device (0: unused)."""
    import ctypes
    lib = _binding.load()
    n = ctypes.c_size_t(0)
    rc = lib.pfa_workspace_bytes(int(T), int(start_pos), int(num_heads), int(num_kv_heads),
                                 int(head_dim), int(window), _DTYPES[dtype], ctypes.byref(n))
    if rc != 0:
        raise PfaError(rc, "pfa_workspace_bytes")
    return int(n.value)


SCHEDULES = {0: "plain", 1: "balanced", 2: "tail"}


def schedule(T: int, start_pos: int, num_heads: int, num_kv_heads: int, head_dim: int,
             window: int = 0, dtype: torch.dtype = torch.bfloat16) -> tuple:
    """(schedule name, workspace bytes) the library uses for a shape with a workspace."""
    import ctypes
    lib = _binding.load()
    kind, n = ctypes.c_int(0), ctypes.c_size_t(0)
    rc = lib.pfa_schedule(int(T), int(start_pos), int(num_heads), int(num_kv_heads),
                          int(head_dim), int(window), _DTYPES[dtype], ctypes.byref(kind),
                          ctypes.byref(n))
    if rc != 0:
        raise PfaError(rc, "pfa_schedule")
    return SCHEDULES[kind.value], int(n.value)


def prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      out: torch.Tensor | None = None, *, start_pos: int | None = None,
                      window: int = 0, scale: float | None = None, stream=None,
                      workspace="auto") -> torch.Tensor:
    """Chunked causal GQA prefill attention through the C ABI.

    q: [T, num_heads, head_dim]; k_cache, v_cache: [num_kv_heads, L, head_dim]
    with L = start_pos + T (start_pos defaults to L - T); all contiguous, of
    one dtype (float32 or bfloat16).  window <= 0 means global causal.  scale
    defaults to 1/sqrt(head_dim) rounded to float32.

    workspace: "auto" (default) allocates the balanced schedule's workspace
    from torch's caching allocator when the shape uses one
    (pfa_prefill_attention_ws); a uint8 CUDA tensor supplies it; None runs
    the plain schedule (pfa_prefill_attention, no workspace).

    CUDA tensors: the call is enqueued on `stream` (default: the current
    stream) and returns without synchronising.  CPU tensors (pinned for full
    copy speed): pfa_prefill_attention_host copies them to the current CUDA
    device into a device buffer the binding keeps for later calls
    (release_host_buffers() frees it), overlapping the copies with the
    kernels by groups of kv heads, copies the result back into `out` (a new
    CPU tensor, pinned if q is, when out is None) and synchronises `stream`
    before returning; `workspace` is not used there.
    """
    if q.dim() != 3 or k_cache.dim() != 3 or v_cache.dim() != 3:
        raise ValueError("q must be [T, H, D]; k_cache and v_cache [Hkv, L, D]")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if q.dtype not in _DTYPES or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("q, k_cache and v_cache must all be float32 or all bfloat16")
    T, H, D = q.shape
    Hkv, L, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("head_dim of q and the cache differ")
    if start_pos is None:
        start_pos = L - T
    if start_pos < 0 or start_pos + T != L:
        raise ValueError(f"cache length {L} must equal start_pos + T = {start_pos + T}")
    if scale is None:
        scale = _default_scale(D)

    if k_cache.device != q.device or v_cache.device != q.device:
        raise ValueError("q, k_cache and v_cache must be on one device")
    if q.device.type == "cpu":
        return _prefill_host(q, k_cache, v_cache, out, T, start_pos, H, Hkv, D, window, scale,
                             stream)
    dev = q.device
    qd, kd, vd = q, k_cache, v_cache
    od = out if out is not None else torch.empty_like(q)
    if od.shape != q.shape or od.dtype != q.dtype or od.device != q.device:
        raise ValueError("out must match q in shape, dtype and device")
    for name, t in (("q", qd), ("k_cache", kd), ("v_cache", vd), ("out", od)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")

    lib = _binding.load()
    with torch.cuda.device(dev):
        st = _stream_handle(dev, stream)
        ws_ptr, ws_bytes = None, 0
        if isinstance(workspace, str):
            if workspace != "auto":
                raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
            need = workspace_bytes(T, start_pos, H, Hkv, D, window, q.dtype) if T > 0 else 0
            if need > 0:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
            else:
                workspace = None
        if workspace is not None:
            if workspace.device != dev or workspace.dtype != torch.uint8:
                raise ValueError("workspace must be a uint8 tensor on the output's device")
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
        rc = lib.pfa_prefill_attention_ws(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                          od.data_ptr(), int(T), int(start_pos), int(H), int(Hkv),
                                          int(D), int(window), float(scale), _DTYPES[q.dtype],
                                          ws_ptr, ws_bytes, st)
        if workspace is not None and stream is not None:
            # the caching allocator must not hand the workspace out again
            # before the work on `stream` is done
            workspace.record_stream(stream)
    if rc != 0:
        raise PfaError(rc, "pfa_prefill_attention")
    return od


# Device buffers of the host path, one per device, kept for reuse by later
# calls (grown when a call needs more); the lock keeps two threads from using
# one buffer at the same time.  release_host_buffers() returns them.
_host_lock = threading.Lock()
_host_bufs: dict = {}


def release_host_buffers() -> None:
    """Free the device buffers kept by prefill_attention on CPU tensors."""
    with _host_lock:
        _host_bufs.clear()


def _prefill_host(q, k_cache, v_cache, out, T, start_pos, H, Hkv, D, window, scale, stream):
    """prefill_attention on CPU tensors through pfa_prefill_attention_host."""
    import ctypes
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    elif out.shape != q.shape or out.dtype != q.dtype or out.device.type != "cpu":
        raise ValueError("out must match q in shape and dtype and be a CPU tensor")
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if T == 0:
        return out
    lib = _binding.load()
    dev = torch.cuda.current_device()
    dt = _DTYPES[q.dtype]
    cuda_stream = stream if stream is not None else torch.cuda.current_stream(dev)
    args = (q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(), int(T),
            int(start_pos), int(H), int(Hkv), int(D), int(window), float(scale), dt)
    with _host_lock:
        buf = _host_bufs.get(dev)
        rc = -2
        if buf is not None:   # the kept buffer; PFA_ERR_SHAPE if it is too small
            rc = lib.pfa_prefill_attention_host(*args, buf.data_ptr(), buf.numel(),
                                                int(cuda_stream.cuda_stream))
        if rc == -2:
            n = ctypes.c_size_t(0)
            rc = lib.pfa_host_buffer_bytes(int(T), int(start_pos), int(H), int(Hkv), int(D),
                                           int(window), dt, ctypes.byref(n))
            if rc != 0:
                raise PfaError(rc, "pfa_host_buffer_bytes")
            if buf is None or buf.numel() < n.value:
                _host_bufs.pop(dev, None)
                buf = torch.empty(int(n.value), dtype=torch.uint8,
                                  device=torch.device("cuda", dev))
                _host_bufs[dev] = buf
            rc = lib.pfa_prefill_attention_host(*args, buf.data_ptr(), buf.numel(),
                                                int(cuda_stream.cuda_stream))
        if rc != 0:
            raise PfaError(rc, "pfa_prefill_attention_host")
        # out is read by the caller on return, and buf is free for the next call
        cuda_stream.synchronize()
    return out


def prefill_attention_cache(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            out: torch.Tensor | None = None, *, start_pos: int, window: int = 0,
                            scale: float | None = None, ring: bool = False, stream=None,
                            workspace="auto") -> torch.Tensor:
    """Prefill attention on the caller's buffer layout (pfa_prefill_attention_cache).

    q: [T, H, D] CUDA tensor whose heads and elements are dense (strides
    (qkv_dim, D, 1), e.g. a column slice of a [T, qkv_dim] projection
    buffer); out: None (allocated with q's strides) or a tensor with q's
    shape and strides, of which only the head elements are written.
    k_cache, v_cache: the whole cache allocation, contiguous
    [Hkv, max_seq_len, D]; key j of the sequence is in row j, or in row
    j % max_seq_len when ``ring`` (a circular sliding-window cache; then
    window > 0 and max_seq_len >= min(L, window + T - 1)).  start_pos is
    required.  Other arguments: as for prefill_attention.
    """
    if q.dim() != 3 or k_cache.dim() != 3 or v_cache.dim() != 3:
        raise ValueError("q must be [T, H, D]; k_cache and v_cache [Hkv, max_seq_len, D]")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if q.dtype not in _DTYPES or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("q, k_cache and v_cache must all be float32 or all bfloat16")
    if q.device.type != "cuda" or k_cache.device != q.device or v_cache.device != q.device:
        raise ValueError("q, k_cache and v_cache must be CUDA tensors on one device")
    T, H, D = q.shape
    Hkv, max_seq_len, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("head_dim of q and the cache differ")
    if q.stride(2) != 1 or (H > 1 and q.stride(1) != D):
        raise ValueError("q's heads and elements must be dense (strides (qkv_dim, D, 1))")
    qkv_dim = q.stride(0) if T > 1 else H * D
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("k_cache and v_cache must be contiguous allocations")
    if out is None:
        out = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
    if (out.shape != q.shape or out.dtype != q.dtype or out.device != q.device
            or (T > 1 and out.stride() != q.stride())):
        raise ValueError("out must match q in shape, strides, dtype and device")
    if scale is None:
        scale = _default_scale(D)
    dev = q.device
    lib = _binding.load()
    with torch.cuda.device(dev):
        st = _stream_handle(dev, stream)
        ws_ptr, ws_bytes = None, 0
        if isinstance(workspace, str):
            if workspace != "auto":
                raise ValueError("workspace must be 'auto', None or a uint8 CUDA tensor")
            need = workspace_bytes(T, start_pos, H, Hkv, D, window, q.dtype) if T > 0 else 0
            workspace = torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None
        if workspace is not None:
            if workspace.device != dev or workspace.dtype != torch.uint8:
                raise ValueError("workspace must be a uint8 tensor on the output's device")
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
        rc = lib.pfa_prefill_attention_cache(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(), int(T),
            int(start_pos), int(H), int(Hkv), int(D), int(window), float(scale),
            _DTYPES[q.dtype], int(qkv_dim), int(max_seq_len), 1 if ring else 0, ws_ptr,
            ws_bytes, st)
        if workspace is not None and stream is not None:
            workspace.record_stream(stream)
    if rc != 0:
        raise PfaError(rc, "pfa_prefill_attention_cache")
    return out


def prefill_attention_graph(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            out: torch.Tensor, lengths: torch.Tensor, *, window: int = 0,
                            scale: float | None = None, ring: bool = False,
                            stream=None) -> torch.Tensor:
    """Prefill attention whose {T, start_pos} are read on the device (pfa_prefill_attention_graph).

    q, out: [max_T, H, D] CUDA tensors with dense heads (strides (qkv_dim, D, 1));
    k_cache, v_cache: contiguous [Hkv, max_seq_len, D]; lengths: a CUDA int64
    tensor of two elements {T, start_pos}, read when the kernel runs -- so a
    CUDA graph captured around this call replays for any chunk that fits.
    Rows of out past the run-time T are not written.
    """
    if q.dim() != 3 or k_cache.dim() != 3 or v_cache.dim() != 3:
        raise ValueError("q must be [max_T, H, D]; k_cache and v_cache [Hkv, max_seq_len, D]")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if q.dtype not in _DTYPES or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("q, k_cache and v_cache must all be float32 or all bfloat16")
    devs = {t.device for t in (q, k_cache, v_cache, out, lengths)}
    if len(devs) != 1 or q.device.type != "cuda":
        raise ValueError("all tensors must be CUDA tensors on one device")
    if lengths.dtype != torch.int64 or lengths.numel() != 2 or not lengths.is_contiguous():
        raise ValueError("lengths must be a contiguous int64 tensor {T, start_pos}")
    max_T, H, D = q.shape
    Hkv, max_seq_len, Dk = k_cache.shape
    if Dk != D:
        raise ValueError("head_dim of q and the cache differ")
    if q.stride(2) != 1 or (H > 1 and q.stride(1) != D):
        raise ValueError("q's heads and elements must be dense (strides (qkv_dim, D, 1))")
    qkv_dim = q.stride(0) if max_T > 1 else H * D
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("k_cache and v_cache must be contiguous allocations")
    if (out.shape != q.shape or out.dtype != q.dtype
            or (max_T > 1 and out.stride() != q.stride())):
        raise ValueError("out must match q in shape, strides and dtype")
    if scale is None:
        scale = _default_scale(D)
    dev = q.device
    lib = _binding.load()
    with torch.cuda.device(dev):
        rc = lib.pfa_prefill_attention_graph(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
            lengths.data_ptr(), int(max_T), int(H), int(Hkv), int(D), int(window), float(scale),
            _DTYPES[q.dtype], int(qkv_dim), int(max_seq_len), 1 if ring else 0,
            _stream_handle(dev, stream))
    if rc != 0:
        raise PfaError(rc, "pfa_prefill_attention_graph")
    return out


def last_device_error(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    lib = _binding.load()
    with torch.cuda.device(dev):
        return lib.pfa_last_device_error(_stream_handle(dev, stream))


def status_string(status: int) -> str:
    return _binding.load().pfa_status_string(int(status)).decode()


def version() -> tuple:
    v = _binding.load().pfa_version()
    return (v >> 16, v & 0xFFFF)


def debug_configure(wait_limit_ms: float = 0.0, force_timeout: bool = False) -> None:
    """Device-side wait limit and the forced-timeout test hook (see pfa.h)."""
    _binding.load().pfa_debug_configure(float(wait_limit_ms), 1 if force_timeout else 0)
