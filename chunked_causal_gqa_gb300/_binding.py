"""ctypes binding of libpfa.so (the C ABI declared in include/pfa.h).

Argument marshalling only: every step of the attention runs in the library's
CUDA kernels.  There is no CPU fallback: if the library has not been built,
or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpfa.so")

PFA_F32 = 0
PFA_BF16 = 1

STATUS = {
    0: "PFA_OK", -1: "PFA_ERR_NULL", -2: "PFA_ERR_SHAPE", -3: "PFA_ERR_DTYPE",
    -4: "PFA_ERR_ALIGNMENT", -5: "PFA_ERR_DEVICE", -6: "PFA_ERR_LAUNCH",
    -7: "PFA_ERR_TIMEOUT", -8: "PFA_ERR_VALUE", -9: "PFA_ERR_ALIAS", -10: "PFA_ERR_SCRATCH",
    -11: "PFA_ERR_LENGTHS",
}
EXPORTS = ("pfa_prefill_attention", "pfa_prefill_attention_ws", "pfa_workspace_bytes",
           "pfa_prefill_attention_noalloc", "pfa_prefill_attention_cache",
           "pfa_prefill_attention_graph", "pfa_schedule",
           "pfa_prefill_attention_host", "pfa_host_buffer_bytes",
           "pfa_status_string",
           "pfa_last_device_error", "pfa_version", "pfa_debug_configure",
           "pfa_debug_check_schedule", "pfa_debug_check_schedule_d512")

_lock = threading.Lock()
_lib = None


class PfaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{what}: {self.name}" if what else self.name)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libpfa.so (raises if it is missing: build it with build.build())."""
    global _lib
    if _lib is not None and path is None:      # loaded: no lock on the call path
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(
                f"libpfa.so not found at {p}; build it with "
                "`python -c 'import chunked_causal_gqa_gb300.build as b; b.build()'`")
        lib = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.pfa_prefill_attention.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32, i32,
                                              ctypes.c_float, i32, vp]
        lib.pfa_prefill_attention.restype = i32
        sz = ctypes.c_size_t
        lib.pfa_prefill_attention_ws.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32, i32,
                                                 ctypes.c_float, i32, vp, sz, vp]
        lib.pfa_prefill_attention_ws.restype = i32
        lib.pfa_workspace_bytes.argtypes = [i64, i64, i32, i32, i32, i32, i32,
                                            ctypes.POINTER(sz)]
        lib.pfa_workspace_bytes.restype = i32
        lib.pfa_schedule.argtypes = [i64, i64, i32, i32, i32, i32, i32, ctypes.POINTER(i32),
                                     ctypes.POINTER(sz)]
        lib.pfa_schedule.restype = i32
        lib.pfa_prefill_attention_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                                      i32, ctypes.c_float, i32, vp]
        lib.pfa_prefill_attention_noalloc.restype = i32
        lib.pfa_prefill_attention_cache.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                                    i32, ctypes.c_float, i32, i64, i64, i32, vp,
                                                    sz, vp]
        lib.pfa_prefill_attention_cache.restype = i32
        lib.pfa_prefill_attention_graph.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32,
                                                    i32, ctypes.c_float, i32, i64, i64, i32, vp]
        lib.pfa_prefill_attention_graph.restype = i32
        lib.pfa_prefill_attention_host.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32,
                                                   i32, ctypes.c_float, i32, vp, sz, vp]
        lib.pfa_prefill_attention_host.restype = i32
        lib.pfa_host_buffer_bytes.argtypes = [i64, i64, i32, i32, i32, i32, i32,
                                              ctypes.POINTER(sz)]
        lib.pfa_host_buffer_bytes.restype = i32
        lib.pfa_status_string.argtypes = [i32]
        lib.pfa_status_string.restype = ctypes.c_char_p
        lib.pfa_last_device_error.argtypes = [vp]
        lib.pfa_last_device_error.restype = i32
        lib.pfa_version.argtypes = []
        lib.pfa_version.restype = i32
        lib.pfa_debug_configure.argtypes = [ctypes.c_double, i32]
        lib.pfa_debug_configure.restype = i32
        ip = ctypes.POINTER(i32)
        lib.pfa_debug_check_schedule.argtypes = [i64, i64, i32, i32, i32, i32, ip, ip, ip]
        lib.pfa_debug_check_schedule.restype = i32
        lib.pfa_debug_check_schedule_d512.argtypes = [i64, i64, i32, i32, i32, i32, ip, ip, ip]
        lib.pfa_debug_check_schedule_d512.restype = i32
        if path is None:
            _lib = lib
        return lib
