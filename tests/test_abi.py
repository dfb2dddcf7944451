"""The C-ABI library: builds, loads, exports every declared symbol, and
rejects bad arguments before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import chunked_causal_gqa_gb300 as pkg
from chunked_causal_gqa_gb300 import _binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pfa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _binding.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PFA_API\s+[\w\s\*]*?\b(pfa_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in _binding.STATUS.items():
        assert lib.pfa_status_string(code).decode().startswith(name)
    assert lib.pfa_status_string(12345)


def test_version(lib):
    assert pkg.version()[0] == 1


BF16, F32 = _binding.PFA_BF16, _binding.PFA_F32
A, B, C, O = 0x10000, 0x20000000, 0x40000000, 0x60000000   # aligned, disjoint fake pointers


def call(lib, q=A, k=B, v=C, o=O, T=16, sp=0, H=8, Hkv=2, D=128, w=0, scale=0.1, dt=BF16):
    return lib.pfa_prefill_attention(q, k, v, o, T, sp, H, Hkv, D, w, scale, dt, None)


def test_argument_validation_without_gpu(lib):
    assert call(lib, dt=7) == -3                       # dtype
    assert call(lib, T=-1) == -2                       # shape
    assert call(lib, sp=-3) == -2
    assert call(lib, H=6, Hkv=4) == -2                 # H % Hkv
    assert call(lib, H=0) == -2
    assert call(lib, D=96) == -2                       # bf16 head_dim
    assert call(lib, D=130, dt=F32) == -2              # fp32 head_dim not a multiple of 4
    assert call(lib, D=516, dt=F32) == -2
    assert call(lib, H=256, Hkv=1) == -2               # bf16 group > 128
    assert call(lib, scale=float("nan")) == -8
    assert call(lib, scale=float("inf")) == -8
    assert call(lib, T=0, q=None, k=None, v=None, o=None) == 0   # empty chunk: no-op
    assert call(lib, q=None) == -1
    assert call(lib, o=None) == -1
    assert call(lib, k=B + 8) == -4                    # alignment
    assert call(lib, o=A + 64) == -9                   # out overlaps q
    assert call(lib, o=B + 4096) == -9                 # out overlaps k_cache


def test_workspace_entry_points_validate_without_gpu(lib):
    n = ctypes.c_size_t(123)
    assert lib.pfa_workspace_bytes(16, 0, 6, 4, 128, 0, BF16, ctypes.byref(n)) == -2
    assert n.value == 0
    assert lib.pfa_workspace_bytes(16, 0, 8, 2, 128, 0, BF16, None) == -1
    assert lib.pfa_workspace_bytes(0, 0, 8, 2, 128, 0, BF16, ctypes.byref(n)) == 0
    assert lib.pfa_prefill_attention_ws(A, B, C, O, 16, 0, 8, 2, 128, 0, 0.1, BF16,
                                        0x70000000, 4096, None) in (-5,)   # no GPU here
    assert lib.pfa_prefill_attention_ws(A, B, C, O, 16, 0, 6, 4, 128, 0, 0.1, BF16,
                                        0x70000000, 4096, None) == -2


def host_call(lib, q=A, k=B, v=C, o=O, T=16, sp=0, H=8, Hkv=2, D=128, w=0, scale=0.1, dt=BF16,
              buf=0x7000000000, nbuf=1 << 30):
    return lib.pfa_prefill_attention_host(q, k, v, o, T, sp, H, Hkv, D, w, scale, dt, buf, nbuf,
                                          None)


def test_host_entry_validates_without_gpu(lib):
    import torch
    no_gpu = not torch.cuda.is_available()
    n = ctypes.c_size_t(7)
    assert lib.pfa_host_buffer_bytes(16, 0, 6, 4, 128, 0, BF16, ctypes.byref(n)) == -2
    assert lib.pfa_host_buffer_bytes(16, 0, 8, 2, 128, 0, BF16, None) == -1
    assert lib.pfa_host_buffer_bytes(0, 0, 8, 2, 128, 0, BF16, ctypes.byref(n)) == 0
    assert n.value == 0
    if no_gpu:   # the size depends on the device (its schedules)
        assert lib.pfa_host_buffer_bytes(16, 0, 8, 2, 128, 0, BF16, ctypes.byref(n)) == -5
    # checks that come before any CUDA call
    assert host_call(lib, dt=7) == -3
    assert host_call(lib, H=6, Hkv=4) == -2
    assert host_call(lib, scale=float("nan")) == -8
    assert host_call(lib, T=0, q=None, k=None, v=None, o=None, buf=None) == 0
    assert host_call(lib, q=None) == -1
    assert host_call(lib, buf=None) == -1
    assert host_call(lib, k=B + 8) == -4                 # host buffers: 16-byte aligned
    assert host_call(lib, buf=0x7000000000 + 16) == -4   # device buffer: 256-byte aligned
    assert host_call(lib, o=A + 64) == -9                # out overlaps q
    if no_gpu:
        assert host_call(lib) == -5                      # valid arguments: the device check


def test_valid_arguments_reach_the_device_check(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: covered by the gpu tests")
    assert call(lib) == -5
    assert call(lib, D=100, dt=F32) == -5


def test_python_binding_checks_tensors():
    import torch
    q = torch.zeros(4, 8, 128, dtype=torch.bfloat16)
    k = torch.zeros(2, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkg.prefill_attention(q, k, k.float())
    with pytest.raises(ValueError):
        pkg.prefill_attention(q, k[:, :3], k[:, :3])
    with pytest.raises(ValueError):
        pkg.prefill_attention(q[0], k, k)
    # CPU tensors (the host-buffer path): layout checks before any device use
    with pytest.raises(ValueError):
        pkg.prefill_attention(q, k, k, out=torch.zeros(4, 8, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        pkg.prefill_attention(q.transpose(0, 1).contiguous().transpose(0, 1), k, k)
    assert pkg.prefill_attention(q[:0], k[:, :0], k[:, :0]).shape == (0, 8, 128)   # T = 0
    pkg.release_host_buffers()   # nothing kept: a no-op


def cache_call(lib, q=A, k=B, v=C, o=O, T=16, sp=100, H=8, Hkv=2, D=128, w=64, dt=BF16,
               qkv_dim=None, cap=512, ring=1):
    qkv_dim = H * D if qkv_dim is None else qkv_dim
    return lib.pfa_prefill_attention_cache(q, k, v, o, T, sp, H, Hkv, D, w, 0.1, dt, qkv_dim,
                                           cap, ring, None, 0, None)


def test_cache_layout_validation_without_gpu(lib):
    assert cache_call(lib, ring=1, w=0) == -2              # ring needs a window
    assert cache_call(lib, sp=1000, w=600) == -2           # 600 + 15 rows > 512
    assert cache_call(lib, sp=1000, cap=300, w=100) == -2  # wrapped bf16 ring, 300 % 128
    assert cache_call(lib, ring=0, cap=100) == -2          # linear cache shorter than L
    assert cache_call(lib, qkv_dim=8 * 128 - 8) == -2      # rows shorter than the heads
    assert cache_call(lib, qkv_dim=8 * 128 + 4) == -4      # 2056-byte rows
    assert cache_call(lib, T=0, q=None, k=None, v=None, o=None) == 0


def test_graph_entry_validation_without_gpu(lib):
    def g(lens=0x80000, max_T=16, cap=512, ring=0, w=0, dt=BF16, D=128):
        return lib.pfa_prefill_attention_graph(A, B, C, O, lens, max_T, 8, 2, D, w, 0.1, dt,
                                               8 * D, cap, ring, None)
    assert g(lens=None) == -1
    assert g(lens=0x80004) == -4                           # lengths not 8-byte aligned
    assert g(max_T=-1) == -2
    assert g(max_T=600) == -2                              # max_T > max_seq_len
    assert g(ring=1, w=0) == -2
    assert g(max_T=0) == 0                                 # no-op


def test_c_program_uses_the_abi_without_a_gpu(lib, tmp_path):
    """include/pfa.h compiles as C and the library links into a plain C program."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(_binding.LIB_PATH)
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(here, "..", "include"),
                    os.path.join(here, "c_abi", "abi_check.c"), "-L", libdir, "-lpfa",
                    "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
