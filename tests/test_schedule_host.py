"""The head_dim-128 work assignment, replayed on the host (no GPU): for many
shapes and SM counts, every schedule the planner picks -- plain, tail split,
balanced table -- computes each key tile of each query-tile pair exactly once,
keeps key tiles inside the cache, gives partial results distinct workspace
slots, and merges exactly the split pairs' pieces in key order
(pfa_debug_check_schedule).  This stands in for a sanitizer, which the GPU
pool does not offer, on the index arithmetic of every launch shape."""
import ctypes
import itertools

import pytest

from chunked_causal_gqa_gb300 import _binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _binding.load()


def check(lib, T, sp, H, Hkv, window, sms):
    kind, ctas, failed = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    rc = lib.pfa_debug_check_schedule(T, sp, H, Hkv, window, sms, ctypes.byref(kind),
                                      ctypes.byref(ctas), ctypes.byref(failed))
    assert rc == 0, (T, sp, H, Hkv, window, sms, rc)
    return kind.value, ctas.value, failed.value


SHAPES = list(itertools.product(
    [1, 31, 33, 128, 300, 1358, 2048],          # T
    [0, 5, 129, 3000, 20000, 61440],            # start_pos
    [(32, 8), (8, 2), (4, 4), (16, 2), (6, 2), (128, 1)],  # (H, Hkv)
    [0, 1, 64, 1024],                           # window
))


@pytest.mark.parametrize("sms", [152, 148, 132, 17])
def test_every_schedule_keeps_its_invariants(lib, sms):
    kinds = set()
    for T, sp, (H, Hkv), w in SHAPES:
        kind, ctas, failed = check(lib, T, sp, H, Hkv, w, sms)
        assert failed == 0, f"check {failed} failed for T={T} sp={sp} H={H}/{Hkv} w={w} sms={sms}"
        assert ctas > 0
        kinds.add(kind)
    assert kinds == {0, 1, 2}, kinds   # plain, balanced and tail split all exercised


def test_workloads_get_the_expected_schedules(lib):
    # (T, start_pos, H, Hkv, window) -> schedule on a 152-SM GB300
    assert check(lib, 1358, 0, 32, 8, 0, 152)[:2] == (0, 176)      # Mistral layer: plain
    assert check(lib, 2048, 61440, 32, 8, 0, 152)[0] == 2          # 64k chunk: tail split
    assert check(lib, 2048, 129024, 32, 8, 0, 152)[0] == 2         # 128k chunk: tail split
    assert check(lib, 128, 63360, 32, 8, 0, 152)[:2] == (2, 144)   # short deep chunk: every pair split
    assert check(lib, 1358, 0, 8, 2, 0, 152)[0] == 1               # few uneven pairs: balanced
    # every pair split, one wave: pairs x parts CTAs, at most one per SM
    assert check(lib, 64, 1000, 8, 2, 0, 152)[:2] == (2, 18)       # 2 pairs x 9 ranges
    kind, ctas, failed = check(lib, 128, 63360, 32, 8, 0, 100)
    assert kind == 2 and ctas <= 100 and ctas % 16 == 0 and failed == 0


def test_arguments_are_checked(lib):
    kind = ctypes.c_int()
    assert lib.pfa_debug_check_schedule(16, 0, 8, 2, 0, 152, None, None, None) == -1
    assert lib.pfa_debug_check_schedule(16, 0, 6, 4, 0, 152, ctypes.byref(kind),
                                        ctypes.byref(kind), ctypes.byref(kind)) == -2
    assert lib.pfa_debug_check_schedule(16, 0, 8, 2, 0, 0, ctypes.byref(kind),
                                        ctypes.byref(kind), ctypes.byref(kind)) == -2


# ---- head_dim 512: pairs of CTAs (clusters) per pair of query tiles and output half

def check512(lib, T, sp, H, Hkv, window, sms):
    kind, ctas, failed = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_int(-1)
    rc = lib.pfa_debug_check_schedule_d512(T, sp, H, Hkv, window, sms, ctypes.byref(kind),
                                           ctypes.byref(ctas), ctypes.byref(failed))
    assert rc == 0, (T, sp, H, Hkv, window, sms, rc)
    return kind.value, ctas.value, failed.value


SHAPES512 = list(itertools.product(
    [1, 33, 40, 130, 640, 650, 2048],           # T (odd and even tile counts)
    [0, 5, 129, 4000, 6144, 20000],             # start_pos
    [(8, 2), (16, 2), (4, 4), (6, 2), (8, 1), (32, 4)],  # (H, Hkv): groups 4, 8, 1, 3, 8, 8
    [0, 1, 64, 1024],                           # window
))


@pytest.mark.parametrize("sms", [152, 148, 132, 17])
def test_every_head_dim_512_schedule_keeps_its_invariants(lib, sms):
    kinds = set()
    for T, sp, (H, Hkv), w in SHAPES512:
        kind, ctas, failed = check512(lib, T, sp, H, Hkv, w, sms)
        assert failed == 0, f"check {failed} failed for T={T} sp={sp} H={H}/{Hkv} w={w} sms={sms}"
        assert ctas > 0 and ctas % 4 == 0
        kinds.add(kind)
    assert kinds == {0, 2}, kinds   # plain and tail split both exercised


def test_head_dim_512_workloads_get_the_expected_schedules(lib):
    # Gemma-style layers (2048 tokens of 8/2 heads at 6144): plain, 2 x 2 x 32 x 2 CTAs
    assert check512(lib, 2048, 6144, 8, 2, 0, 152) == (0, 256, 0)
    assert check512(lib, 2048, 6144, 8, 2, 1024, 152) == (0, 256, 0)
    # 640 tokens of 16/2 heads at 4000: 40 units on 38 per wave -> tail split
    kind, ctas, failed = check512(lib, 640, 4000, 16, 2, 0, 152)
    assert kind == 2 and failed == 0 and ctas > 4 * 40
    # odd number of query tiles (7 per head): the last pair's second tile is past T
    assert check512(lib, 200, 100, 8, 2, 0, 152) == (0, 32, 0)


def test_head_dim_512_check_arguments(lib):
    kind = ctypes.c_int()
    assert lib.pfa_debug_check_schedule_d512(16, 0, 8, 2, 0, 152, None, None, None) == -1
    assert lib.pfa_debug_check_schedule_d512(16, 0, 6, 4, 0, 152, ctypes.byref(kind),
                                             ctypes.byref(kind), ctypes.byref(kind)) == -2
