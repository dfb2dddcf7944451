"""The fp64 oracle against pins fixed by the pages and by mathematics."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


def _oracle(q, k, v, window, scale):
    return oracle.prefill_attention(q, k, v, window=window, scale=scale, threads=2)


def test_all_pins_hold():
    assert pins.pin_failures(_oracle) == []


@pytest.mark.parametrize("case", pins.load_golden(), ids=lambda c: c["name"])
def test_golden_worked_examples(case):
    got = _oracle(case["q"], case["k"], case["v"], case["window"], case["scale"])
    np.testing.assert_allclose(got, case["out"], rtol=0, atol=1e-13)


@pytest.mark.parametrize("case", pins.tiny_cases(), ids=lambda c: c["name"])
def test_brute_force_mpmath(case):
    got = _oracle(case["q"], case["k"], case["v"], case["window"], case["scale"])
    want = pins.brute_force_mp(case["q"], case["k"], case["v"], case["window"], case["scale"])
    assert np.max(np.abs(got - want)) <= 1e-12


# Plants in the cache-layout arithmetic (strided rows, circular cache) are
# inert for the contiguous entry; tests/test_oracle_cache_layout.py covers them.
LAYOUT_PLANTS = ("ring_offset", "qkv_stride")


@pytest.mark.parametrize("plant", sorted(set(oracle.PLANTS) - set(LAYOUT_PLANTS)))
def test_planted_mistake_is_caught(plant):
    """Each deliberate mistake planted in the oracle must break some pin."""
    def planted(q, k, v, window, scale):
        return oracle.prefill_attention(q, k, v, window=window, scale=scale, threads=1,
                                        plant=plant)
    assert pins.pin_failures(planted), f"no pin caught planted mistake {plant!r}"


def _rand(rng, T, sp, H, Hkv, D):
    L = sp + T
    return (rng.standard_normal((T, H, D)), rng.standard_normal((Hkv, L, D)),
            rng.standard_normal((Hkv, L, D)))


@pytest.mark.parametrize("window", [0, 3, 16])
def test_masked_keys_never_change_outputs(window):
    """Replacing K/V at masked positions (j > pos, or j <= pos - window) with
    other finite values leaves every output bit-identical."""
    rng = np.random.default_rng(5)
    T, sp, H, Hkv, D = 9, 20, 4, 2, 6
    q, k, v = _rand(rng, T, sp, H, Hkv, D)
    base = _oracle(q, k, v, window, 0.4)
    for t in range(T):
        pos = sp + t
        k2, v2 = k.copy(), v.copy()
        k2[:, pos + 1:] = rng.standard_normal(k2[:, pos + 1:].shape) * 50
        v2[:, pos + 1:] = rng.standard_normal(v2[:, pos + 1:].shape) * 50
        if window > 0 and pos - window + 1 > 0:
            k2[:, :pos - window + 1] = 123.0
            v2[:, :pos - window + 1] = -77.0
        got = _oracle(q, k2, v2, window, 0.4)
        assert np.array_equal(got[t], base[t])


def test_group_heads_with_equal_queries_agree_and_groups_differ():
    """Query heads of one GQA group read the same K/V: equal q rows give
    bit-identical outputs; a head of another group (different K/V) does not."""
    rng = np.random.default_rng(6)
    T, sp, H, Hkv, D = 5, 7, 8, 2, 4
    q, k, v = _rand(rng, T, sp, H, Hkv, D)
    q[:, 1] = q[:, 0]; q[:, 3] = q[:, 0]; q[:, 4] = q[:, 0]
    out = _oracle(q, k, v, 0, 0.5)
    assert np.array_equal(out[:, 0], out[:, 1])
    assert np.array_equal(out[:, 0], out[:, 3])
    assert not np.allclose(out[:, 0], out[:, 4])


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 13, 11, 8, 4, 8)
    a = oracle.prefill_attention(q, k, v, window=5, scale=0.3, threads=1)
    b = oracle.prefill_attention(q, k, v, window=5, scale=0.3, threads=7)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("window", [0, 6])
def test_multi_chunk_equals_one_shot(window):
    """A chunk prefilled at start_pos = T1 against the cache equals the same
    rows of one prefill of T1 + T2 tokens from position 0 (the page's
    multi-chunk-vs-one-forward parity test)."""
    rng = np.random.default_rng(8)
    T1, T2, H, Hkv, D = 7, 5, 4, 2, 4
    q, k, v = _rand(rng, T1 + T2, 0, H, Hkv, D)
    full = _oracle(q, k, v, window, 0.5)
    chunk = _oracle(q[T1:], k, v, window, 0.5)
    assert np.array_equal(chunk, full[T1:])


def test_scale_folds_into_keys():
    rng = np.random.default_rng(9)
    q, k, v = _rand(rng, 6, 4, 4, 2, 4)
    a = _oracle(q, k, v, 0, 0.25)
    b = _oracle(q, k * 0.25, v, 0, 1.0)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_rows_entry_matches_full_output():
    rng = np.random.default_rng(10)
    q, k, v = _rand(rng, 9, 6, 8, 2, 4)
    full = _oracle(q, k, v, 4, 0.5)
    rows = [(0, 0), (8, 7), (3, 5), (5, 2)]
    got = oracle.prefill_attention_rows(q, k, v, rows, window=4, scale=0.5, threads=3)
    for i, (t, h) in enumerate(rows):
        assert np.array_equal(got[i], full[t, h])


def test_bad_arguments_are_rejected():
    rng = np.random.default_rng(11)
    q, k, v = _rand(rng, 4, 0, 3, 2, 4)        # H % Hkv != 0
    with pytest.raises(ValueError):
        oracle.prefill_attention(q, k, v)
    q, k, v = _rand(rng, 4, 0, 4, 2, 4)
    with pytest.raises(ValueError):
        oracle.prefill_attention(q, k[:, :3], v[:, :3])   # cache shorter than T
