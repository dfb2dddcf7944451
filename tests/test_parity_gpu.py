"""The CUDA path (through the C ABI) against the fp64 oracle.

Every configuration compares every output element: the small cases against
an oracle run in the test, the full-size 64k/128k chunks and head_dim-512
layers against the whole oracle output, computed once per input recipe and
cached on disk.  Tolerances are the
ones stated for the two dtypes (fp32: max |err| <= 1e-4; bf16 inputs with fp32
accumulation: |err| <= 2e-2 + 1e-2 |oracle|).
"""
import numpy as np
import pytest
import torch

import oracle
from chunked_causal_gqa_gb300 import workloads as W
from tests import gpu_util as G
from tests import oracle_cache as OC

pytestmark = pytest.mark.gpu


# (H, Hkv, D, T, start_pos, window): tiles of 128 rows (group heads x 128/group
# tokens), key tiles of 128, ragged tails, every supported group-size regime.
BF16_CASES = [
    (32, 8, 128, 300, 200, 0),     # Mistral-like GQA 4, ragged T and L
    (8, 2, 128, 257, 0, 0),        # prompt from position 0, one token past a tile
    (8, 2, 128, 64, 1000, 0),      # short chunk deep in the cache
    (4, 4, 128, 130, 5, 0),        # group 1: 128 tokens per tile
    (16, 8, 128, 200, 33, 0),      # group 2
    (16, 2, 128, 100, 50, 0),      # group 8
    (6, 2, 128, 150, 20, 0),       # group 3: 126-row tiles
    (32, 1, 128, 40, 10, 0),       # group 32: 4 tokens per tile
    (128, 1, 128, 5, 3, 0),        # group 128: 1 token per tile
    (8, 2, 128, 300, 500, 100),    # window inside one key tile
    (8, 2, 128, 300, 500, 129),    # window band crossing key tiles
    (8, 2, 128, 200, 0, 1000),     # window longer than the prompt
    (8, 2, 128, 1, 0, 0),          # a single first token
    (8, 2, 128, 1, 777, 0),        # a single token deep in the cache
    # head_dim 512 (key tiles of 128; a cluster of two CTAs per pair of query
    # tiles and half of the output columns)
    (8, 2, 512, 200, 100, 0),      # 7 tiles per head: the last pair's second tile past T
    (8, 2, 512, 130, 0, 64),       # window of exactly one key tile
    (8, 2, 512, 150, 300, 1000),   # window longer than the visible prefix
    (4, 4, 512, 150, 10, 0),       # group 1: 128 tokens per tile
    (8, 1, 512, 40, 300, 100),     # group 8
    (6, 2, 512, 70, 5, 0),         # group 3: 126-row tiles
    (16, 1, 512, 50, 300, 0),      # group 16: 8 tokens per tile, 7 tiles
    (32, 1, 512, 33, 1000, 200),   # group 32: 4 tokens per tile, window
    (128, 1, 512, 5, 7, 0),        # group 128: 1 token per tile, odd count
    (8, 2, 512, 1, 50, 0),
]


@pytest.mark.parametrize("case", BF16_CASES, ids=lambda c: "H%d_Hkv%d_D%d_T%d_sp%d_w%d" % c)
def test_bf16_small_full_parity(case):
    H, Hkv, D, T, sp, w = case
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=sum(case), q_std=1.0, kv_std=0.5)
    got = G.to_np(G.run(q, k, v, window=w))
    want = oracle.prefill_attention(q, k, v, window=w)
    G.check(got, want, "bf16", str(case))


F32_CASES = [
    (8, 2, 64, 77, 30, 0),
    (4, 1, 100, 50, 10, 7),
    (8, 2, 512, 33, 20, 0),
    (6, 3, 36, 40, 0, 5),
    (2, 2, 128, 1, 100, 0),
    # head_dim 128: the tensor-core kernel (three bf16 products, key tiles of 128)
    (8, 2, 128, 300, 200, 0),      # GQA 4, ragged T and L
    (8, 2, 128, 129, 0, 0),        # one token past a tile, prompt from 0
    (4, 4, 128, 130, 5, 0),        # group 1: 128 tokens per tile
    (16, 2, 128, 100, 50, 0),      # group 8
    (6, 2, 128, 150, 20, 0),       # group 3: 126-row tiles
    (128, 1, 128, 5, 3, 0),        # group 128: 1 token per tile
    (8, 2, 128, 300, 500, 100),    # window inside one key tile
    (8, 2, 128, 300, 500, 65),     # window band crossing key tiles
    (8, 2, 128, 64, 3000, 0),      # short chunk deep in the cache
    (32, 8, 128, 200, 1000, 0),    # Mistral-like heads
    (256, 1, 128, 3, 5, 0),        # group 256: too large for a tile, the CUDA-core kernel
]


@pytest.mark.parametrize("case", F32_CASES, ids=lambda c: "H%d_Hkv%d_D%d_T%d_sp%d_w%d" % c)
def test_f32_small_full_parity(case):
    H, Hkv, D, T, sp, w = case
    q, k, v = W.make_random(T, sp, H, Hkv, D, "f32", seed=sum(case))
    got = G.to_np(G.run(q, k, v, window=w))
    want = oracle.prefill_attention(q, k, v, window=w)
    G.check(got, want, "f32", str(case))


# The head_dim-128 bf16 kernel has two instances: plain launches whose longest
# query-tile pair holds at most 64 key tiles of 128 keys (all the shapes
# above) take the short-launch one (Q_A loaded before Q_B, output staged in
# shared memory); longer ones take the other.  These shapes keep the long
# instance under the same ragged / odd-group / window cases, and pin the
# switch at exactly 64 and 65 key tiles (L = 8192 and 8193).
LONG_BF16_CASES = [
    (8, 2, 128, 64, 8128, 0),      # L = 8192: 64 key tiles, the short instance's limit
    (8, 2, 128, 64, 8129, 0),      # L = 8193: 65 key tiles, the long instance
    (6, 2, 128, 150, 9000, 0),     # group 3, ragged T
    (16, 2, 128, 100, 9000, 0),    # group 8
    (128, 1, 128, 5, 9000, 0),     # group 128: 1 token per tile
    (8, 2, 128, 257, 8500, 0),     # one token past a tile
    (8, 2, 128, 200, 9000, 8300),  # window wider than 64 key tiles
]


@pytest.mark.parametrize("workspace", [None, "auto"])
@pytest.mark.parametrize("case", LONG_BF16_CASES, ids=lambda c: "H%d_Hkv%d_D%d_T%d_sp%d_w%d" % c)
def test_bf16_long_instance_full_parity(case, workspace):
    H, Hkv, D, T, sp, w = case
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=sum(case), q_std=1.0, kv_std=0.5)
    got = G.to_np(G.run(q, k, v, window=w, workspace=workspace))
    want = oracle.prefill_attention(q, k, v, window=w)
    G.check(got, want, "bf16", str(case))


def test_tiny_f32_workload_full_parity():
    wl = W.WORKLOADS["tiny_f32"]
    q, k, v = W.make_inputs(wl)
    got = G.to_np(G.run(q, k, v, window=wl.window, scale=wl.scale))
    want = oracle.prefill_attention(q, k, v, window=wl.window, scale=wl.scale)
    G.check(got, want, "f32", wl.name)


def test_mistral_layer_full_parity():
    wl = W.WORKLOADS["mistral_1358"]
    q, k, v = W.make_inputs(wl)
    got = G.to_np(G.run(q, k, v, window=wl.window, scale=wl.scale))
    want = oracle.prefill_attention(q, k, v, window=wl.window, scale=wl.scale)
    G.check(got, want, "bf16", wl.name)


@pytest.mark.parametrize("workspace", ["auto", None])
@pytest.mark.parametrize("name", ["chunk_64k", "chunk_128k", "gemma_d512_global"])
def test_large_config_full_output_parity(name, workspace):
    """Every output element of the 64k and 128k chunks and of the head_dim-512
    global layer against the whole fp64 oracle output (cached on disk per
    input recipe), for the schedule the library picks and for the plain one.
    The stricter reading of the bf16 bar is reported beside the asserted
    allclose form."""
    import chunked_causal_gqa_gb300 as pkg
    wl = W.WORKLOADS[name]
    sched, nbytes = pkg.schedule(wl.T, wl.start_pos, wl.num_heads, wl.num_kv_heads,
                                 wl.head_dim, wl.window)
    if workspace == "auto" and wl.head_dim == 128:
        assert nbytes > 0 and sched == "tail"
    q, k, v = W.make_inputs(wl)
    want = OC.full_output(wl, (q, k, v))
    out = G.run(q, k, v, window=wl.window, scale=wl.scale, workspace=workspace)
    got = G.to_np(out)
    err = G.check(got, want, "bf16", name)
    G.report(f"{name} schedule={sched if workspace else 'plain'}",
             {"allclose_max_abs_err": err, **G.strict_report(got, want)})


def test_f32_long_chunk_full_parity_and_bits():
    """The fp32 tensor-core path at a size where it streams 16k keys per query tile:
    every output element against the whole oracle output, and bit-identical
    reruns."""
    wl = W.WORKLOADS["f32_chunk_16k"]
    q, k, v = W.make_inputs(wl)
    out = G.run(q, k, v, window=wl.window, scale=wl.scale)
    want = OC.full_output(wl, (q, k, v))
    err = G.check(G.to_np(out), want, "f32", wl.name)
    G.report(wl.name, {"max_abs_err": err})
    assert G.digest(G.run(q, k, v, window=wl.window, scale=wl.scale)) == G.digest(out)


def test_gemma_window_layer_full_parity():
    wl = W.WORKLOADS["gemma_d512_window"]
    q, k, v = W.make_inputs(wl)
    got = G.to_np(G.run(q, k, v, window=wl.window, scale=wl.scale))
    want = OC.full_output(wl, (q, k, v))
    err = G.check(got, want, "bf16", wl.name)
    G.report(wl.name, {"allclose_max_abs_err": err, **G.strict_report(got, want)})


@pytest.mark.parametrize("D", [128, 512])
def test_repeated_runs_are_bit_identical_small(D):
    q, k, v = (x.to(G.dev()) for x in W.make_random(333, 129, 8, 2, D, "bf16", seed=47))
    digests = {G.digest(G.run(q, k, v, window=100)) for _ in range(5)}
    assert len(digests) == 1


@pytest.mark.parametrize("name", ["mistral_1358", "chunk_64k"])
def test_repeated_runs_are_bit_identical(name):
    wl = W.WORKLOADS[name]
    q, k, v = (x.to(G.dev()) for x in W.make_inputs(wl))
    digests = {G.digest(G.run(q, k, v, scale=wl.scale)) for _ in range(5)}
    assert len(digests) == 1


@pytest.mark.parametrize("window", [0, 200])
def test_chunked_prefill_equals_one_shot(window):
    """Prefilling the second chunk against the cache gives the same rows as a
    single prefill of the whole prompt: bit for bit with the plain schedule
    (each row sees the same key tiles in the same order), and within rounding
    with the balanced one (whose split points depend on the shape)."""
    H, Hkv, D, T1, T2 = 32, 8, 128, 384, 300
    q, k, v = W.make_random(T1 + T2, 0, H, Hkv, D, "bf16", seed=41, kv_std=0.5)
    full = G.run(q, k, v, window=window, workspace=None)
    chunk = G.run(q[T1:].contiguous(), k, v, window=window, workspace=None)
    assert torch.equal(chunk, full[T1:])
    full_b = G.run(q, k, v, window=window)
    chunk_b = G.run(q[T1:].contiguous(), k, v, window=window)
    want = oracle.prefill_attention(q[T1:], k, v, window=window)
    G.check(G.to_np(chunk_b), want, "bf16", "balanced chunk")
    assert torch.allclose(chunk_b.float(), full_b[T1:].float(), atol=2e-2, rtol=1e-2)


# Shapes where a workspace schedule is chosen (the balanced table, or every
# pair split into equal key ranges): short chunks deep into the cache (fewer
# query-tile pairs than SMs), with and without a window.
SCHEDULE_CASES = [
    (32, 8, 128, 128, 30000, 0),
    (8, 2, 128, 300, 20000, 0),
    (8, 2, 128, 200, 8000, 2048),
    (4, 4, 128, 130, 12000, 0),
    (16, 2, 128, 64, 5000, 0),
    (8, 2, 128, 40, 3000, 0),
    (8, 2, 128, 700, 3000, 0),
    (32, 8, 128, 1280, 2000, 0),   # 160 pairs on 152 SMs: the tail split cuts the last 8
]


@pytest.mark.parametrize("case", SCHEDULE_CASES, ids=lambda c: "H%d_Hkv%d_D%d_T%d_sp%d_w%d" % c)
def test_plain_and_balanced_schedules_agree_with_oracle(case):
    import chunked_causal_gqa_gb300 as pkg
    H, Hkv, D, T, sp, w = case
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=sum(case) + 7, kv_std=0.5)
    want = oracle.prefill_attention(q, k, v, window=w)
    plain = G.run(q, k, v, window=w, workspace=None)
    G.check(G.to_np(plain), want, "bf16", "plain " + str(case))
    assert pkg.workspace_bytes(T, sp, H, Hkv, D, w) > 0     # the balanced path is taken
    bal = G.run(q, k, v, window=w)
    G.check(G.to_np(bal), want, "bf16", "balanced " + str(case))
    # an explicit workspace gives the same bits; one byte short falls back to plain
    need = pkg.workspace_bytes(T, sp, H, Hkv, D, w)
    ws = torch.full((need,), 255, dtype=torch.uint8, device=G.dev())
    assert torch.equal(G.run(q, k, v, window=w, workspace=ws), bal)
    small = torch.empty(need - 1, dtype=torch.uint8, device=G.dev())
    assert torch.equal(G.run(q, k, v, window=w, workspace=small), plain)


def test_balanced_schedule_is_bit_identical_across_runs():
    import chunked_causal_gqa_gb300 as pkg
    q, k, v = (x.to(G.dev()) for x in W.make_random(300, 20000, 8, 2, 128, "bf16", seed=63))
    assert pkg.workspace_bytes(300, 20000, 8, 2, 128, 0) > 0
    digests = {G.digest(G.run(q, k, v)) for _ in range(5)}
    assert len(digests) == 1


@pytest.mark.parametrize("window", [0, 150])
def test_masked_keys_never_change_outputs(window):
    H, Hkv, D, T, sp = 8, 2, 128, 256, 300
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=43)
    base = G.run(q, k, v, window=window)
    t_cut = 100
    k2, v2 = k.clone(), v.clone()
    k2[:, sp + t_cut + 1:] = 7.0          # keys after row t_cut's position
    v2[:, sp + t_cut + 1:] = -3.0
    got = G.run(q, k2, v2, window=window)
    assert torch.equal(got[:t_cut + 1], base[:t_cut + 1])
    if window > 0:
        # keys at or before pos - window for every row t >= t_lo
        t_lo = 200
        cut = sp + t_lo - window + 1
        k3, v3 = k.clone(), v.clone()
        k3[:, :cut] = 5.0
        v3[:, :cut] = 9.0
        got = G.run(q, k3, v3, window=window)
        assert torch.equal(got[t_lo:], base[t_lo:])


def test_group_heads_with_equal_queries_agree():
    H, Hkv, D, T, sp = 8, 2, 128, 100, 60
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=44)
    q[:, 1] = q[:, 0]
    q[:, 3] = q[:, 0]
    q[:, 4] = q[:, 0]      # first head of the other group
    out = G.run(q, k, v)
    assert torch.equal(out[:, 0], out[:, 1])
    assert torch.equal(out[:, 0], out[:, 3])
    assert not torch.equal(out[:, 0], out[:, 4])
    q, k, v = W.make_random(T, sp, H, Hkv, 512, "bf16", seed=48)
    q[:, 2] = q[:, 1]
    q[:, 5] = q[:, 1]
    out = G.run(q, k, v)
    assert torch.equal(out[:, 1], out[:, 2])
    assert not torch.equal(out[:, 1], out[:, 5])


@pytest.mark.parametrize("D", [128, 512])
def test_window_one_returns_own_value_row(D):
    H, Hkv, T, sp = 8, 2, 200, 90
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=45)
    out = G.run(q, k, v, window=1).cpu()
    want = torch.stack([v[h // 4, sp:sp + T] for h in range(H)], dim=1)
    assert torch.equal(out, want)


def test_out_argument_and_host_tensors():
    H, Hkv, D, T, sp = 8, 2, 128, 70, 10
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=46)
    d = G.dev()
    out = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device=d)
    import chunked_causal_gqa_gb300 as pkg
    r = pkg.prefill_attention(q.to(d), k.to(d), v.to(d), out=out)
    assert r.data_ptr() == out.data_ptr()
    host = pkg.prefill_attention(q, k, v)      # CPU tensors: copied in and out
    assert host.device.type == "cpu"
    assert torch.equal(host, out.cpu())


def test_errors_from_the_device_path():
    import chunked_causal_gqa_gb300 as pkg
    d = G.dev()
    q = torch.zeros(4, 8, 96, dtype=torch.bfloat16, device=d)
    k = torch.zeros(2, 4, 96, dtype=torch.bfloat16, device=d)
    with pytest.raises(pkg.PfaError) as e:
        pkg.prefill_attention(q, k, k)
    assert e.value.status == -2
    q = torch.zeros(4, 8, 128, dtype=torch.bfloat16, device=d)
    k = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device=d)
    empty = pkg.prefill_attention(q[:0], k[:, :0], k[:, :0])
    assert empty.shape == (0, 8, 128)


# Score profiles over the four 128-key tiles of a 500-key cache, in units of
# the shared component's score (~16 in log2 units): exercise every exponent-
# base path of the bf16 softmax -- a first tile far below 0, a first tile far
# above 0, a maximum that jumps by more than 2^8 in a later tile, and a plain
# profile.
SCORE_PROFILES = {
    "first_tile_far_below": (-6.0, 0.0, 1.5, 0.2),
    "first_tile_far_above": (2.0, 0.0, -1.0, 0.5),
    "late_jump": (0.1, 0.2, 1.5, 3.0),
    "flat": (0.0, 0.0, 0.0, 0.0),
}


@pytest.mark.parametrize("D", [128, 512])
@pytest.mark.parametrize("profile", sorted(SCORE_PROFILES))
def test_softmax_dynamic_range(profile, D):
    H, Hkv, T, sp = 8, 2, 200, 300
    L = sp + T
    g = torch.Generator().manual_seed(17)
    u = torch.randn(D, generator=g)
    q = (u + 0.1 * torch.randn(T, H, D, generator=g)).to(torch.bfloat16)
    beta = torch.empty(L)
    for tile, b in enumerate(SCORE_PROFILES[profile]):
        beta[tile * 128:(tile + 1) * 128] = b
    k = (beta[None, :, None] * u[None, None, :] + 0.3 * torch.randn(Hkv, L, D, generator=g))
    k = k.to(torch.bfloat16)
    v = torch.randn(Hkv, L, D, generator=g).to(torch.bfloat16)
    got = G.to_np(G.run(q, k, v))
    want = oracle.prefill_attention(q, k, v)
    G.check(got, want, "bf16", f"{profile} D{D}")


def test_schedule_query_names_the_schedule_each_workload_gets():
    import chunked_causal_gqa_gb300 as pkg
    expect = {"mistral_1358": "plain", "chunk_64k": "tail", "chunk_128k": "tail",
              "chunk_64k_t128": "tail", "gemma_d512_global": "plain", "tiny_f32": "plain"}
    for name, kind in expect.items():
        wl = W.WORKLOADS[name]
        got, nbytes = pkg.schedule(wl.T, wl.start_pos, wl.num_heads, wl.num_kv_heads,
                                   wl.head_dim, wl.window, W.torch_dtype(wl.dtype))
        assert got == kind, (name, got)
        assert (nbytes > 0) == (kind != "plain")
        assert nbytes == pkg.workspace_bytes(wl.T, wl.start_pos, wl.num_heads,
                                             wl.num_kv_heads, wl.head_dim, wl.window,
                                             W.torch_dtype(wl.dtype))


def test_tail_split_on_a_windowed_layer():
    """A long windowed chunk deep in a cache larger than L2 takes the tail split."""
    import chunked_causal_gqa_gb300 as pkg
    H, Hkv, D, T, sp, w = 32, 8, 128, 1280, 60000, 1024
    assert pkg.schedule(T, sp, H, Hkv, D, w)[0] == "tail"
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=77, q_std=1.0, kv_std=0.5)
    got = G.run(q, k, v, window=w)
    rows = G.sample_rows(T, H, 48, seed=77)
    want = oracle.prefill_attention_rows(q, k, v, rows, window=w)
    G.check(G.to_np(got)[[t for t, _ in rows], [h for _, h in rows]], want, "bf16", "tail+window")
    plain = G.run(q, k, v, window=w, workspace=None)
    G.check(G.to_np(plain)[[t for t, _ in rows], [h for _, h in rows]], want, "bf16",
            "plain+window")


# head_dim 512 with a last, partial wave of units: the tail split cuts each
# unit of that wave into equal key ranges (groups of 8 heads: 16 tokens per
# tile; 40 or 42 units -- pairs of query tiles of one kv head, four CTAs each
# -- on 38 per wave).
D512_TAIL_CASES = [
    (16, 2, 512, 640, 4000, 0),
    (16, 2, 512, 650, 4000, 0),      # ragged T
    (16, 2, 512, 640, 4000, 1000),   # sliding window
]


@pytest.mark.parametrize("case", D512_TAIL_CASES, ids=lambda c: "H%d_Hkv%d_D%d_T%d_sp%d_w%d" % c)
def test_d512_tail_split_agrees_with_oracle_and_plain(case):
    import chunked_causal_gqa_gb300 as pkg
    H, Hkv, D, T, sp, w = case
    sched, need = pkg.schedule(T, sp, H, Hkv, D, w)
    assert sched == "tail" and need > 0
    q, k, v = W.make_random(T, sp, H, Hkv, D, "bf16", seed=sum(case) + 3, kv_std=0.5)
    want = oracle.prefill_attention(q, k, v, window=w)
    plain = G.run(q, k, v, window=w, workspace=None)
    G.check(G.to_np(plain), want, "bf16", "plain " + str(case))
    tail = G.run(q, k, v, window=w)
    G.check(G.to_np(tail), want, "bf16", "tail " + str(case))
    # an explicit workspace gives the same bits; one byte short falls back to
    # plain; reruns are bit-identical
    ws = torch.full((need,), 255, dtype=torch.uint8, device=G.dev())
    assert torch.equal(G.run(q, k, v, window=w, workspace=ws), tail)
    small = torch.empty(need - 1, dtype=torch.uint8, device=G.dev())
    assert torch.equal(G.run(q, k, v, window=w, workspace=small), plain)
    assert G.digest(G.run(q, k, v, window=w)) == G.digest(tail)
