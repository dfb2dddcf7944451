"""Two ranks (gloo, CPU) each compute their kv-head shard of one layer with the
oracle; gathering the shards along the head axis reproduces the full output
bit for bit.  This covers the host logic of the multi-process path."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from chunked_causal_gqa_gb300 import sharding


def test_kv_head_ranges_partition_the_heads():
    for hkv in (1, 2, 3, 8, 13):
        for world in (1, 2, 3, 4, 8):
            spans = [sharding.kv_head_range(hkv, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == hkv
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result):
    import oracle
    from chunked_causal_gqa_gb300 import workloads as W
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v = W.make_random(20, 13, 8, 2, 16, "f32", seed=5)
    (qs, ks, vs), (h0, h1) = sharding.shard(q, k, v, world, rank)
    part = torch.from_numpy(oracle.prefill_attention(qs.contiguous(), ks.contiguous(),
                                                     vs.contiguous(), window=6, scale=0.25,
                                                     threads=1))
    parts = [None] * world
    dist.all_gather_object(parts, (h0, h1, part))
    if rank == 0:
        full = torch.cat([p for _, _, p in sorted(parts, key=lambda x: x[0])], dim=1)
        ref = oracle.prefill_attention(q, k, v, window=6, scale=0.25, threads=1)
        result.put(bool(np.array_equal(full.numpy(), ref)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_head_sharding_matches_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    assert q.get(timeout=5) is True
