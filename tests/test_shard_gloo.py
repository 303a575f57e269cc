"""Multi-rank decomposition on CPU with gloo, world size 2.

Each rank projects its batch slice (the oracle stands in for the device work,
so this needs no GPU); gathering the slices must reproduce the single-process
result exactly, and the reported time must be the slowest rank's.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from ff_input_projection_gb300.shard import batch_shard, max_over_ranks


def test_batch_shard_partitions():
    for n in range(0, 11):
        for world in range(1, 5):
            spans = [batch_shard(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        batch_shard(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import fpsynth
        import oracle
        from ff_input_projection_gb300.shard import shard_view
        w = fpsynth.Workload("shard_case", (3, 2, 16, 4, 4, 1), 2, 1, 16, 32, 2, 8,
                             fpsynth.ACT_GELU_ERF, 10000.0, True, "f32", 9)
        inp = fpsynth.make_inputs(w)
        x = torch.from_numpy(inp["x"])
        xs = shard_view(x, 0, rank, world).contiguous().numpy()
        local = oracle.forward(xs, inp["W"], inp["b"], channel_dim=2, n_batch_dims=1, C=w.C,
                               F=w.F, heads=w.heads, head_dim=w.head_dim, act=w.act,
                               rope_base=w.rope_base, dtype="f32", threads=1)
        gathered = [None] * world
        dist.all_gather_object(gathered, {k: v for k, v in local.items()})
        t = max_over_ranks(1.0 + rank)
        if rank == 0:
            full = oracle.forward_workload(w, inp, threads=1)
            ok = all(np.array_equal(np.concatenate([g[k] for g in gathered]), full[k])
                     for k in ("ff", "q", "k", "v"))
            result_q.put((ok, t))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reproduce_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok, t = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok
    assert t == 2.0
