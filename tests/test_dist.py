"""Multi-rank host logic on CPU (gloo, world size 2).

Each rank takes its block of value heads, computes it (the float64 oracle
stands in for the GPU kernels here: what is tested is the sharding and the
combination of results and timings), and the blocks gathered on rank 0 must
equal the unsharded run exactly. The job's step time is the max over ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from chunkwise_gated_delta_gdr_gb300 import inputs as gin
from chunkwise_gated_delta_gdr_gb300 import shard


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = gin.shrink(gin.WORKLOADS["kda_gqa_t8192"], B=1, T=40, H=4, HV=8, K=8, V=6)
        x = gin.make_inputs(w)
        s = shard.head_shard(rank, world, w.H, w.HV)
        xs = shard.shard_inputs(x, s)
        o, S = oracle.recurrent(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], xs["s0"],
                                scale=w.scale)
        parts_o = [torch.zeros(1, w.T, w.HV // world, w.V, dtype=torch.float64) for _ in range(world)]
        parts_S = [torch.zeros(1, w.HV // world, w.K, w.V, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(parts_o, torch.from_numpy(np.ascontiguousarray(o)))
        dist.all_gather(parts_S, torch.from_numpy(np.ascontiguousarray(S)))
        t = shard.step_time_across_ranks(1.0 + rank, dist)
        if rank == 0:
            o_full, S_full = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["s0"],
                                              scale=w.scale)
            ok = (np.array_equal(torch.cat(parts_o, 2).numpy(), o_full)
                  and np.array_equal(torch.cat(parts_S, 1).numpy(), S_full))
            q.put((ok, t))
    finally:
        dist.destroy_process_group()


def test_head_sharding_two_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs)
    ok, t = q.get(timeout=10)
    assert ok, "gathered head shards differ from the unsharded run"
    assert t == 2.0   # slowest rank


def test_head_shard_blocks():
    s0 = shard.head_shard(0, 4, 16, 32)
    s3 = shard.head_shard(3, 4, 16, 32)
    assert (s0.h0, s0.h1, s0.hv0, s0.hv1) == (0, 4, 0, 8)
    assert (s3.h0, s3.h1, s3.hv0, s3.hv1) == (12, 16, 24, 32)
    with pytest.raises(ValueError):
        shard.head_shard(0, 3, 16, 32)
    with pytest.raises(ValueError):
        shard.head_shard(2, 2, 4, 4)
