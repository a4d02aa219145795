"""Head sharding of the forward pass across ranks (one process per GPU).

Every (batch row, value head) sequence of the gated delta rule is independent,
so N ranks split the value heads into N contiguous blocks and run the forward
pass on their block alone: no exchange is needed on the data path. A block of
value heads keeps whole groups of the grouped-query layout (value head hv reads
q/k head hv // (HV // H)), so each rank also owns a contiguous block of q/k
heads. This is the head sharding that the optimisation script's memory
analysis assumes ("heads=48 (local=12)").
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class HeadShard:
    rank: int
    world: int
    hv0: int   # first value head of this rank
    hv1: int   # one past the last value head
    h0: int    # first q/k head
    h1: int    # one past the last q/k head


def head_shard(rank: int, world: int, H: int, HV: int) -> HeadShard:
    """Contiguous block of value heads (and their q/k heads) owned by `rank`."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank / world size")
    if HV % H:
        raise ValueError("HV must be a multiple of H")
    group = HV // H
    if H % world:
        raise ValueError("the q/k heads must split evenly across ranks")
    per_h = H // world
    h0, h1 = rank * per_h, (rank + 1) * per_h
    return HeadShard(rank, world, h0 * group, h1 * group, h0, h1)


def shard_inputs(x: dict, s: HeadShard) -> dict:
    """Slice full [B,T,H,K] / [B,T,HV,...] / [B,HV,K,V] tensors to one rank's heads."""
    out = {}
    for name, t in x.items():
        if t is None:
            out[name] = None
        elif name in ("q", "k"):
            out[name] = t[:, :, s.h0:s.h1].contiguous()
        elif name == "s0":
            out[name] = t[:, s.hv0:s.hv1].contiguous()
        else:   # v, g, beta: value heads on axis 2
            out[name] = t[:, :, s.hv0:s.hv1].contiguous()
    return out


def step_time_across_ranks(local_ms: float, dist=None) -> float:
    """The step time of the whole job: the slowest rank's (max over ranks)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(local_ms)
    import torch
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
