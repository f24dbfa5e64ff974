"""Host-side helpers for running the head on several GPUs, one process each.

The path shards over rows (tokens are independent): rank r takes a
contiguous slice of the rows and the whole tied table W.  nll, lse and dh
stay local.  Only two reductions cross ranks:
  * the bits-per-byte sums (sum nll fp64, sum bytes, row count: 24 bytes),
    gathered and added in rank order so the result does not depend on
    arrival order;
  * dW (the data-parallel gradient of the tied table), a sum all-reduce.
These run through torch.distributed (NCCL on GPUs, gloo on CPU).
"""
from __future__ import annotations

import torch


def row_shard(N: int, rank: int, world: int) -> tuple:
    """[start, stop) of rank's contiguous row slice; sizes differ by <= 1."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank / world")
    return (N * rank) // world, (N * (rank + 1)) // world


def combine_bpb(parts) -> tuple:
    """Sum per-rank (sum_nll, sum_bytes, n) triples in the given (rank) order."""
    sn, sb, n = 0.0, 0, 0
    for a, b, c in parts:
        sn += float(a)
        sb += int(b)
        n += int(c)
    return sn, sb, n


def allreduce_bpb(local: tuple, group=None) -> tuple:
    """All ranks receive the rank-ordered combination of every rank's sums."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(local[0]), float(local[1]), float(local[2])], dtype=torch.float64, device=dev)
    out = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(out, t, group=group)
    parts = [(float(o[0]), int(round(float(o[1]))), int(round(float(o[2])))) for o in out]
    return combine_bpb(parts)


def allgather_bpb_acc(acc: torch.Tensor, group=None) -> torch.Tensor:
    """Device-side exchange of the 24-byte bpb accumulators (no host sync):
    returns a [world, 3] float64 tensor whose row r holds rank r's
    accumulator bytes (sum_nll, then the two int64 counts bit-cast); combine
    it with :func:`combine_bpb_acc` in rank order when the values are needed."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    out = torch.empty((world, 3), dtype=torch.float64, device=acc.device)
    dist.all_gather(list(out.unbind(0)), acc.reshape(3).contiguous(), group=group)
    return out


def combine_bpb_acc(gathered: torch.Tensor) -> tuple:
    """(sum_nll, sum_bytes, n) from allgather_bpb_acc's [world, 3] tensor,
    added in rank order."""
    g = gathered.detach().cpu().contiguous()
    ints = g.view(torch.int64)
    return combine_bpb([(float(g[r, 0]), int(ints[r, 1]), int(ints[r, 2])) for r in range(g.shape[0])])


def any_rank(flag: bool, group=None) -> bool:
    """True on every rank if `flag` is true on any rank.  Loops whose steps
    hold collectives (the benchmark's warm-up runs until a time has passed)
    decide with it, so that every rank runs the same number of steps."""
    import torch.distributed as dist

    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([1 if flag else 0], dtype=torch.int32, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return bool(t.item())


def allreduce_dW(dW: torch.Tensor, group=None) -> torch.Tensor:
    """Sum the tied-table gradient over ranks in place."""
    import torch.distributed as dist

    dist.all_reduce(dW, op=dist.ReduceOp.SUM, group=group)
    return dW
