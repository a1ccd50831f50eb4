"""Independent replicas, one engine per GPU (the only multi-GPU mode).

The batched step is one weight stream shared by all of its rows ("20.3 服务、
批处理与流式", 20.3.2: a step costs (W + B*A)/beta), so splitting one batch over
GPUs would read W on every GPU; instead every rank runs its own engine, KV
pool and scheduler on its own share of the requests ("RWKV-Runner Albatross"
article, section on multiple GPUs: one worker per device).  Nothing on the
data path crosses ranks; the only collectives are the host-side timing and
bookkeeping reductions below (gloo on CPU in tests, NCCL in bench.py).
"""
from __future__ import annotations


def route(request_ids, rank: int, world: int) -> list:
    """This rank's requests: round-robin by arrival order (request i goes to
    rank i mod world), so every request has exactly one owner."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    return [r for i, r in enumerate(request_ids) if i % world == rank]


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's value (step time): every rank calls this."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist=None, device=None) -> float:
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_throughput(units_local: float, seconds_local: float, dist=None, device=None) -> float:
    """Whole-job throughput: the units every rank processed divided by the
    slowest rank's time (weak scaling: each rank owns a fixed share)."""
    total = sum_over_ranks(units_local, dist, device)
    slowest = max_over_ranks(seconds_local, dist, device)
    return total / slowest
