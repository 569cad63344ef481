"""Host-side bookkeeping for running independent replicas of the block on several GPUs.

The attention block has no cross-GPU exchange step (kv groups and canvases are independent), so a
multi-GPU run is N replicas, one per rank.  The whole-job figure is the work of all ranks divided
by the slowest rank's time.
"""
from __future__ import annotations


def aggregate(local_ms: float, local_units: float, device=None):
    """All-reduce over the default process group: (max time in ms, summed work units).

    ``device`` is where the reduction tensors live (a CUDA device under NCCL, None for gloo)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def throughput(max_ms: float, total_units: float) -> float:
    """Whole-job units per second."""
    return total_units / (max_ms / 1e3)
