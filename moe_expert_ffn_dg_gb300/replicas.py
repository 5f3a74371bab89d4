"""Host-side logic of running the block as independent replicas, one per GPU.

The block acts on every token independently ("DiffusionGemma Explained":
the MoE block operates across the token axis independently), so several
GPUs split work by whole canvases and exchange nothing on the data path.
What is shared between ranks is bookkeeping only: which canvas a rank draws,
the slowest rank's time, and the aggregate throughput.
"""

from __future__ import annotations


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of the canvas that rank draws: rank 0 uses the workload's own
    seed, rank r > 0 a distinct one, so replicas process different data."""
    return base_seed if rank == 0 else base_seed + 1000 * rank


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The maximum of a per-rank scalar over all ranks (the slowest rank's
    elapsed time); returns the value itself without a process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(world: int, tokens_per_replica: int, seconds: float) -> float:
    """Whole-job tokens per second: every replica processes its own canvas
    in the (slowest rank's) time."""
    return world * tokens_per_replica / seconds
