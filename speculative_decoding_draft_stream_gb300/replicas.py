"""Replica layout of the draft sub-head over several GPUs.

The dynamic-vocabulary draft head works on one sequence's candidate stream
at a time, and nothing in a decode step reads another sequence's state: the
stream, its window counts, the bitmap, I_t and the packed sub-head are all
per sequence, and W_head is read-only.  N GPUs therefore run N independent
replicas (one process per GPU), each decoding its own sequences, with no
collective on the data path.  The only cross-rank traffic is bookkeeping of
the measurement: a barrier around the timed region and the maximum over
ranks of its duration.

Everything here is host logic and runs under any ``torch.distributed``
backend (NCCL on GPUs, gloo on CPU).
"""

from __future__ import annotations

from typing import List, Optional


def rank_sequences(rank: int, world: int, per_rank: int = 1) -> List[int]:
    """Sequence indices rank ``rank`` decodes under weak scaling.

    Every rank owns ``per_rank`` consecutive sequences of the seeded
    workload, so per-GPU work stays fixed as the world grows and the ranks'
    sets are disjoint: rank r takes r*per_rank .. (r+1)*per_rank - 1.
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if per_rank < 1:
        raise ValueError("per_rank must be positive")
    return list(range(rank * per_rank, (rank + 1) * per_rank))


def max_over_ranks(x: float, dist=None, device: Optional[object] = None) -> float:
    """Largest value of ``x`` over all ranks (the whole job ends with its
    slowest replica).  ``dist`` is ``torch.distributed`` or None for a single
    process; ``device`` is where the reduction tensor lives (a CUDA device for
    NCCL, the CPU for gloo)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units all ranks processed per second, over the slowest rank's time."""
    if seconds <= 0:
        raise ValueError("the timed region must have positive length")
    return world * units_per_rank / seconds
