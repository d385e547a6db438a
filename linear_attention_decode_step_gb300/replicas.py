"""Host-side logic for running the decode step as independent replicas on N
GPUs (one process per GPU, weak scaling).

The KDA step shards by (stream, head) with no exchange, so ranks never talk
on the data path. The only collective is on the timing: every rank times the
same region between barriers, and the job's time is the maximum over ranks.
Each rank draws its own streams (its own seeds), so replicas do distinct work
of identical size.
"""
from __future__ import annotations

from . import inputs

RANK_SEED_STRIDE = 100_000


def rank_layer_seed(space: int, layer: int, rank: int) -> int:
    """Seed of `layer` on `rank`: the single-GPU seed, offset per rank."""
    return inputs.layer_seed(space, layer) + RANK_SEED_STRIDE * rank


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of a list of floats over all ranks (all-reduce
    MAX); returns the list unchanged without an initialised process group."""
    if dist is None or not dist.is_available() or not dist.is_initialized() \
            or dist.get_world_size() == 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(bytes_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput in bytes/s: all ranks' bytes over the slowest
    rank's time (weak scaling: every rank processes bytes_per_rank)."""
    return world * bytes_per_rank / max_seconds
