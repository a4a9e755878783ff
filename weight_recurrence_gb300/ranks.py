"""Host-side bookkeeping for one process per GPU.

The forward and decode passes of kernelised linear attention treat every
(batch, head) pair on its own ("Transformers are RNNs", sec. 3.2: each head
is an independent sum over its own sequence), so a job that spans several
GPUs gives each rank its own batch and runs no collective on the data path.
What ranks exchange is bookkeeping only: the slowest rank's step time, from
which the whole-job rate follows.
"""
from __future__ import annotations

import os


def world_from_env():
    """(rank, local_rank, world_size) from the launcher's environment (1 process if unset)."""
    def _int(name, default):
        try:
            return int(os.environ.get(name, default))
        except ValueError:
            return default
    return _int("RANK", 0), _int("LOCAL_RANK", 0), _int("WORLD_SIZE", 1)


def reduce_max(x: float, dist=None, device="cpu") -> float:
    """Maximum of ``x`` over all ranks of the default process group.

    ``dist`` is ``torch.distributed`` (or None for a single process);
    ``device`` is where the one-element tensor lives (a CUDA device for NCCL,
    "cpu" for gloo)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds_per_step: float) -> float:
    """Units per second of the whole job when each of ``world`` ranks handles
    ``units_per_rank`` units per step and the step lasts ``seconds_per_step``
    (the slowest rank's time)."""
    if world < 1 or seconds_per_step <= 0:
        raise ValueError("world must be >= 1 and the step time > 0")
    return world * units_per_rank / seconds_per_step
