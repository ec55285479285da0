"""Independent replicas of the workload, one process per GPU.

The expert path has no exchange step on one GPU, so N GPUs run N independent
copies of the benchmark workload (weak scaling).  The only cross-rank logic is
the timing: every rank times its own region between two barriers, and the job's
throughput is the units all ranks processed divided by the slowest rank's time.
"""

from __future__ import annotations

import os
from typing import Mapping, Optional, Tuple

import torch


def env_ranks() -> Tuple[int, int, int]:
    """(rank, world_size, local_rank) from the launcher's environment (1 process if unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def replica_throughput(local_ms: float, local_units: float,
                       device: Optional[torch.device] = None) -> Tuple[float, float, float]:
    """Whole-job throughput of independent replicas.

    Returns (units per second over all ranks, the slowest rank's milliseconds, the
    units of all ranks).  With no process group (or one rank) it is the local figure.
    ``device`` holds the reduction tensors: the GPU for NCCL, the CPU for gloo.
    """
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_units / (local_ms / 1e3), local_ms, local_units
    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    max_ms, units = float(t.item()), float(u.item())
    return units / (max_ms / 1e3), max_ms, units


def launch_plan(gpus: int, env: Mapping[str, str]) -> Tuple[str, str]:
    """What a benchmark asked for ``gpus`` GPUs does, given the launcher's environment.

    ("run", "")        run in this process: one GPU, or one rank of a launcher with WORLD_SIZE == gpus;
    ("relaunch", "")   no launcher and gpus > 1: start gpus local ranks (one per GPU) and wait;
    ("error", why)     gpus < 1, or a launcher whose WORLD_SIZE differs from gpus.
    """
    if gpus < 1:
        return "error", f"--gpus {gpus}: at least one GPU"
    world = env.get("WORLD_SIZE")
    if world is None:
        return ("relaunch", "") if gpus > 1 else ("run", "")
    if int(world) != gpus:
        return "error", f"--gpus {gpus} but the launcher started WORLD_SIZE={world} ranks"
    return "run", ""
