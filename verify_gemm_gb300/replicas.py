"""Host-side logic of running the verify pass as independent replicas, one
process per GPU (launched by torchrun): the product has no exchange step on
one GPU, so N GPUs run N independent copies of the same pass and the job's
throughput is the bytes all ranks streamed divided by the slowest rank's
time.  Nothing here touches a GPU; the tests run it on CPU with gloo."""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class Ranks:
    world: int = 1
    rank: int = 0
    local: int = 0


def from_env(env=None) -> Ranks:
    """World size, rank and local rank as torchrun exports them (defaults: a
    single process)."""
    env = os.environ if env is None else env
    return Ranks(int(env.get("WORLD_SIZE", "1")), int(env.get("RANK", "0")),
                 int(env.get("LOCAL_RANK", "0")))


def init(ranks: Ranks, backend: str) -> None:
    """Join the process group (nccl for GPU ranks, gloo for CPU-only ones)."""
    if ranks.world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend)


def barrier(ranks: Ranks) -> None:
    if ranks.world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, ranks: Ranks, device=None) -> float:
    """The largest `value` over all ranks (every rank gets it)."""
    if ranks.world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_step: int, steps: int, slowest_ms: float, ranks: Ranks) -> float:
    """Whole-job GB/s: every rank streamed bytes_per_step per step, and the
    job took as long as its slowest rank."""
    return bytes_per_step * steps * ranks.world / (slowest_ms / 1e3) / 1e9
