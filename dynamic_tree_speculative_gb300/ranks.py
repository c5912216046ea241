"""One process per GPU: rank bookkeeping for weak-scaled batches of trees.

Trees are independent problems, so each rank builds and verifies its own
batch (its own seed); nothing is exchanged on the data path.  The only
collectives are a barrier around the timed region and a max over ranks of the
elapsed time, which turn per-rank timings into a whole-job rate.
"""
from __future__ import annotations

import dataclasses
import os

import torch
import torch.distributed as dist


@dataclasses.dataclass
class RankInfo:
    rank: int
    world: int
    local_rank: int

    @property
    def is_root(self) -> bool:
        return self.rank == 0


def rank_info() -> RankInfo:
    return RankInfo(int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
                    int(os.environ.get("LOCAL_RANK", 0)))


def init(info: RankInfo, backend: str):
    if info.world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=info.rank, world_size=info.world)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's batch: distinct per rank, equal to `seed` on rank 0."""
    return seed + 1000003 * rank


def barrier(info: RankInfo, device=None):
    if info.world > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.device(device).index or 0])
        else:
            dist.barrier()


def max_over_ranks(x: float, info: RankInfo, device="cpu") -> float:
    if info.world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, info: RankInfo, device="cpu") -> float:
    if info.world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds: float, info: RankInfo, device="cpu") -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    total = sum_over_ranks(units_per_rank, info, device)
    slowest = max_over_ranks(seconds, info, device)
    return total / slowest
