"""Replica bookkeeping for runs with one process per GPU.

The verification step has no exchange between requests on different GPUs
(attention, accept and commit are per request; the budget selection is per
batch), so N GPUs run N independent replicas of the step.  What the ranks
share is only the timing protocol: a barrier on both sides of the timed
region, the slowest rank's time, and the sum of the units every rank
processed.  The process group carries nothing else (no data-path
collective).

The rank layout comes from the launcher's environment (RANK, LOCAL_RANK,
WORLD_SIZE, MASTER_ADDR / MASTER_PORT, as torchrun sets them).
"""

from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass
class Replicas:
    rank: int = 0
    local_rank: int = 0
    world: int = 1
    device: str = "cpu"
    _dist: object = None

    @classmethod
    def from_env(cls, backend: str = "nccl", device: str | None = None) -> "Replicas":
        """Join the launcher's process group when WORLD_SIZE > 1.  `device`
        is where the timing scalars live (the rank's GPU for NCCL, the CPU
        for gloo)."""
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        r = cls(rank=rank, local_rank=local_rank, world=world, device=device or "cpu")
        if world > 1:
            import torch
            import torch.distributed as dist
            if not dist.is_initialized():
                kw = {}
                if backend == "nccl" and device is not None:
                    kw["device_id"] = torch.device(device)
                dist.init_process_group(backend, **kw)
            r._dist = dist
        return r

    @property
    def leader(self) -> bool:
        return self.rank == 0

    def barrier(self) -> None:
        if self.world > 1:
            self._dist.barrier()

    def _reduce(self, x: float, op_name: str) -> float:
        if self.world == 1:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        self._dist.all_reduce(t, op=getattr(self._dist.ReduceOp, op_name))
        return float(t.item())

    def max_over_ranks(self, x: float) -> float:
        """The slowest rank's value (the job's time)."""
        return self._reduce(x, "MAX")

    def sum_over_ranks(self, x: float) -> float:
        """Units processed by the whole job."""
        return self._reduce(x, "SUM")

    def throughput(self, units_this_rank: float, seconds_this_rank: float) -> float:
        """Whole-job throughput: every rank's units over the slowest rank's
        time (weak scaling: each replica has the same fixed work)."""
        return self.sum_over_ranks(units_this_rank) / self.max_over_ranks(seconds_this_rank)

    def close(self) -> None:
        if self.world > 1 and self._dist.is_initialized():
            self._dist.destroy_process_group()
