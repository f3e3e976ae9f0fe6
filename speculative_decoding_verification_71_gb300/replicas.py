"""Host-side helpers for running verification as independent replicas.

Sequences are independent, so N GPUs verify N shards of a batch (or N
batches) with no exchange on the data path; only scalar results cross ranks:
the counters are summed and the slowest rank's time is taken.
"""
from __future__ import annotations

import torch


def shard(B: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, stop) of a batch of B sequences for `rank`; the
    first B % world ranks get one extra sequence."""
    if world <= 0 or not 0 <= rank < world or B < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


COUNT_KEYS = ("sequences", "drafts_proposed", "drafts_accepted", "emitted", "spec_off",
              "zero_residual", "error_sequences")


def reduce_counts(stats: dict, group=None) -> dict:
    """Sum the integer counters of `spec_verify_stats` over all ranks and
    recompute the means (torch.distributed must be initialised)."""
    import torch.distributed as dist
    t = torch.tensor([int(stats[k]) for k in COUNT_KEYS], dtype=torch.int64)
    if dist.get_backend(group) == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    out = {k: int(v) for k, v in zip(COUNT_KEYS, t.tolist())}
    seqs = out["sequences"]
    out["mean_emitted"] = out["emitted"] / seqs if seqs else 0.0
    out["mean_accepted"] = out["drafts_accepted"] / seqs if seqs else 0.0
    out["accept_rate"] = out["drafts_accepted"] / out["drafts_proposed"] if out["drafts_proposed"] else 0.0
    return out


def max_over_ranks(x: float, group=None) -> float:
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    if dist.get_backend(group) == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())
