"""Host-side logic of a real multi-rank job (one process per GPU).

The step shards with no data-path exchange except one: the global gradient
norm and the overflow flag need every rank's partition ("10.6 ZeRO 与 FSDP"
§10.6.1: all-reduce; "从'年糕切片'理解ZeRO" §4.2 global clipping).  Each rank
reduces its partitions (zero_reduce_partition), reads its local sum of squares
and overflow (zero_partition_stats), and all ranks exchange them here.  Every
rank then adds the same values in the same (rank) order, so all ranks hand
zero_step_set_global_stats bit-identical totals and take the same decision.
"""
from typing import List, Optional, Tuple


def partitions_for(world_size: int, rank: int, n_partitions: int) -> List[int]:
    """The partitions one process owns: round-robin over the world."""
    if world_size < 1 or not 0 <= rank < world_size:
        raise ValueError("bad world size / rank")
    return list(range(rank, n_partitions, world_size))


def combine_stats(per_rank: List[Tuple[float, int]]) -> Tuple[float, int]:
    """Sum of squares added in rank order, overflow OR-ed."""
    total, of = 0.0, 0
    for ss, o in per_rank:
        total += float(ss)
        of |= 1 if o else 0
    return total, of


def exchange_stats(local_sumsq: float, local_overflow: int, group=None,
                   device: Optional[str] = None) -> Tuple[float, int]:
    """All-gather every rank's (sum of squares, overflow) and combine them in
    rank order.  device: where the exchange tensor lives ("cpu" for gloo,
    "cuda" for nccl; default from the backend)."""
    import torch
    import torch.distributed as dist
    if device is None:
        device = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    ws = dist.get_world_size(group)
    t = torch.tensor([float(local_sumsq), float(1 if local_overflow else 0)],
                     dtype=torch.float64, device=device)
    out = [torch.empty_like(t) for _ in range(ws)]
    dist.all_gather(out, t, group=group)
    return combine_stats([(float(o[0]), int(o[1].item() != 0)) for o in out])
