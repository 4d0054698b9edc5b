"""Host side of a multi-rank ZeRO job: one process per data-parallel rank (or
per group of simulated ranks), with torch.distributed moving the bytes.

What crosses between ranks in one step ("10.6 ZeRO 与 FSDP" §10.6.1 and
§10.6.2 Steps 2-4; "从'年糕切片'理解ZeRO" §4.2 for the global norm):
 - the reduce-scatter's input: rank j sends rank r the r-th 1/N of its flat
   gradient (an all-to-all).  Rank r's reduce kernel then adds the N received
   slices in rank order 0..N-1, so no collective's summation order enters the
   result;
 - two scalars per partition (sum of squares, overflow): the vectors of
   zero_partition_stats, summed element-wise by an all-reduce.  Each partition
   has one owner and every other rank holds an exact +0 there, so the sum is
   exact in any order and equals the vector of one process that reduced every
   partition; zero_step_set_global_stats then makes every rank take the same
   decision, bit for bit;
 - stages 1/2: the updated lp partitions, all-gathered into the full layout
   (Step 4).  Stage 3 gathers a layer's shards the same way when it is needed.
This module only moves bytes and orders calls: every addition of the step runs
in libzero's kernels.  With the gloo backend, device tensors are staged
through host memory (gloo moves host buffers); with nccl they move directly.
"""
from typing import List


def partitions_for(world_size: int, rank: int, n_partitions: int) -> List[int]:
    """The partitions one process owns: round-robin over the world."""
    if world_size < 1 or not 0 <= rank < world_size:
        raise ValueError("bad world size / rank")
    return list(range(rank, n_partitions, world_size))


def _staged(t, group):
    """(tensor the collective works on, whether it is a host copy of t)."""
    import torch.distributed as dist
    if t.is_cuda and dist.get_backend(group) == "gloo":
        return t.cpu(), True
    return t, False


def allreduce_stats(stats, group=None):
    """Sum the (2*N float64) statistics vectors of every rank in place."""
    import torch.distributed as dist
    work, staged = _staged(stats, group)
    dist.all_reduce(work, op=dist.ReduceOp.SUM, group=group)
    if staged:
        stats.copy_(work)
    return stats


def exchange_gradients(grad_full, slices, group=None):
    """Reduce-scatter input of a world of N = world-size ranks: grad_full is
    this rank's flat lp gradient (N*P elements, partition r at [r*P, (r+1)*P));
    slices ([N, P], same dtype) receives row j = rank j's gradient over this
    rank's partition, the input zero_reduce_partition adds in rank order."""
    import torch.distributed as dist
    n = dist.get_world_size(group)
    if slices.dim() != 2 or slices.shape[0] != n or grad_full.numel() != slices.numel():
        raise ValueError("slices must be [world, P] and grad_full N*P elements")
    src, s_staged = _staged(grad_full.reshape(-1), group)
    dst, d_staged = _staged(slices.reshape(-1), group)
    dist.all_to_all_single(dst, src, group=group)
    if d_staged:
        slices.reshape(-1).copy_(dst)
    return slices


def allgather_partitions(param_full, rank: int, part_len: int, group=None):
    """Stage-1/2 step end: every rank's updated partition [r*P, (r+1)*P) of its
    full lp layout is all-gathered into every rank's full layout, in place."""
    import torch.distributed as dist
    mine = param_full[rank * part_len:(rank + 1) * part_len]
    out, staged = _staged(param_full, group)
    if staged or dist.get_backend(group) == "gloo":
        src = mine.cpu() if mine.is_cuda else mine.clone()
    else:
        src = mine  # nccl: the input aliases its own place in the output
    dist.all_gather_into_tensor(out, src, group=group)
    if staged:
        param_full.copy_(out)
    return param_full


def allgather_unit(plan, unit: int, shard, layer, group=None):
    """Stage 3 ("10.6 ZeRO 与 FSDP" §10.6.4 step 1): all-gather unit `unit`'s
    shards of every rank (this rank's is its P-element shard buffer `shard`)
    into `layer`, whose first N * U_p/N elements receive the unit in full
    layout (rank j's shard at [j * U_p/N, (j+1) * U_p/N))."""
    import torch.distributed as dist
    n = dist.get_world_size(group)
    if n != plan.n_ranks:
        raise ValueError("one process per rank: world size must equal N")
    sl, off = plan.shard_len(unit), plan.unit_shard_offset(unit)
    mine = shard[off:off + sl]
    out = layer[:n * sl]
    work, staged = _staged(out, group)
    if staged or dist.get_backend(group) == "gloo":
        src = mine.cpu() if mine.is_cuda else mine.clone()
    else:
        src = mine
    dist.all_gather_into_tensor(work, src, group=group)
    if staged:
        out.copy_(work)
    return out


def global_decision_inputs(plan, stats, group=None):
    """The multi-rank exchange of one step, between the reduces and the first
    Adam call: export this rank's per-partition statistics into `stats`
    (2*N float64 on the device), all-reduce them, and hand the result to the
    plan.  Everything is ordered on torch's current stream (the plan's
    default stream; nccl's all-reduce is joined to it, and gloo's host staging
    copies synchronise with it)."""
    plan.partition_stats(stats)
    allreduce_stats(stats, group)
    plan.set_global_stats(stats)
    return stats
