"""Multi-rank host logic on CPU (gloo, world sizes 2 and 3).

Two processes each own half of the partitions of a small job.  The device
kernels are stood in for by the CPU oracle (this is a host-logic test): each
rank reduces its partitions, the ranks exchange (sum of squares, overflow)
with parallel_host.exchange_stats, decide, update, and all-gather the new
parameters.  Both ranks must take the identical decision, and the result must
equal the single-process step over all partitions bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from zero_partitioned_mixed_flat_gb300.parallel_host import (combine_stats, exchange_stats,
                                                            partitions_for)

N, P, LP, S = 4, 4096, 0, 1024.0
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01, adamw=1, clip=0.5)


def _inputs(step, inject=None):
    rng = np.random.default_rng(100 + step)
    g = (rng.standard_normal((N, N, P)) * 1e-3 * S).astype(np.float16)  # [partition, rank, elem]
    if inject is not None:
        g[inject] = np.inf
    return g.view(np.uint16)


def _step_partitions(orc, parts, grads, state, t, remote=None):
    """Reduce + (exchange) + decide + Adam on `parts`; returns (decision, params)."""
    local = []
    red = {}
    for p in parts:
        red[p], ss, of = orc.reduce(list(grads[p]), LP, S)
        local.append((ss, of))
    ss, of = combine_stats(local)
    if remote is not None:
        ss, of = remote(ss, of)
    d = orc.decide(ss, of, HP["clip"], S, t, 0, 1000, HP["beta1"], HP["beta2"])
    params = {}
    for p in parts:
        master, m, v = state[p]
        params[p] = orc.adam(red[p], master, m, v, LP, d["coef"], d["skip"], HP["lr"],
                             HP["beta1"], HP["beta2"], HP["eps"], HP["wd"], HP["adamw"],
                             d["bc1"], d["bc2"])
    return d, params


def _fresh_state():
    rng = np.random.default_rng(7)
    return {p: ((rng.standard_normal(P) * 0.02).astype(np.float32), np.zeros(P, np.float32),
                np.zeros(P, np.float32)) for p in range(N)}


def _worker(rank, world, port, inject_at, q):
    import torch.distributed as dist
    import oracle as orc
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = partitions_for(world, rank, N)
        state = _fresh_state()
        t = 0
        out = []
        for step in range(1, 4):
            grads = _inputs(step, inject_at if step == 2 else None)
            # the combine must be in rank order: sum of each rank's (already
            # rank-ordered) partition sums -- exchange_stats does exactly that
            d, params = _step_partitions(orc, mine, grads, state, t,
                                         remote=lambda ss, of: exchange_stats(ss, of))
            if not d["skip"]:
                t = d["step"]
            full = [None] * world
            dist.all_gather_object(full, {p: params[p].tolist() for p in mine})
            merged = {}
            for f in full:
                merged.update(f)
            out.append((d["norm"], d["coef"], d["skip"], d["step"],
                        [merged[p] for p in range(N)] if not d["skip"] else None))
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_partitions_for_covers_each_partition_once():
    for world in (1, 2, 3, 8):
        for n in (1, 4, 16, 17):
            owned = sorted(p for r in range(world) for p in partitions_for(world, r, n))
            assert owned == list(range(n))
    with pytest.raises(ValueError):
        partitions_for(2, 2, 4)


@pytest.mark.parametrize("world,inject_at", [(2, None), (2, (3, 1, 77)), (3, None), (3, (0, 2, 5))])
def test_ranks_equal_one_process(orc, world, inject_at):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, inject_at, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank took the same decisions
    for r in range(1, world):
        for a, b in zip(res[0], res[r]):
            assert a[:4] == b[:4]
    # and they equal one process owning every partition; the single process
    # combines per-rank sums in the same order the exchange does
    state = _fresh_state()
    t = 0
    for step, got in zip(range(1, 4), res[0]):
        grads = _inputs(step, inject_at if step == 2 else None)
        owners = [partitions_for(world, r, N) for r in range(world)]

        def remote(_ss, _of, grads=grads, owners=owners):
            return combine_stats([combine_stats([orc.reduce(list(grads[p]), LP, S)[1:]
                                                 for p in o]) for o in owners])
        d, params = _step_partitions(orc, list(range(N)), grads, state, t, remote=remote)
        if not d["skip"]:
            t = d["step"]
        assert (d["norm"], d["coef"], d["skip"], d["step"]) == got[:4]
        if not d["skip"]:
            assert [params[p].tolist() for p in range(N)] == got[4]
    if inject_at is not None:
        assert res[0][1][2] == 1     # the overflow on one rank skipped the step everywhere
