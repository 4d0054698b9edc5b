"""Multi-rank host logic on CPU (gloo, world sizes 2 and 3).

Processes each own some of the partitions of a small job.  The device kernels
are stood in for by the CPU oracle (this is a host-logic test; the same flow
through libzero runs on the GPU in test_gpu_multirank.py).  Each rank reduces
its partitions into a per-partition statistics vector (zero for partitions it
does not own), the ranks all-reduce the vectors with
parallel_host.allreduce_stats, decide, update their partitions, and
all-gather the new parameters with parallel_host.allgather_partitions.

The all-reduced vector must equal, bit for bit, the vector of one process
that reduced every partition (only exact zeros are added), so every rank and
the single process take the same decision and produce the same parameters,
whatever the world size or the ownership.  The reduce-scatter's data path
(exchange_gradients, an all-to-all) is checked on its own.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from zero_partitioned_mixed_flat_gb300.parallel_host import (allgather_partitions,
                                                            allreduce_stats,
                                                            exchange_gradients,
                                                            partitions_for)

N, P, LP, S = 4, 4096, 0, 1024.0
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01, adamw=1, clip=0.5)


def _inputs(step, inject=None):
    rng = np.random.default_rng(100 + step)
    g = (rng.standard_normal((N, N, P)) * 1e-3 * S).astype(np.float16)  # [partition, rank, elem]
    if inject is not None:
        g[inject] = np.inf
    return g.view(np.uint16)


def _fresh_state():
    rng = np.random.default_rng(7)
    return {p: ((rng.standard_normal(P) * 0.02).astype(np.float32), np.zeros(P, np.float32),
                np.zeros(P, np.float32)) for p in range(N)}


def _reduce_into_vector(orc, parts, grads):
    """Reduced gradients of `parts` and the 2N statistics vector (zeros elsewhere)."""
    vec = np.zeros(2 * N, np.float64)
    red = {}
    for p in parts:
        red[p], ss, of = orc.reduce(list(grads[p]), LP, S)
        vec[p] = ss
        vec[N + p] = 1.0 if of else 0.0
    return red, vec


def _decide_and_update(orc, parts, red, vec, state, t):
    # any fixed order stands in for the library's tree: every rank applies it
    # to the same vector
    ss = 0.0
    for p in range(N):
        ss += float(vec[p])
    of = int(np.any(vec[N:] != 0))
    d = orc.decide(ss, of, HP["clip"], S, t, 0, 1000, HP["beta1"], HP["beta2"])
    params = {}
    for p in parts:
        master, m, v = state[p]
        params[p] = orc.adam(red[p], master, m, v, LP, d["coef"], d["skip"], HP["lr"],
                             HP["beta1"], HP["beta2"], HP["eps"], HP["wd"], HP["adamw"],
                             d["bc1"], d["bc2"])
    return d, params


def _worker(rank, world, port, inject_at, q):
    import torch.distributed as dist
    import oracle as orc
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = partitions_for(world, rank, N)
        state = _fresh_state()
        full = torch.zeros(N * P, dtype=torch.int16)       # lp codes of the full layout
        t = 0
        out = []
        for step in range(1, 4):
            grads = _inputs(step, inject_at if step == 2 else None)
            red, vec = _reduce_into_vector(orc, mine, grads)
            stats = torch.from_numpy(vec)
            allreduce_stats(stats)
            d, params = _decide_and_update(orc, mine, red, stats.numpy(), state, t)
            if not d["skip"]:
                t = d["step"]
                for p in mine:
                    full[p * P:(p + 1) * P] = torch.from_numpy(params[p].view(np.int16))
            # every partition's owner sends it; round-robin owners -> gather per owner
            for p in range(N):
                owner = p % world
                piece = full[p * P:(p + 1) * P].clone().view(torch.float16)  # gloo moves fp16 bytes
                dist.broadcast(piece, src=owner)
                full[p * P:(p + 1) * P] = piece.view(torch.int16)
            out.append((stats.numpy().copy(), d["norm"], d["coef"], d["skip"], d["step"],
                        full.numpy().copy()))
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _spawn(target, world, *args, timeout=120):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port) + args + (q,)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        res = dict(q.get(timeout=timeout) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    for p in procs:
        assert p.exitcode == 0
    return res


def test_partitions_for_covers_each_partition_once():
    for world in (1, 2, 3, 8):
        for n in (1, 4, 16, 17):
            owned = sorted(p for r in range(world) for p in partitions_for(world, r, n))
            assert owned == list(range(n))
    with pytest.raises(ValueError):
        partitions_for(2, 2, 4)


@pytest.mark.parametrize("world,inject_at", [(2, None), (2, (3, 1, 77)), (3, None), (3, (0, 2, 5))])
def test_ranks_equal_one_process(orc, world, inject_at):
    res = _spawn(_worker, world, inject_at)
    for r in range(1, world):      # every rank holds the same vector, decision and layout
        for a, b in zip(res[0], res[r]):
            assert a[0].tobytes() == b[0].tobytes()
            assert a[1:5] == b[1:5]
            assert np.array_equal(a[5], b[5])
    state = _fresh_state()
    full = np.zeros(N * P, np.int16)
    t = 0
    for step, got in zip(range(1, 4), res[0]):
        grads = _inputs(step, inject_at if step == 2 else None)
        red, vec = _reduce_into_vector(orc, list(range(N)), grads)
        assert vec.tobytes() == got[0].tobytes()   # the all-reduce added only exact zeros
        d, params = _decide_and_update(orc, list(range(N)), red, vec, state, t)
        assert (d["norm"], d["coef"], d["skip"], d["step"]) == got[1:5]
        if not d["skip"]:
            t = d["step"]
            for p in range(N):
                full[p * P:(p + 1) * P] = params[p].view(np.int16)
        assert np.array_equal(full, got[5])
    if inject_at is not None:
        assert res[0][1][3] == 1     # the overflow on one rank skipped the step everywhere


def _data_path_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        part = 40
        # rank j's flat gradient: value 1000*j + flat index (exact in fp16 below 2048)
        grad = (torch.arange(world * part, dtype=torch.float32) + 1000 * rank).to(torch.float16)
        slices = torch.empty((world, part), dtype=torch.float16)
        exchange_gradients(grad, slices)
        layout = torch.full((world * part,), -1, dtype=torch.float16)
        layout[rank * part:(rank + 1) * part] = rank
        allgather_partitions(layout, rank, part)
        q.put((rank, (slices.float().numpy(), layout.float().numpy())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_reduce_scatter_input_and_allgather_move_the_right_bytes(world):
    res = _spawn(_data_path_worker, world)
    part = 40
    for r in range(world):
        slices, layout = res[r]
        for j in range(world):      # row j: rank j's gradient over partition r
            exp = 1000 * j + np.arange(r * part, (r + 1) * part)
            assert np.array_equal(slices[j], exp.astype(np.float16).astype(np.float32)), (r, j)
        assert np.array_equal(layout, np.repeat(np.arange(world), part))
