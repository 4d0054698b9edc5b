"""libzero's multi-rank path across processes, on one GPU (stages 2 and 3).

Two or three processes share the GPU and exchange bytes with gloo (through
host memory).  No kernel of one process waits for another process: the only
exchanges are host-side collectives between a step's launches.  Two flows:

 - ownership: N = 4 partitions owned round-robin by W = 2 or 3 processes.
   Each process reduces the partitions it owns (their slices generated in
   place), exports its per-partition statistics (zero_partition_stats),
   all-reduces them, hands the sum to zero_step_set_global_stats, and updates
   its partitions;
 - full data path: W = N = 2 or 3 ranks, each holding its own flat gradient.
   An all-to-all hands every rank the N slices of its partition (the
   reduce-scatter's input), the statistics go as above, and after the update
   the lp partitions are all-gathered into every rank's full layout;
 - stage 3, W = N = 2 or 3: the same reduce-scatter and statistics, the update
   into each rank's own shard, then every unit all-gathered across the ranks
   into a layer buffer, checked against the oracle's gather of the shards.

Every rank's decision must be identical, and its master, m, v and parameters
bit-identical to one process stepping all N partitions through the parity
harness, which itself checks every step against the CPU oracle (reduced
gradient bit for bit, decision, state within the stated bars).
"""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from zero_partitioned_mixed_flat_gb300 import synth
from zero_partitioned_mixed_flat_gb300.workloads import Workload

from .zstep import Harness

pytestmark = pytest.mark.gpu

SEED = 0
STEPS = 3


def _workload(n, stage=2):
    if stage == 3:
        return Workload(name="multirank3", sizes=[70_000, 5, 33_000, 100_000, 7], n_ranks=n,
                        stage=3, unit_of_tensor=[0, 0, 1, 2, 2], lp=0, ranks=list(range(n)),
                        steps=STEPS, loss_scale=1024.0, growth_interval=1000,
                        grads_times_scale=True, inject_inf_step=2, align=8, lr=1e-3, clip=0.05)
    return Workload(name="multirank", sizes=[100_000, 7, 33_333], n_ranks=n, stage=2, lp=0,
                    ranks=list(range(n)), steps=STEPS, loss_scale=1024.0, growth_interval=1000,
                    grads_times_scale=True, inject_inf_step=2, align=8, lr=1e-3, clip=0.05)


def _child(rank, world, port, wfields, mode, q):
    import torch.distributed as dist
    import zero_partitioned_mixed_flat_gb300 as Z
    from zero_partitioned_mixed_flat_gb300 import synth
    from zero_partitioned_mixed_flat_gb300.parallel_host import (allgather_partitions,
                                                                allgather_unit,
                                                                exchange_gradients,
                                                                global_decision_inputs,
                                                                partitions_for)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        Z.load()
        w = Workload(**wfields)
        N = w.n_ranks
        plan = Z.ZeroPlan(-1, N, w.sizes, w.align, w.stage, w.unit_of_tensor, w.lp,
                          growth_interval=w.growth_interval)
        P = plan.part_len
        mine = partitions_for(world, rank, N) if mode == "owned" else [rank]
        keep = {p: plan.keep_ranges(p) for p in range(N)}
        master = {p: synth.master_init(P, w.master_std, SEED, p, dev, keep[p]) for p in mine}
        m = {p: torch.zeros(P, device=dev) for p in mine}
        v = {p: torch.zeros(P, device=dev) for p in mine}
        g = {p: torch.empty(P, device=dev) for p in mine}
        param = torch.zeros(plan.psi_padded, dtype=synth.LP_DTYPES[w.lp], device=dev)
        shard = torch.zeros(P, dtype=synth.LP_DTYPES[w.lp], device=dev)      # stage 3
        layer = torch.empty(max(plan.shard_len(u) for u in range(plan.n_units)) * N,
                            dtype=synth.LP_DTYPES[w.lp], device=dev)
        stats = torch.empty(2 * N, dtype=torch.float64, device=dev)
        S = w.loss_scale
        out = []
        for step in range(1, STEPS + 1):
            scale = S if w.grads_times_scale else 1.0
            inject = None
            if w.inject_inf_step and step == w.inject_inf_step:
                inject = synth.inject_position(SEED, step, 0, N, keep[0])  # partition 0
            if mode == "owned":
                for p in mine:
                    sl = [synth.grad_slice(P, w.lp, w.grad_std, scale, SEED, step, j, p, dev, keep[p])
                          for j in range(N)]
                    if inject is not None and p == 0:
                        sl[inject[0]][inject[1]] = float("inf")
                    plan.reduce(p, sl, g[p], S)
            else:
                # this rank's own flat gradient over every partition
                full = torch.empty(N * P, dtype=synth.LP_DTYPES[w.lp], device=dev)
                for p in range(N):
                    full[p * P:(p + 1) * P] = synth.grad_slice(P, w.lp, w.grad_std, scale, SEED, step,
                                                               rank, p, dev, keep[p])
                if inject is not None and inject[0] == rank:
                    full[inject[1]] = float("inf")
                slices = torch.empty((N, P), dtype=full.dtype, device=dev)
                exchange_gradients(full, slices)
                plan.reduce(rank, [slices[j] for j in range(N)], g[rank], S)
            global_decision_inputs(plan, stats)
            for p in mine:
                plan.adam(p, g[p], master[p], m[p], v[p], shard if w.stage == 3 else param, w.lr,
                          w.beta1, w.beta2, w.eps, w.wd, int(w.adamw), S, w.clip)
            res = plan.result()
            layers = None
            if w.stage == 3:
                # every unit's shards all-gathered into a layer buffer
                layers = []
                for u in range(plan.n_units):
                    layers.append(allgather_unit(plan, u, shard, layer).view(torch.int16).cpu().numpy())
            elif mode == "data":
                allgather_partitions(param, rank, P)
            torch.cuda.synchronize()
            own = shard if w.stage == 3 else None
            state = {p: (master[p].cpu().numpy(), m[p].cpu().numpy(), v[p].cpu().numpy(),
                         (own if own is not None else param[p * P:(p + 1) * P]).view(torch.int16)
                         .cpu().numpy()) for p in mine}
            full_param = param.view(torch.int16).cpu().numpy() if (mode == "data" and w.stage != 3) \
                else None
            out.append((res, state, full_param, layers))
            S = res["loss_scale"]
        plan.close()
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(world, w, mode):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    fields = dataclasses.asdict(w)
    procs = [ctx.Process(target=_child, args=(r, world, port, fields, mode, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        res = dict(q.get(timeout=600) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=120)
            if p.is_alive():
                p.kill()
    for p in procs:
        assert p.exitcode == 0
    return res


def _same_decision(a, b):
    """Step results equal, the norm compared by its bits (inf/NaN on a skipped step)."""
    return (a.keys() == b.keys() and np.float64(a["norm"]).tobytes() == np.float64(b["norm"]).tobytes()
            and all(a[k] == b[k] for k in a if k != "norm"))


def _reference(w):
    """One process, every partition: per step (decision, state per partition,
    param, and in stage 3 the oracle's gather of every unit from the shards)."""
    import oracle
    h = Harness(w)
    ref = []
    for _ in range(STEPS):
        info = h.step()                      # checked against the oracle
        P = h.P
        torch.cuda.synchronize()
        if w.stage == 3:
            lp_of = {r: h.st[r].shard for r in h.ranks}
        else:
            lp_of = {r: h.param[r * P:(r + 1) * P] for r in h.ranks}
        state = {r: (h.st[r].master.cpu().numpy(), h.st[r].m.cpu().numpy(),
                     h.st[r].v.cpu().numpy(), lp_of[r].view(torch.int16).cpu().numpy())
                 for r in h.ranks}
        layers = None
        if w.stage == 3:
            layers = []
            for u in range(h.plan.n_units):
                sl, off = h.plan.shard_len(u), h.plan.unit_shard_offset(u)
                layers.append(oracle.gather([synth.to_numpy_codes(h.st[r].shard[off:off + sl])
                                             for r in h.ranks]).view(np.int16))
        full = h.param.view(torch.int16).cpu().numpy() if h.param is not None else None
        ref.append((info["gpu"], state, full, layers))
    h.close()
    return ref


@pytest.mark.parametrize("world,mode,stage", [(2, "owned", 2), (3, "owned", 2), (2, "data", 2),
                                              (3, "data", 2), (2, "data", 3), (3, "data", 3)])
def test_ranks_across_processes_equal_one_process(zlib, world, mode, stage):
    w = _workload(4 if mode == "owned" else world, stage)
    ref = _reference(w)
    res = _run(world, w, mode)
    seen_skip = False
    for step in range(STEPS):
        r_dec, r_state, r_param, r_layers = ref[step]
        seen_skip |= bool(r_dec["skipped"])
        for rank in range(world):
            dec, state, full, layers = res[rank][step]
            assert _same_decision(dec, r_dec), (step, rank, dec, r_dec)
            for p, arrays in state.items():
                for name, a, b in zip(("master", "m", "v", "param"), arrays, r_state[p]):
                    assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (step, rank, p, name)
            if full is not None:
                assert np.array_equal(full, r_param), (step, rank)
            if stage == 3:      # every unit gathered across the ranks = the oracle's gather
                assert len(layers) == len(r_layers)
                for u, (a, b) in enumerate(zip(layers, r_layers)):
                    assert np.array_equal(a, b), (step, rank, u)
    assert seen_skip    # the overflow on partition 0 skipped the step on every rank


@pytest.mark.parametrize("seed", [1, 2])
def test_random_jobs_across_processes(zlib, seed):
    # random layouts, world sizes and stages through the full data path
    rng = np.random.default_rng(300 + seed)
    world = int(rng.choice([2, 3]))
    stage = int(rng.choice([2, 3]))
    k = int(rng.integers(2, 6))
    sizes = [int(x) for x in rng.integers(1, 60_000, k)]
    units = None
    if stage == 3:
        units, u = [0], 0
        for _ in range(k - 1):
            u += int(rng.integers(0, 2))
            units.append(u)
    w = dataclasses.replace(_workload(world, stage), sizes=sizes, unit_of_tensor=units,
                            lp=int(rng.integers(0, 2)), clip=float(rng.choice([0.0, 0.05])),
                            adamw=bool(rng.integers(0, 2)))
    if w.lp == 1:
        w = dataclasses.replace(w, loss_scale=1.0, grads_times_scale=False, inject_inf_step=0)
    ref = _reference(w)
    res = _run(world, w, "data")
    for step in range(STEPS):
        r_dec, r_state, r_param, r_layers = ref[step]
        for rank in range(world):
            dec, state, full, layers = res[rank][step]
            assert _same_decision(dec, r_dec), (seed, step, rank)
            for p, arrays in state.items():
                for name, a, b in zip(("master", "m", "v", "param"), arrays, r_state[p]):
                    assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (seed, step, rank, name)
            if stage == 3:
                for a, b in zip(layers, r_layers):
                    assert np.array_equal(a, b), (seed, step, rank)
            else:
                assert np.array_equal(full, r_param), (seed, step, rank)
