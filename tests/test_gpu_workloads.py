"""GPU parity on the five workloads at their full sizes, in the launch
configuration the benchmark times (same plan, same calls, same buckets).

Small workloads are compared element by element over whole partitions; the
7.5B and 13B partitions compare the reduced gradient over the whole partition
(the oracle reduces every element, chunked over host threads, to get the
global norm) and master/m/v/param at ~1M sampled positions (all tile
boundaries, both ends, random interior points), whose oracle state evolves on
its own across the steps.
"""
import numpy as np
import pytest
import torch

import oracle
from zero_partitioned_mixed_flat_gb300 import synth
from zero_partitioned_mixed_flat_gb300.workloads import WORKLOADS

from .zstep import Harness

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(h, steps):
    infos = [h.step() for _ in range(steps)]
    h.close()
    return infos


def test_gpt2_small_zero1_all_partitions(zlib):
    w = WORKLOADS["gpt2-small-zero1"]
    infos = _run(Harness(w, full=True, threads=16), w.steps)
    assert all(i["gpu"]["skipped"] == 0 for i in infos)


@pytest.mark.parametrize("rank", [0, 63])
def test_gpt2_xl_zero2_overflow_step(zlib, rank):
    w = WORKLOADS["gpt2-xl-zero2"]
    infos = _run(Harness(w, ranks=[rank], full=True, threads=16, chunk=1 << 21), w.steps)
    seen = [(i["gpu"]["skipped"], i["gpu"]["loss_scale"], i["gpu"]["step"]) for i in infos]
    assert seen == [(0, 65536.0, 1), (1, 32768.0, 1), (0, 32768.0, 2)]


def _check_gathers(h, others, gen):
    """Gather every unit (forward order) and compare sampled windows with the
    oracle's concatenation of the same windows of the N shards."""
    plan, n = h.plan, h.w.n_ranks
    shards = [h.st[0].shard] + others
    biggest = max(plan.shard_len(u) for u in range(plan.n_units)) * n
    out = torch.empty(biggest, dtype=synth.LP_DTYPES[h.w.lp], device=h.dev)
    for u in range(plan.n_units):
        sl, off = plan.shard_len(u), plan.unit_shard_offset(u)
        plan.gather(u, shards, out)
        torch.cuda.synchronize()
        starts = [0, max(0, sl - 2048)] + list(gen.integers(0, max(1, sl - 2048), 6))
        for k0 in starts:
            L = min(2048, sl - k0)
            win = [synth.to_numpy_codes(s[off + k0: off + k0 + L]) for s in shards]
            exp = oracle.gather(win).reshape(n, L)
            got = synth.to_numpy_codes(out[:sl * n].view(n, sl)[:, k0:k0 + L])
            assert np.array_equal(got, exp), (u, k0)
    plan.check()


def test_7p5b_zero3_with_gathers(zlib):
    w = WORKLOADS["7.5b-zero3"]
    h = Harness(w, full=False, threads=16, chunk=1 << 21)
    others = [synth.lp_shard(h.P, w.lp, w.master_std, 0, j, h.dev) for j in range(1, w.n_ranks)]
    gen = np.random.default_rng(7)
    for _ in range(w.steps):
        h.step()
        _check_gathers(h, others, gen)
    h.close()


def test_13b_zero2(zlib):
    w = WORKLOADS["13b-zero2"]
    infos = _run(Harness(w, full=False, threads=16, chunk=1 << 22), w.steps)
    assert all(i["gpu"]["skipped"] == 0 for i in infos)
    assert all(i["oracle"]["coef"] < 1.0 for i in infos)   # clipping is active
