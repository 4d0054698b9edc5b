"""GPU parity on the five workloads at their full sizes, in the launch
configuration the benchmark times (the schedule module's call list: same plan,
same calls, same buckets, the same two-stream gather prefetch).

Every workload is compared element by element over whole partitions: the
reduced gradient bit for bit, and master, m, v and the lp parameters against
the oracle's own state, which evolves on its own across the steps (the oracle
runs piecewise on the host's threads: 812.5M elements per step at 13B).  The
7.5B step's 66 unit gathers are checked against the oracle's gather in sampled
windows of every rank's segment of every unit.
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


def _synthetic_shards(plan, w, dev):
    """Every rank's lp shard buffer as seeded synthetic data: the gathers are
    checked on inputs that no kernel produced."""
    return [synth.lp_shard(plan.part_len, w.lp, w.master_std, 9, j, dev) for j in range(w.n_ranks)]


def _windows(sl, gen):
    """Block-aligned (128) windows of one unit shard: both ends + 6 random."""
    L = min(2048, sl)
    starts = {0, (sl - L) // 128 * 128}
    starts |= {int(x) // 128 * 128 for x in gen.integers(0, max(1, sl - L), 6)}
    return [(k0, min(L, sl - k0)) for k0 in sorted(starts)]


def _check_gathers(plan, w, shards, gen, quantized, fmt=0):
    """Gather every unit (forward order) and compare sampled windows with the
    oracle's gather (or quantize + dequantizing gather) of the same windows."""
    n, dev = w.n_ranks, shards[0].device
    plan.set_gather_quantization(fmt)
    o_quant = oracle.quantize_blocks_fp8 if fmt else oracle.quantize_blocks
    o_dequant = oracle.dequant_gather_fp8 if fmt else oracle.dequant_gather
    biggest = max(plan.shard_len(u) for u in range(plan.n_units)) * n
    out = torch.empty(biggest, dtype=synth.LP_DTYPES[w.lp], device=dev)
    if quantized:
        codes = [torch.empty(plan.part_len, dtype=torch.int8, device=dev) for _ in range(n)]
        scales = [torch.empty(plan.part_len // 128, dtype=torch.float32, device=dev) for _ in range(n)]
        for j in range(n):
            plan.quantize(shards[j], codes[j], scales[j])
    for u in range(plan.n_units):
        sl, off = plan.shard_len(u), plan.unit_shard_offset(u)
        if quantized:
            plan.gather_quantized(u, codes, scales, out)
        else:
            plan.gather(u, shards, out)
        torch.cuda.synchronize()
        for k0, L in _windows(sl, gen):
            win = [synth.to_numpy_codes(t[off + k0: off + k0 + L]) for t in shards]
            if quantized:
                qs = [o_quant(x, w.lp, 128) for x in win]
                exp = o_dequant([q for q, _ in qs], [c for _, c in qs], w.lp, 128)
            else:
                exp = oracle.gather(win)
            got = synth.to_numpy_codes(out[:sl * n].view(n, sl)[:, k0:k0 + L])
            assert np.array_equal(got, exp.reshape(n, L)), (u, k0)
    plan.check()


def test_7p5b_zero3_with_gathers(zlib):
    w = WORKLOADS["7.5b-zero3"]
    h = Harness(w, full=True, threads=16, chunk=1 << 21, gather_windows=True)
    for _ in range(w.steps):
        h.step()
    assert h.gather_log == [2 * h.plan.n_units] * w.steps
    shards = _synthetic_shards(h.plan, w, h.dev)
    _check_gathers(h.plan, w, shards, np.random.default_rng(7), quantized=False)
    _check_gathers(h.plan, w, shards, np.random.default_rng(8), quantized=True)
    _check_gathers(h.plan, w, shards, np.random.default_rng(9), quantized=True, fmt=1)
    h.close()


def test_13b_zero2(zlib):
    w = WORKLOADS["13b-zero2"]
    infos = _run(Harness(w, full=True, threads=16, chunk=1 << 22), w.steps)
    assert all(i["gpu"]["skipped"] == 0 for i in infos)
    assert all(i["oracle"]["coef"] < 1.0 for i in infos)   # clipping is active
    assert all(i["compared"][0] == 812_500_096 for i in infos)
