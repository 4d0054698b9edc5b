"""GPU parity of libzero against the CPU oracle (small and odd sizes).

Every case runs through the C ABI on seeded synthetic inputs and compares
with the oracle element by element: the reduced gradient, flags and the
skip/scale decision bit for bit, master/m/v within 1e-6 relative (bit-exact
when the clip coefficients agree), the norm within 1e-5, the fp16/bf16
parameters within 1 ulp, and gathers bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import zero_partitioned_mixed_flat_gb300 as Z
from zero_partitioned_mixed_flat_gb300 import synth
from zero_partitioned_mixed_flat_gb300.workloads import WORKLOADS, Workload

from .zstep import Harness, lp_ulp_dist, max_rel_err, plan_stats, same_floats

pytestmark = pytest.mark.gpu
TILE = 4096


def _plan(psi, n, lp, stage=1, align=8, sizes=None, units=None):
    return Z.ZeroPlan(psi if sizes is None else -1, n, sizes, align, stage, units, lp)


def _reduce_case(zlib, n, part, lp, scale, bucket=0, rank=0, seed=0, acc_lp=False):
    psi = n * part
    plan = _plan(psi, n, lp)
    assert plan.part_len == part
    if acc_lp:
        plan.set_reduce_precision(1)
    dev = torch.device("cuda")
    slices = [synth.grad_slice(part, lp, 1.0, scale, seed, 1, j, rank, dev) for j in range(n)]
    g = torch.empty(part, dtype=torch.float32, device=dev)
    plan.reduce(rank, slices, g, scale, bucket)
    ss, of, _ = plan_stats(plan)
    host = [synth.to_numpy_codes(t) for t in slices]
    og, oss, oof = (oracle.reduce_lp_accum if acc_lp else oracle.reduce)(host, lp, scale)
    assert same_floats(g.cpu().numpy(), og)
    assert of == oof
    assert abs(ss - oss) <= 1e-6 * oss
    plan.close()
    return g, ss


@pytest.mark.parametrize("n", [1, 2, 3, 5, 16, 17, 64, 65, 130, Z.ZERO_MAX_RANKS])
@pytest.mark.parametrize("lp", [0, 1])
def test_reduce_ragged_and_wide(zlib, n, lp):
    # 3 whole norm tiles plus a ragged tail of 136 elements
    _reduce_case(zlib, n, 3 * TILE + 136, lp, 1024.0 if lp == 0 else 1.0)


@pytest.mark.parametrize("n", [2, 3, 16, 64, 65])
@pytest.mark.parametrize("lp", [0, 1])
def test_reduce_in_lp_dtype(zlib, n, lp):
    # sums rounded to fp16/bf16 at every rank (reduce_dtype=float16)
    _reduce_case(zlib, n, 2 * TILE + 72, lp, 64.0 if lp == 0 else 1.0, acc_lp=True)


@pytest.mark.parametrize("part", [8, 64, 4096, TILE - 8, TILE, TILE + 8, 7 * TILE + 4000])
def test_reduce_sizes(zlib, part):
    _reduce_case(zlib, 4, part, 0, 4.0)


def test_bucket_size_never_changes_a_bit(zlib):
    n, part, lp = 8, 5 * TILE + 1000, 1
    ref = None
    for bucket in [0, 1, TILE, 2 * TILE + 3, 10 ** 9]:
        g, ss = _reduce_case(zlib, n, part, lp, 1.0, bucket=bucket)
        cur = (g.cpu().numpy(), ss)
        if ref is None:
            ref = cur
        else:
            assert same_floats(cur[0], ref[0]) and cur[1] == ref[1]


def test_empty_partition(zlib):
    plan = _plan(0, 4, 0)
    assert plan.part_len == 0
    dev = torch.device("cuda")
    e = torch.empty(0, dtype=torch.float16, device=dev)
    f = torch.empty(0, dtype=torch.float32, device=dev)
    plan.reduce(0, [e] * 4, f, 1.0)
    plan.adam(0, f, f, f, f, None, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, 1.0, 1.0)
    r = plan.result()
    assert r["norm"] == 0.0 and r["skipped"] == 0 and r["step"] == 1
    plan.close()


def _tiny(**kw):
    w = WORKLOADS["tiny-zero1"]
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


def test_tiny_zero1_all_partitions(zlib):
    h = Harness(WORKLOADS["tiny-zero1"])
    for _ in range(3):
        info = h.step()
        assert info["coef_equal"]
    h.close()


def test_ddp_replica_equals_sharded_step(zlib):
    # "ZeRO does not change the math": the stage-0 replica over the whole
    # buffer and the four stage-1 partitions give the same bits.
    w = WORKLOADS["tiny-zero1"]
    a = Harness(w)
    b = Harness(w, ranks=[0], stage=0)
    b.st[0].master.copy_(torch.cat([a.st[r].master for r in a.ranks]))
    # feed stage 0 the concatenation of the four partitions' slices
    for _ in range(3):
        a.step_no += 1
        for r in a.ranks:
            a.make_slices(r)
        ra = a.gpu_step()
        b.st[0].slices = [torch.cat([a.st[r].slices[j] for r in a.ranks]) for j in range(w.n_ranks)]
        rb = b.gpu_step()
        assert (ra["skipped"], ra["step"], ra["loss_scale"]) == (rb["skipped"], rb["step"], rb["loss_scale"])
        assert abs(ra["norm"] - rb["norm"]) <= 1e-12 * ra["norm"]
        full = lambda t: torch.cat([getattr(a.st[r], t) for r in a.ranks]).cpu().numpy()
        for t in ("master", "m", "v", "g"):
            assert same_floats(full(t), getattr(b.st[0], t).cpu().numpy()), t
        assert torch.equal(a.param, b.param)
    a.close()
    b.close()


@pytest.mark.parametrize("kw", [
    dict(adamw=False),                                     # L2 Adam
    dict(lp=1, loss_scale=1.0, grads_times_scale=False),   # bf16
    dict(clip=0.0),                                        # no clipping
    dict(clip=0.05),                                       # clipping active
    dict(n_ranks=3, ranks=[0, 1, 2], sizes=[100_000, 7, 33_333]),  # odd N, ragged
    dict(n_ranks=1, ranks=[0]),                            # N = 1: plain mixed-precision Adam
    dict(bucket_elems=40_000),                             # several buckets
    dict(reduce_lp_accum=True),                            # fp16 reduce dtype
    dict(reduce_lp_accum=True, lp=1, loss_scale=1.0, grads_times_scale=False),
    dict(growth_interval=2, steps=5),                      # the scale doubles every 2 good steps
    dict(growth_interval=3, inject_inf_step=2, steps=6),   # a skip restarts the good-step count
    dict(growth_interval=0, inject_inf_step=2, steps=3),   # static scale: a skip keeps it
])
def test_tiny_variants(zlib, kw):
    h = Harness(_tiny(**kw))
    scales = [h.step()["gpu"]["loss_scale"] for _ in range(kw.get("steps", 2))]
    h.close()
    if "growth_interval" in kw:   # the scale after each step (from 1024)
        expect = {2: [1024, 2048, 2048, 4096, 4096], 3: [1024, 512, 512, 512, 1024, 1024],
                  0: [1024, 1024, 1024]}[kw["growth_interval"]]
        assert scales == expect, scales


def test_all_ranks_of_a_maximal_plan_in_one_step(zlib):
    # N = ZERO_MAX_RANKS partitions reduced on one plan: one decision over all
    # 1024 partitions' partials, then every partition updated with it
    n, part, lr, b1, b2, eps, wd = Z.ZERO_MAX_RANKS, 16, 1e-3, 0.9, 0.999, 1e-8, 0.01
    dev = torch.device("cuda")
    plan = _plan(n * part, n, 0)
    assert plan.part_len == part
    big = synth.grad_slice(n * n * part, 0, 1e-2, 1.0, 5, 1, 0, 0, dev).view(n, n, part)
    base, row = big.data_ptr(), part * 2        # slice j of rank r: big[r, j]
    g = torch.empty((n, part), dtype=torch.float32, device=dev)
    w0 = synth.master_init(n * part, 0.02, 5, 0, dev).view(n, part)
    w, m, v = w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0)
    for r in range(n):
        plan.reduce(r, [base + (r * n + j) * row for j in range(n)], g[r], 1.0)
    for r in range(n):
        plan.adam(r, g[r], w[r], m[r], v[r], None, lr, b1, b2, eps, wd, 1, 1.0, 0.05)
    res = plan.result()
    host = synth.to_numpy_codes(big.reshape(-1)).reshape(n, n, part)
    og = np.empty((n, part), np.float32)
    ss = 0.0
    for r in range(n):
        og[r], r_ss, r_of = oracle.reduce(list(host[r]), 0, 1.0)
        ss += r_ss
        assert r_of == 0
    assert same_floats(g.cpu().numpy(), og)
    d = oracle.decide(ss, 0, np.float32(0.05), 1.0, 0, 0, 1000, np.float32(b1), np.float32(b2))
    assert abs(res["norm"] - d["norm"]) <= 1e-5 * d["norm"] and res["step"] == 1
    ow, om, ov = w0.cpu().numpy().reshape(-1).copy(), np.zeros(n * part, np.float32), np.zeros(n * part, np.float32)
    oracle.adam(og.reshape(-1), ow, om, ov, 0, d["coef"], d["skip"], np.float32(lr), np.float32(b1),
                np.float32(b2), np.float32(eps), np.float32(wd), 1, d["bc1"], d["bc2"])
    for got, exp in ((w, ow), (m, om), (v, ov)):
        assert max_rel_err(got.cpu().numpy().reshape(-1), exp) <= 1e-6
    plan.close()


@pytest.mark.parametrize("n,ranks,lp,bucket,stage", [
    (8, list(range(8)), 1, 0, 2),
    (8, [5, 2, 7], 0, 3 * TILE, 1),         # a subset, out of order, ragged bucket pieces
    (3, [0, 1, 2], 0, 0, 2),                # the few-slice reduce variant
    (70, list(range(70)), 1, 0, 2),         # > 64 slices: 14 partitions per launch; Adam in 2 launches
    (16, list(range(16)), 0, 5 * TILE + 8, 2),
    (4, [3, 0, 1], 1, 0, 3),                # stage 3: units, per-unit tiles, lp shards
    (1, [0], 0, 0, 0),                      # stage 0: the DDP replica
])
def test_many_partitions_in_one_call_equal_one_by_one(zlib, n, ranks, lp, bucket, stage):
    # zero_reduce_partitions / zero_adam_step_partitions against the same
    # per-partition calls: outputs, statistics, decision and state bit for bit
    dev = torch.device("cuda")
    if stage == 3:
        sizes, units = [70_000, 5, 33_000, 100_000, 7], [0, 0, 1, 2, 2]
        probe = _plan(-1, n, lp, stage=3, sizes=sizes, units=units)
    else:
        sizes, units = None, None
        probe = _plan(n * (2 * TILE + 8 * (n % 5 + 1)), n, lp, stage=stage)
    part = probe.part_len
    probe.close()
    scale = 64.0 if lp == 0 else 1.0
    sl = {r: [synth.grad_slice(part, lp, 1e-2, scale, 21, 1, j, r, dev) for j in range(n)] for r in ranks}
    w0 = {r: synth.master_init(part, 0.02, 21, r, dev) for r in ranks}
    hp = (1e-3, .9, .999, 1e-8, 0.01, 1, scale, 0.05)
    res = []
    for mode in ("one", "many"):
        if stage == 3:
            plan = _plan(-1, n, lp, stage=3, sizes=sizes, units=units)
        else:
            plan = _plan(n * part, n, lp, stage=stage)
        g = {r: torch.full((part,), float("nan"), device=dev) for r in ranks}
        w = {r: w0[r].clone() for r in ranks}
        m = {r: torch.zeros(part, device=dev) for r in ranks}
        v = {r: torch.zeros(part, device=dev) for r in ranks}
        if stage == 3:
            shard = {r: torch.zeros(part, dtype=synth.LP_DTYPES[lp], device=dev) for r in ranks}
            outs = [shard[r] for r in ranks]
            param = torch.cat([shard[r] for r in ranks])   # snapshot below
        else:
            param = torch.zeros(plan.psi_padded, dtype=synth.LP_DTYPES[lp], device=dev)
            outs = [param] * len(ranks)
        for step in range(2):
            if mode == "one":
                for r in ranks:
                    plan.reduce(r, sl[r], g[r], scale, bucket)
            else:
                plan.reduce_many(ranks, [sl[r] for r in ranks], [g[r] for r in ranks], scale, bucket)
            _, _, vec = plan_stats(plan)
            if mode == "one":
                for r, out in zip(ranks, outs):
                    plan.adam(r, g[r], w[r], m[r], v[r], out, *hp)
            else:
                plan.adam_many(ranks, [g[r] for r in ranks], [w[r] for r in ranks], [m[r] for r in ranks],
                               [v[r] for r in ranks], outs, *hp)
            if stage == 3:
                param = torch.cat([shard[r] for r in ranks])
            res.append((mode, step, plan.result(), vec, {r: (g[r].clone(), w[r].clone(), m[r].clone(),
                                                             v[r].clone()) for r in ranks}, param.clone()))
        plan.close()
    one, many = res[:2], res[2:]
    for a, b in zip(one, many):
        assert a[2] == b[2] and a[3].tobytes() == b[3].tobytes()
        for r in ranks:
            for x, y in zip(a[4][r], b[4][r]):
                assert torch.equal(x, y), r
        assert torch.equal(a[5], b[5])
    # and the reduced gradients are the oracle's
    og, _, _ = oracle.reduce([synth.to_numpy_codes(t) for t in sl[ranks[-1]]], lp, scale)
    assert same_floats(many[0][4][ranks[-1]][0].cpu().numpy(), og)


def test_many_partitions_validation(zlib):
    dev = torch.device("cuda")
    plan = _plan(4 * 64, 4, 0)
    buf = torch.zeros(64, dtype=torch.float16, device=dev)
    g = torch.zeros(64, device=dev)
    with pytest.raises(Z.ZeroError) as e:
        plan.reduce_many([1, 1], [[buf] * 4, [buf] * 4], [g, g], 1.0)
    assert e.value.code == Z.ZERO_EINVAL and "twice" in Z.zero_last_error()
    with pytest.raises(Z.ZeroError) as e:
        plan.reduce_many([0, 4], [[buf] * 4, [buf] * 4], [g, g], 1.0)
    assert e.value.code == Z.ZERO_EINVAL
    plan.reduce_many([0, 1], [[buf] * 4, [buf] * 4], [g, torch.zeros(64, device=dev)], 1.0)
    with pytest.raises(Z.ZeroError) as e:
        plan.adam_many([0, 0], [g, g], [g, g], [g, g], [g, g], [None, None], 1e-3, .9, .999, 1e-8,
                       0., 1, 1.0, 1.0)
    assert e.value.code == Z.ZERO_EINVAL
    plan.result()
    plan.close()


def test_all_ranks_of_a_maximal_plan_in_few_calls(zlib):
    # the 1024 partitions of a maximal plan through zero_reduce_partitions (one
    # partition per launch: 1024 slice pointers fill the table) and
    # zero_adam_step_partitions (16 launches of 64): the bits of the
    # per-partition calls
    n, part, lr, b1, b2, eps, wd = Z.ZERO_MAX_RANKS, 16, 1e-3, 0.9, 0.999, 1e-8, 0.01
    dev = torch.device("cuda")
    big = synth.grad_slice(n * n * part, 0, 1e-2, 1.0, 5, 1, 0, 0, dev).view(n, n, part)
    base, row = big.data_ptr(), part * 2
    w0 = synth.master_init(n * part, 0.02, 5, 0, dev).view(n, part)
    out = []
    for many in (False, True):
        plan = _plan(n * part, n, 0)
        g = torch.empty((n, part), dtype=torch.float32, device=dev)
        w, m, v = w0.clone(), torch.zeros_like(w0), torch.zeros_like(w0)
        param = torch.zeros(n * part, dtype=torch.float16, device=dev)
        sl = [[base + (r * n + j) * row for j in range(n)] for r in range(n)]
        hp = (lr, b1, b2, eps, wd, 1, 1.0, 0.05)
        if many:
            plan.reduce_many(list(range(n)), sl, [g[r] for r in range(n)], 1.0)
            plan.adam_many(list(range(n)), [g[r] for r in range(n)], [w[r] for r in range(n)],
                           [m[r] for r in range(n)], [v[r] for r in range(n)], [param] * n, *hp)
        else:
            for r in range(n):
                plan.reduce(r, sl[r], g[r], 1.0)
            for r in range(n):
                plan.adam(r, g[r], w[r], m[r], v[r], param, *hp)
        out.append((plan.result(), g.clone(), w.clone(), m.clone(), v.clone(), param.clone()))
        plan.close()
    assert out[0][0] == out[1][0]
    for a, b in zip(out[0][1:], out[1][1:]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("sub_group", [8, 40_000, 1 << 20])
def test_adam_in_sub_groups(zlib, sub_group):
    # the optimizer step taken a sub-group at a time (sub_group_size) against
    # the oracle, and bit for bit against the whole-partition call
    w = _tiny(n_ranks=3, ranks=[0, 1, 2], sizes=[100_000, 7, 33_333], clip=0.05)
    a = Harness(w, sub_group=sub_group)
    b = Harness(w)
    for _ in range(2):
        a.step()
        b.step()
        for r in a.ranks:
            for t in ("master", "m", "v"):
                assert torch.equal(getattr(a.st[r], t), getattr(b.st[r], t)), (r, t)
        assert torch.equal(a.param, b.param)
        assert a.plan.result() == b.plan.result()
    a.close()
    b.close()


@pytest.mark.parametrize("seed", range(12))
def test_random_layouts_full_step(zlib, seed):
    # random plans: N, stage, tensor list, stage-3 units, align, lp, buckets,
    # partitions updated; two whole steps against the oracle, every element
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.choice([1, 2, 3, 5, 8, 17, 64, 70]))
    stage = int(rng.integers(1, 4))
    k = int(rng.integers(1, 6))
    sizes = [int(x) for x in rng.integers(1, 50_000, k)]
    units = None
    if stage == 3:
        units, u = [], 0
        for i in range(k):
            if i > 0 and rng.random() < 0.5:
                u += 1
            units.append(u)
    lp = int(rng.integers(0, 2))
    ranks = sorted(set(int(r) for r in rng.integers(0, n, min(n, 3))))
    w = _tiny(n_ranks=n, ranks=ranks, sizes=sizes, unit_of_tensor=units, stage=stage, lp=lp,
              align=int(rng.choice([8, 128])), bucket_elems=int(rng.choice([0, 4096, 12_288])),
              loss_scale=1024.0 if lp == 0 else 1.0, grads_times_scale=lp == 0,
              clip=float(rng.choice([0.0, 0.05, 1.0])), adamw=bool(rng.integers(0, 2)))
    h = Harness(w)
    for _ in range(2):
        h.step()
    h.close()


def test_overflow_skips_and_halves_scale(zlib):
    w = _tiny(growth_interval=1000, inject_inf_step=2, loss_scale=65536.0, steps=3)
    h = Harness(w)
    seen = []
    for _ in range(3):
        info = h.step()
        seen.append((info["gpu"]["skipped"], info["gpu"]["loss_scale"], info["gpu"]["step"]))
    assert seen == [(0, 65536.0, 1), (1, 32768.0, 1), (0, 32768.0, 2)]
    h.close()


def test_nan_and_remote_terms(zlib):
    dev = torch.device("cuda")
    n, part = 2, 4096
    plan = _plan(n * part, n, 0)
    sl = [synth.grad_slice(part, 0, 1e-2, 1.0, 0, 1, j, 0, dev) for j in range(n)]
    g = torch.empty(part, device=dev)
    w = torch.zeros(part, device=dev); m = torch.zeros(part, device=dev); v = torch.zeros(part, device=dev)
    # remote overflow forces a skip even when this partition is finite
    plan.reduce(0, sl, g, 1.0)
    plan.adam(0, g, w, m, v, None, 1e-3, .9, .999, 1e-8, 0., 1, 1.0, 1.0, 0.0, 1)
    r = plan.result()
    assert r["skipped"] == 1 and r["step"] == 0 and not w.any().item()
    # remote sum of squares joins the global norm
    plan.reduce(0, sl, g, 1.0)
    ss, _, _ = plan_stats(plan)
    plan.adam(0, g, w, m, v, None, 1e-3, .9, .999, 1e-8, 0., 1, 1.0, 1.0, 3.0 * ss, 0)
    r = plan.result()
    assert abs(r["norm"] - np.sqrt(4.0 * ss)) <= 1e-6 * r["norm"] and r["step"] == 1
    # a NaN gradient is an overflow
    sl[1][17] = float("nan")
    plan.reduce(0, sl, g, 1.0)
    before = w.clone()
    plan.adam(0, g, w, m, v, None, 1e-3, .9, .999, 1e-8, 0., 1, 1.0, 1.0)
    r = plan.result()
    assert r["skipped"] == 1 and torch.equal(before, w)
    plan.close()


@pytest.mark.parametrize("skips", [0, 3, 9])
def test_bias_corrections_after_unread_skips(zlib, skips):
    # the decision takes 1 - beta^t from a host table around the counter the
    # host expects; skipped steps that were never read back move the device
    # counter off that guess (9 skips: outside the table, computed on the
    # device).  Every case must match the oracle's step at t = 501.
    dev = torch.device("cuda")
    n, part, b1, b2 = 2, 2 * TILE + 40, 0.9, 0.999
    plan = _plan(n * part, n, 0)
    plan.set_state(500)
    sl = [synth.grad_slice(part, 0, 1e-2, 1.0, 4, 1, j, 0, dev) for j in range(n)]
    g = torch.empty(part, device=dev)
    w0 = synth.master_init(part, 0.02, 4, 0, dev)
    w, m, v = w0.clone(), torch.full((part,), 1e-3, device=dev), torch.full((part,), 1e-6, device=dev)
    m0, v0 = m.cpu().numpy().copy(), v.cpu().numpy().copy()
    for _ in range(skips):   # remote overflow: skipped, counter unchanged, nothing read back
        plan.reduce(0, sl, g, 1.0)
        plan.adam(0, g, w, m, v, None, 1e-3, b1, b2, 1e-8, 0.01, 1, 1.0, 1.0, 0.0, 1)
    plan.reduce(0, sl, g, 1.0)
    plan.adam(0, g, w, m, v, None, 1e-3, b1, b2, 1e-8, 0.01, 1, 1.0, 1.0)
    r = plan.result()
    assert r["step"] == 501 and r["skipped"] == 0
    host = [synth.to_numpy_codes(t) for t in sl]
    og, oss, oof = oracle.reduce(host, 0, 1.0)
    d = oracle.decide(oss, oof, 1.0, 1.0, 500, 0, 0, np.float32(b1), np.float32(b2))
    ow, om, ov = w0.cpu().numpy().copy(), m0, v0
    oracle.adam(og, ow, om, ov, 0, d["coef"], d["skip"], np.float32(1e-3), np.float32(b1),
                np.float32(b2), np.float32(1e-8), np.float32(0.01), 1, d["bc1"], d["bc2"])
    for got, exp in ((w, ow), (m, om), (v, ov)):
        assert max_rel_err(got.cpu().numpy(), exp) <= 1e-6
    plan.close()


@pytest.mark.parametrize("steps", [3, 10])
def test_captured_step_replays_like_eager_steps(zlib, steps):
    # one step (reduce of every partition, decision, Adam) captured into a CUDA
    # graph after an eager first step, replayed `steps` times, against the same
    # number of eager steps; 10 replays run past the bias-correction table
    # baked into the captured launch (the device then computes the powers)
    w = _tiny(n_ranks=3, ranks=[0, 1, 2], sizes=[100_000, 7, 33_333], clip=0.05)
    a, b = Harness(w), Harness(w)
    for h in (a, b):
        h.step_no = 1
        for r in h.ranks:
            h.make_slices(r)
        h.gpu_step()
    for _ in range(steps):
        a.gpu_step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for r in b.ranks:
                s = b.st[r]
                b.plan.reduce(r, s.slices, s.g, b.S, b.bucket, stream=int(cap.cuda_stream))
            for r in b.ranks:
                s = b.st[r]
                b.plan.adam(r, s.g, s.master, s.m, s.v, b.param, w.lr, w.beta1, w.beta2, w.eps,
                            w.wd, int(w.adamw), b.S, w.clip, stream=int(cap.cuda_stream))
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(steps):
        g.replay()
    torch.cuda.synchronize()
    ra, rb = a.plan.result(), b.plan.result()
    assert ra == rb and rb["step"] == 1 + steps
    for r in a.ranks:
        for t in ("master", "m", "v"):
            assert torch.equal(getattr(a.st[r], t), getattr(b.st[r], t)), (r, t)
    assert torch.equal(a.param, b.param)
    a.close()
    b.close()


def test_resume_is_bit_identical(zlib):
    w = WORKLOADS["tiny-zero1"]
    a = Harness(w)
    for _ in range(3):
        a.step()
    # replay: two steps, checkpoint (state + step counter), fresh plan, step 3
    b = Harness(w)
    b.step()
    b.step()
    ck = {r: (b.st[r].master.clone(), b.st[r].m.clone(), b.st[r].v.clone()) for r in b.ranks}
    step, S = b.o_step, b.S
    b.close()
    c = Harness(w)
    c.plan.set_state(step, 0)
    for r in c.ranks:
        c.st[r].master.copy_(ck[r][0]); c.st[r].m.copy_(ck[r][1]); c.st[r].v.copy_(ck[r][2])
    c.step_no, c.S = 3, S
    for r in c.ranks:
        c.make_slices(r)
    res = c.gpu_step()
    assert res["step"] == 3
    for r in c.ranks:
        for t in ("master", "m", "v"):
            assert torch.equal(getattr(c.st[r], t), getattr(a.st[r], t))
    a.close()
    c.close()


# ------------------------------------------------------------------ gather

def _gather_case(n, sizes, units, lp=0, align=8, spin=None):
    dev = torch.device("cuda")
    plan = _plan(-1, n, lp, stage=3, align=align, sizes=sizes, units=units)
    shards = [synth.lp_shard(plan.part_len, lp, 1.0, 3, j, dev) for j in range(n)]
    host = [synth.to_numpy_codes(s) for s in shards]
    if spin is not None:
        plan.set_spin_limit(spin)
    outs = []
    for u in range(plan.n_units):
        sl = plan.shard_len(u)
        off = plan.unit_shard_offset(u)
        out = torch.full((sl * n,), 7, dtype=synth.LP_DTYPES[lp], device=dev)
        plan.gather(u, shards, out)
        outs.append((u, out, [h[off:off + sl] for h in host]))
    return plan, outs


@pytest.mark.parametrize("n", [1, 2, 3, 64, 65, Z.ZERO_MAX_RANKS])
def test_gather_units(zlib, n):
    sizes = [1000, 24, 4096 * 9 + 8, 5, 16384 * 3, 100_000]
    units = [0, 0, 1, 2, 2, 3]
    plan, outs = _gather_case(n, sizes, units)
    plan.check()
    for u, out, host in outs:
        assert np.array_equal(synth.to_numpy_codes(out), oracle.gather(host)), u
    plan.close()


def test_gather_large_unit_many_chunks(zlib):
    plan, outs = _gather_case(8, [3_000_000, 1_000_008], [0, 1], lp=1, align=128)
    plan.check()
    for u, out, host in outs:
        assert np.array_equal(synth.to_numpy_codes(out), oracle.gather(host)), u
    plan.close()


def test_gather_wait_timeout_is_reported_and_recoverable(zlib):
    # spin limit 0: every bounded wait gives up at once; the kernel drains its
    # copies, sets the error word and returns; the context stays usable
    plan, outs = _gather_case(4, [200_000], None, spin=0)
    with pytest.raises(Z.ZeroError) as e:
        plan.check()
    assert e.value.code == Z.ZERO_ETIMEOUT
    plan.check()   # the error word was cleared
    plan.close()
    plan2, outs2 = _gather_case(4, [200_000], None)
    plan2.check()
    u, out, host = outs2[0]
    assert np.array_equal(synth.to_numpy_codes(out), oracle.gather(host))
    plan2.close()


@pytest.mark.parametrize("part", [40_000, 4_000_000])
def test_adam_wait_timeout_is_reported_and_recoverable(zlib, part):
    # spin limit 0: every pipeline wait of the Adam kernel gives up at once.
    # 40,000 elements: one tile per CTA (the producer issues everything, then
    # drains); 4M: ~13 tiles per CTA (the producer's own wait gives up after
    # four tiles, then it drains).  No tile may be stored: master, m, v and
    # the lp param keep their old values; the error word reports ZERO_ETIMEOUT
    # and is cleared; the same plan then redoes the step (counter restored)
    # and matches the oracle.
    dev = torch.device("cuda")
    n, rank, lp, lr, b1, b2, eps, wd, clip = 3, 1, 0, 1e-3, 0.9, 0.999, 1e-8, 0.01, 0.05
    plan = _plan(n * part, n, lp, stage=2)
    assert plan.part_len == part
    sl = [synth.grad_slice(part, lp, 1e-2, 64.0, 8, 1, j, rank, dev) for j in range(n)]
    g = torch.empty(part, device=dev)
    w0 = synth.master_init(part, 0.02, 8, rank, dev)
    m0 = torch.full((part,), 1e-3, device=dev)
    v0 = torch.full((part,), 1e-6, device=dev)
    w, m, v = w0.clone(), m0.clone(), v0.clone()
    param = torch.full((n * part,), 7.0, dtype=torch.float16, device=dev)
    hp = (lr, b1, b2, eps, wd, 1, 64.0, clip)
    plan.reduce(rank, sl, g, 64.0)
    plan.set_spin_limit(0)
    plan.adam(rank, g, w, m, v, param, *hp)
    with pytest.raises(Z.ZeroError) as e:
        plan.result()
    assert e.value.code == Z.ZERO_ETIMEOUT
    plan.check()   # the error word was cleared
    assert torch.equal(w, w0) and torch.equal(m, m0) and torch.equal(v, v0)
    assert bool((param == 7.0).all())
    # redo the step on the same plan and context
    plan.set_state(0, 0)
    plan.set_spin_limit(1 << 22)
    plan.reduce(rank, sl, g, 64.0)
    plan.adam(rank, g, w, m, v, param, *hp)
    r = plan.result()
    og, oss, oof = oracle.reduce([synth.to_numpy_codes(t) for t in sl], lp, 64.0)
    assert same_floats(g.cpu().numpy(), og)
    d = oracle.decide(oss, oof, np.float32(clip), 64.0, 0, 0, 1000, np.float32(b1), np.float32(b2))
    assert r["step"] == d["step"] == 1 and r["skipped"] == 0
    assert abs(r["norm"] - d["norm"]) <= 1e-5 * d["norm"]
    ow, om, ov = w0.cpu().numpy().copy(), m0.cpu().numpy().copy(), v0.cpu().numpy().copy()
    op = oracle.adam(og, ow, om, ov, lp, d["coef"], d["skip"], np.float32(lr), np.float32(b1),
                     np.float32(b2), np.float32(eps), np.float32(wd), 1, d["bc1"], d["bc2"])
    for got, exp in ((w, ow), (m, om), (v, ov)):
        assert max_rel_err(got.cpu().numpy(), exp) <= 1e-6
    assert lp_ulp_dist(synth.to_numpy_codes(param[rank * part:(rank + 1) * part]), op) <= 1
    plan.close()


def test_synchronising_calls_wait_only_for_the_plan(zlib):
    # zero_step_result, zero_plan_check and zero_plan_set_state wait for the
    # plan's own work, not for a long kernel on an unrelated stream
    import time
    dev = torch.device("cuda")
    n, part = 2, 2 * TILE
    plan = _plan(n * part, n, 0)
    sl = [synth.grad_slice(part, 0, 1e-2, 1.0, 9, 1, j, 0, dev) for j in range(n)]
    g = torch.empty(part, device=dev)
    w, m, v = (torch.zeros(part, device=dev) for _ in range(3))
    mine, other = torch.cuda.Stream(), torch.cuda.Stream()
    hp = (1e-3, .9, .999, 1e-8, 0., 1, 1.0, 1.0)
    plan.reduce(0, sl, g, 1.0, stream=mine)          # warm: scratch, modules
    plan.adam(0, g, w, m, v, None, *hp, stream=mine)
    plan.result()
    torch.cuda.synchronize()
    done = torch.cuda.Event()
    with torch.cuda.stream(other):
        torch.cuda._sleep(int(3e9))                  # about 1.5 s of spinning
        done.record(other)
    t0 = time.perf_counter()
    plan.reduce(0, sl, g, 1.0, stream=mine)
    plan.adam(0, g, w, m, v, None, *hp, stream=mine)
    r = plan.result()
    plan.check()
    plan.set_state(r["step"], 0)
    el = time.perf_counter() - t0
    still_running = not done.query()
    torch.cuda.synchronize()
    assert done.query()
    assert r["step"] == 2
    assert still_running, "a synchronising call waited for another stream's kernel (%.3f s)" % el
    plan.close()


def test_plans_on_host_threads_are_independent(zlib):
    # different plans are independent: three plans stepped at once from three
    # host threads, each on its own stream (ctypes releases the GIL inside
    # every call), end bit-identical to one plan stepped alone, decision by
    # decision; one of the threads overflows on its second step and must be
    # the only one that skips
    import threading
    dev = torch.device("cuda")
    n, part, steps, rank = 4, 3 * TILE + 40, 3, 1
    hp = (1e-3, .9, .999, 1e-8, 0.01, 1, 1024.0, 0.05)

    def inputs(inject):
        sl = [[synth.grad_slice(part, 0, 1e-3, 1024.0, 5, s + 1, j, rank, dev) for j in range(n)]
              for s in range(steps)]
        if inject:
            sl[1][2][77] = float("inf")
        return sl

    def state():
        return dict(g=torch.empty(part, device=dev), w=synth.master_init(part, 0.02, 5, rank, dev),
                    m=torch.zeros(part, device=dev), v=torch.zeros(part, device=dev),
                    p=torch.zeros(n * part, dtype=torch.float16, device=dev))

    def run(plan, sl, st, stream, out, errors):
        try:
            scale = hp[6]
            dec = []
            for s in range(steps):
                plan.reduce(rank, sl[s], st["g"], scale, stream=stream)
                plan.adam(rank, st["g"], st["w"], st["m"], st["v"], st["p"], *hp[:6], scale, hp[7],
                          stream=stream)
                r = plan.result()
                dec.append(r)
                scale = r["loss_scale"]
            out.extend(dec)
        except Exception as e:  # reported on the main thread
            errors.append(e)

    cases = [False, True, False]          # the second thread's plan overflows
    plans = [_plan(n * part, n, 0, stage=2) for _ in cases]
    sls = [inputs(inj) for inj in cases]
    sts = [state() for _ in cases]
    streams = [torch.cuda.Stream() for _ in cases]
    outs = [[] for _ in cases]
    errors = []
    torch.cuda.synchronize()
    threads = [threading.Thread(target=run, args=(plans[i], sls[i], sts[i], streams[i], outs[i], errors))
               for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for inj in (False, True):             # the same step alone, one plan, one thread
        ref_plan, ref_st, ref_out, ref_err = _plan(n * part, n, 0, stage=2), state(), [], []
        run(ref_plan, inputs(inj), ref_st, torch.cuda.current_stream(), ref_out, ref_err)
        assert not ref_err, ref_err
        torch.cuda.synchronize()
        for i, c in enumerate(cases):
            if c != inj:
                continue
            assert [d["skipped"] for d in outs[i]] == ([0, 1, 0] if inj else [0, 0, 0])
            for a, b in zip(outs[i], ref_out):
                assert np.float64(a["norm"]).tobytes() == np.float64(b["norm"]).tobytes()
                assert {k: a[k] for k in a if k != "norm"} == {k: b[k] for k in b if k != "norm"}
            for k in ("w", "m", "v", "p"):
                assert torch.equal(sts[i][k].view(torch.int32 if k != "p" else torch.int16),
                                   ref_st[k].view(torch.int32 if k != "p" else torch.int16)), (i, k)
        ref_plan.close()
    # the steps did update the state
    assert not torch.equal(sts[0]["w"], synth.master_init(part, 0.02, 5, rank, dev))
    for p in plans:
        p.close()


@pytest.mark.parametrize("n,lp,bucket", [(2, 0, 0), (3, 1, 4096), (8, 0, 1000), (64, 1, 200_000),
                                         (5, 0, 8)])
def test_allgather_params_buckets(zlib, n, lp, bucket):
    # stage-1/2 step-end all-gather of the updated partitions into the full
    # layout, in buckets (allgather_bucket_size): a concatenation, bit for bit
    dev = torch.device("cuda")
    P = 2 * TILE + 8 * (n + 1)
    plan = _plan(n * P, n, lp, stage=2)
    assert plan.part_len == P
    parts = [synth.lp_shard(P, lp, 0.02, 6, j, dev) for j in range(n)]
    out = torch.full((n * P,), 7, dtype=synth.LP_DTYPES[lp], device=dev)
    plan.allgather(parts, out, bucket)
    plan.check()
    exp = oracle.gather([synth.to_numpy_codes(t) for t in parts])
    assert np.array_equal(synth.to_numpy_codes(out), exp)
    # in place: each rank's source is its own range of the output
    full = torch.full((n * P,), 5, dtype=synth.LP_DTYPES[lp], device=dev)
    full[:P].copy_(parts[0])
    plan.allgather([full[:P]] + parts[1:], full, bucket)
    plan.check()
    assert np.array_equal(synth.to_numpy_codes(full), exp)
    plan.close()


def test_global_stats_replace_the_local_sum(zlib):
    # multi-rank use: an all-reduced statistics vector decides the step.  One
    # process reducing all four partitions (identical slices) and one that
    # reduced only partition 0 but is handed the vector of all four take the
    # same decision, bit for bit.
    dev = torch.device("cuda")
    n, part = 4, 3 * TILE + 40
    sl = [synth.grad_slice(part, 1, 1e-3, 1.0, 0, 1, j, 0, dev) for j in range(n)]
    hp = (1e-3, .9, .999, 1e-8, 0., 1, 1.0, 0.05)

    def fresh():
        z = lambda: torch.zeros(part, device=dev)
        return torch.empty(part, device=dev), z(), z(), z()

    full = _plan(n * part, n, 1)
    gs = [fresh() for _ in range(n)]
    for r in range(n):
        full.reduce(r, sl, gs[r][0], 1.0)
    _, _, vec_all = plan_stats(full)
    for r in range(n):
        full.adam(r, *gs[r], None, *hp)
    ref = full.result()
    one = _plan(n * part, n, 1)
    g, w, m, v = fresh()
    one.reduce(0, sl, g, 1.0)
    _, _, vec0 = plan_stats(one)
    assert vec0[0] == vec_all[0] and not vec0[1:].any()     # only partition 0, exact zeros elsewhere
    assert np.array_equal(vec_all[:n], np.full(n, vec_all[0]))
    stats = torch.from_numpy(vec_all.copy()).to(dev)
    one.set_global_stats(stats)
    one.adam(0, g, w, m, v, None, *hp, 123.0, 1)               # remote terms are ignored
    r1 = one.result()
    assert r1 == ref, (r1, ref)
    assert torch.equal(w, gs[0][1]) and torch.equal(m, gs[0][2]) and torch.equal(v, gs[0][3])
    # the vector's sums match the oracle's
    _, oss, _ = oracle.reduce([synth.to_numpy_codes(t) for t in sl], 1, 1.0)
    assert abs(vec_all[0] - oss) <= 1e-9 * oss
    # an overflow flag of another partition skips this rank's step
    one.reduce(0, sl, g, 1.0)
    flagged = stats.clone()
    flagged[n + 2] = 1.0
    one.set_global_stats(flagged)
    before = w.clone()
    one.adam(0, g, w, m, v, None, *hp)
    r2 = one.result()
    assert r2["skipped"] == 1 and torch.equal(before, w)
    # out of order: after the decision the step's stats are fixed
    with pytest.raises(Z.ZeroError) as e:
        one.set_global_stats(stats)
    assert e.value.code == Z.ZERO_ESTATE
    with pytest.raises(Z.ZeroError) as e:
        one.partition_stats(stats)
    assert e.value.code == Z.ZERO_ESTATE
    full.close()
    one.close()


def test_exported_flags_name_the_overflowing_partition(zlib):
    # three partitions reduced in one process, an inf in partition 1's slices:
    # the export flags exactly that partition, its sum is not finite, the other
    # sums are the oracle's; deciding from the vector skips the step
    dev = torch.device("cuda")
    n, part = 3, TILE + 8
    plan = _plan(n * part, n, 0, stage=2)
    sl = {r: [synth.grad_slice(part, 0, 1e-2, 64.0, 41, 1, j, r, dev) for j in range(n)] for r in range(n)}
    sl[1][2][TILE - 3] = float("inf")
    g = {r: torch.empty(part, device=dev) for r in range(n)}
    for r in range(n):
        plan.reduce(r, sl[r], g[r], 64.0)
    _, _, vec = plan_stats(plan)
    assert list(vec[n:]) == [0.0, 1.0, 0.0]
    assert not np.isfinite(vec[1])
    for r in (0, 2):
        _, oss, oof = oracle.reduce([synth.to_numpy_codes(t) for t in sl[r]], 0, 64.0)
        assert oof == 0 and abs(vec[r] - oss) <= 1e-9 * oss
    stats = torch.from_numpy(vec.copy()).to(dev)
    plan.set_global_stats(stats)
    w = torch.zeros(part, device=dev)
    m, v = torch.zeros_like(w), torch.zeros_like(w)
    plan.adam(0, g[0], w, m, v, None, 1e-3, .9, .999, 1e-8, 0., 1, 64.0, 1.0)
    r = plan.result()
    assert r["skipped"] == 1 and r["step"] == 0 and not w.any().item()
    plan.close()


def test_stats_vector_in_pinned_host_memory(zlib):
    # the statistics vector may live in pinned host memory (e.g. a gloo
    # exchange buffer): exported and read back by the kernels in place
    dev = torch.device("cuda")
    n, part = 3, 2 * TILE + 24
    res = []
    for where in ("device", "host"):
        plan = _plan(n * part, n, 0, stage=2)
        sl = [synth.grad_slice(part, 0, 1e-2, 64.0, 31, 1, j, 1, dev) for j in range(n)]
        g = torch.empty(part, device=dev)
        w, m, v = (torch.zeros(part, device=dev) for _ in range(3))
        plan.reduce(1, sl, g, 64.0)
        stats = (torch.full((2 * n,), float("nan"), dtype=torch.float64, device=dev) if where == "device"
                 else torch.full((2 * n,), float("nan"), dtype=torch.float64, pin_memory=True))
        plan.partition_stats(stats)
        torch.cuda.synchronize()
        vec = stats.cpu().numpy().copy()
        assert vec[0] == 0.0 and vec[2] == 0.0 and vec[1] > 0 and not vec[n:].any()
        plan.set_global_stats(stats)
        plan.adam(1, g, w, m, v, None, 1e-3, .9, .999, 1e-8, 0., 1, 64.0, 0.05)
        res.append((plan.result(), vec, w.clone()))
        plan.close()
    assert res[0][0] == res[1][0] and res[0][1].tobytes() == res[1][1].tobytes()
    assert torch.equal(res[0][2], res[1][2])


def test_exported_stats_decide_like_the_local_sum(zlib):
    # every partition of a ragged random plan reduced in one process: deciding
    # from the exported vector gives the local decision's bits (norm included)
    dev = torch.device("cuda")
    rng = np.random.default_rng(77)
    for n, sizes in [(3, [100_000, 7, 33_333]), (17, [int(x) for x in rng.integers(1, 90_000, 6)])]:
        res = []
        for mode in ("local", "global"):
            plan = _plan(-1, n, 0, stage=2, sizes=sizes)
            P = plan.part_len
            g = torch.empty((n, P), device=dev)
            w = synth.master_init(n * P, 0.02, 3, 0, dev).view(n, P)
            m, v = torch.zeros_like(w), torch.zeros_like(w)
            for r in range(n):
                sl = [synth.grad_slice(P, 0, 1e-2, 64.0, 3, 1, j, r, dev) for j in range(n)]
                plan.reduce(r, sl, g[r], 64.0)
            if mode == "global":
                stats = torch.empty(2 * n, dtype=torch.float64, device=dev)
                plan.partition_stats(stats)
                plan.set_global_stats(stats)
            for r in range(n):
                plan.adam(r, g[r], w[r], m[r], v[r], None, 1e-3, .9, .999, 1e-8, 0.01, 1, 64.0, 0.05)
            res.append((plan.result(), w.clone(), m.clone(), v.clone()))
            plan.close()
        assert res[0][0] == res[1][0]
        for a, b in zip(res[0][1:], res[1][1:]):
            assert torch.equal(a, b)


# ------------------------------------------------------ quantized gather

def _quant_fns(fmt):
    """The oracle's quantizer and dequantizing gather for a code format."""
    if fmt == Z.ZERO_QUANT_FP8_E4M3:
        return oracle.quantize_blocks_fp8, oracle.dequant_gather_fp8, np.uint8
    return oracle.quantize_blocks, oracle.dequant_gather, np.int8


def _quant_case(n, sizes, units, lp, fmt=0):
    dev = torch.device("cuda")
    plan = _plan(-1, n, lp, stage=3, align=128, sizes=sizes, units=units)
    plan.set_gather_quantization(fmt)
    o_quant, o_dequant, code_t = _quant_fns(fmt)
    P = plan.part_len
    shards = [synth.lp_shard(P, lp, 0.02, 5, j, dev) for j in range(n)]
    shards[0][:256].zero_()                       # whole zero blocks: scale 0
    codes = [torch.empty(P, dtype=torch.int8, device=dev) for _ in range(n)]
    scales = [torch.empty(P // 128, dtype=torch.float32, device=dev) for _ in range(n)]
    for j in range(n):
        plan.quantize(shards[j], codes[j], scales[j])
    torch.cuda.synchronize()
    host_q = []
    for j in range(n):
        oq, osc = o_quant(synth.to_numpy_codes(shards[j]), lp, 128)
        assert np.array_equal(codes[j].cpu().numpy().view(code_t), oq), j
        assert np.array_equal(scales[j].cpu().numpy().view(np.uint32), osc.view(np.uint32)), j
        host_q.append((oq, osc))
    for u in range(plan.n_units):
        sl, off = plan.shard_len(u), plan.unit_shard_offset(u)
        out = torch.full((sl * n,), 3, dtype=synth.LP_DTYPES[lp], device=dev)
        plan.gather_quantized(u, codes, scales, out)
        exp = o_dequant([q[off:off + sl] for q, _ in host_q],
                        [c[off // 128:(off + sl) // 128] for _, c in host_q], lp, 128)
        assert np.array_equal(synth.to_numpy_codes(out), exp), u
    plan.close()


@pytest.mark.parametrize("n", [2, 3, 64, 65, Z.ZERO_MAX_RANKS])
@pytest.mark.parametrize("lp", [0, 1])
@pytest.mark.parametrize("fmt", [Z.ZERO_QUANT_INT8, Z.ZERO_QUANT_FP8_E4M3])
def test_quantize_and_dequant_gather(zlib, n, lp, fmt):
    _quant_case(n, [5000, 128, 40_000, 3, 70_000], [0, 0, 1, 2, 2], lp, fmt)


def _boundary_blocks(lp, rng, n_blocks):
    """lp codes of n_blocks 128-element blocks whose quotients x / scale sit on
    or next to half-integers (ties to even and both neighbours), with block
    maxima from tiny to huge (bf16) so that every scale range is exercised."""
    out = np.empty((n_blocks, 128), np.uint16)
    big = 60000.0 if lp == 0 else 1e36
    tiny = 1e-4 if lp == 0 else 1e-36
    for b in range(n_blocks):
        kind = b % 4
        if kind == 0:
            amax = np.float32(127.0)                 # scale exactly 1
        elif kind == 1:
            amax = np.float32(10.0 ** rng.uniform(-3, 3))
        elif kind == 2:
            amax = np.float32(big * rng.uniform(0.5, 1.0))
        else:
            amax = np.float32(tiny * rng.uniform(1.0, 2.0))
        amax_c = oracle.float_to_lp(np.array([amax], np.float32), lp)[0]
        amax = oracle.lp_to_float(np.array([amax_c], np.uint16), lp)[0]
        scale = np.float32(amax / np.float32(127.0))
        k = rng.integers(-127, 127, 127).astype(np.float32) + np.float32(0.5)
        x = oracle.float_to_lp((k * scale).astype(np.float32), lp).astype(np.int32)
        x += rng.integers(-1, 2, 127)                # the tie's code or a neighbour
        x = np.clip(x, 0, 0xFFFF).astype(np.uint16)
        xf = oracle.lp_to_float(x, lp)
        x[~(np.abs(xf) <= amax)] = amax_c           # keep |x| <= amax (and finite)
        out[b, 0] = amax_c
        out[b, 1:] = x
    return out.reshape(-1)


@pytest.mark.parametrize("lp", [0, 1])
def test_quantize_rounding_boundaries(zlib, lp):
    # quotients on and next to half-integers: the codes must be those of the
    # correctly rounded quotient, ties to even
    rng = np.random.default_rng(11 + lp)
    n = 2
    plan = _plan(-1, n, lp, stage=3, align=128, sizes=[n * 128 * 256], units=[0])
    P = plan.part_len
    dev = torch.device("cuda")
    for j in range(n):
        host = _boundary_blocks(lp, rng, P // 128)
        shard = torch.from_numpy(host.view(np.int16)).to(dev).view(synth.LP_DTYPES[lp])
        codes = torch.empty(P, dtype=torch.int8, device=dev)
        scales = torch.empty(P // 128, dtype=torch.float32, device=dev)
        plan.quantize(shard, codes, scales)
        torch.cuda.synchronize()
        oq, osc = oracle.quantize_blocks(host, lp, 128)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), osc.view(np.uint32))
        assert np.array_equal(codes.cpu().numpy(), oq)
    plan.close()


def _fp8_boundary_blocks(lp, rng, n_blocks):
    """lp codes of blocks whose scaled values sit on E4M3 rounding ties (and
    their lp neighbours), subnormal E4M3 codes, and block maxima spanning
    the lp range (bf16 down to float-subnormal blocks: the clamped scale)."""
    c = np.arange(0x7f, dtype=np.uint8)
    vals = oracle.e4m3_decode(c).astype(np.float64)
    mids = (vals[1:] + vals[:-1]) / 2                         # every tie of the format
    out = np.empty((n_blocks, 128), np.uint16)
    lo, hi = (-15, 7) if lp == 0 else (-132, 120)
    for b in range(n_blocks):
        e = int(rng.integers(lo, hi + 1))
        amax = float(rng.uniform(128, 256))
        m = rng.choice(mids[mids < amax], 127) * rng.choice([-1.0, 1.0], 127)
        x = np.concatenate([[amax], m]) * 2.0 ** e
        codes = oracle.float_to_lp(x.astype(np.float32), lp).astype(np.int32)
        codes[1:] += rng.integers(-1, 2, 127)                  # ties and their neighbours
        codes = np.clip(codes, 0, 0xffff).astype(np.uint16)
        xf = oracle.lp_to_float(codes, lp)
        bad = ~np.isfinite(xf) | (np.abs(xf) > np.abs(xf[0]))
        codes[bad] = codes[0]
        out[b] = codes
    return out.reshape(-1)


@pytest.mark.parametrize("lp", [0, 1])
def test_quantize_fp8_rounding_boundaries(zlib, lp):
    rng = np.random.default_rng(41 + lp)
    n = 2
    plan = _plan(-1, n, lp, stage=3, align=128, sizes=[n * 128 * 256], units=[0])
    plan.set_gather_quantization(Z.ZERO_QUANT_FP8_E4M3)
    P = plan.part_len
    dev = torch.device("cuda")
    for j in range(n):
        host = _fp8_boundary_blocks(lp, rng, P // 128)
        shard = torch.from_numpy(host.view(np.int16)).to(dev).view(synth.LP_DTYPES[lp])
        codes = torch.empty(P, dtype=torch.int8, device=dev)
        scales = torch.empty(P // 128, dtype=torch.float32, device=dev)
        plan.quantize(shard, codes, scales)
        torch.cuda.synchronize()
        oq, osc = oracle.quantize_blocks_fp8(host, lp, 128)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), osc.view(np.uint32))
        assert np.array_equal(codes.cpu().numpy().view(np.uint8), oq)
    plan.close()


@pytest.mark.parametrize("lp", [0, 1])
@pytest.mark.parametrize("fmt", [Z.ZERO_QUANT_INT8, Z.ZERO_QUANT_FP8_E4M3])
def test_quantize_every_block_maximum(zlib, lp, fmt):
    # every positive finite lp value as the maximum |x| of a block (the block
    # scale depends on it alone): scales and codes bit for bit against the
    # oracle, so the quantizer's scale arithmetic is checked on its whole domain
    rng = np.random.default_rng(70 + lp)
    top = 0x7BFF if lp == 0 else 0x7F7F                  # the largest finite value
    amax = np.arange(1, top + 1, dtype=np.uint16)
    n_blocks = amax.size + 1                               # plus one all-zero block
    n_blocks += (-n_blocks) % 2
    blocks = np.zeros((n_blocks, 128), np.uint16)
    blocks[:amax.size, 0] = amax
    amax_f = oracle.lp_to_float(amax, lp)
    frac = rng.uniform(-1.0, 1.0, (amax.size, 127)).astype(np.float32)
    x = oracle.float_to_lp((frac * amax_f[:, None]).astype(np.float32), lp)
    xf = oracle.lp_to_float(x, lp)
    x[~(np.abs(xf) <= amax_f[:, None])] = 0                # |x| <= amax after rounding
    blocks[:amax.size, 1:] = x
    host = blocks.reshape(-1)
    n = 2
    plan = _plan(-1, n, lp, stage=3, align=128, sizes=[n * host.size], units=[0])
    plan.set_gather_quantization(fmt)
    P = plan.part_len
    assert P == host.size
    dev = torch.device("cuda")
    shard = torch.from_numpy(host.view(np.int16)).to(dev).view(synth.LP_DTYPES[lp])
    codes = torch.empty(P, dtype=torch.int8, device=dev)
    scales = torch.empty(P // 128, dtype=torch.float32, device=dev)
    plan.quantize(shard, codes, scales)
    torch.cuda.synchronize()
    o_quant, _, code_t = _quant_fns(fmt)
    oq, osc = o_quant(host, lp, 128)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), osc.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy().view(code_t), oq.view(code_t))
    plan.close()


def test_quantized_gather_rejects_small_align(zlib):
    plan = _plan(-1, 2, 0, stage=3, align=8, sizes=[64, 64], units=[0, 1])
    buf = torch.zeros(1024, dtype=torch.float16, device="cuda")
    q = torch.zeros(1024, dtype=torch.int8, device="cuda")
    sc = torch.zeros(8, dtype=torch.float32, device="cuda")
    with pytest.raises(Z.ZeroError) as e:
        plan.quantize(buf, q, sc)
    assert e.value.code == Z.ZERO_EINVAL
    plan.close()


@pytest.mark.parametrize("lp", [0, 1])
def test_reduce_reads_pinned_host_slices(zlib, lp):
    # the slices may stay in pinned host memory: the kernel reads them in place
    n, part = 8, 3 * TILE + 64
    dev = torch.device("cuda")
    dslices = [synth.grad_slice(part, lp, 1e-3, 1.0, 3, 1, j, 0, dev) for j in range(n)]
    hslices = [torch.empty(part, dtype=t.dtype, pin_memory=True) for t in dslices]
    for h, d in zip(hslices, dslices):
        h.copy_(d)
    torch.cuda.synchronize()
    out = []
    for sl in (dslices, hslices):
        plan = _plan(n * part, n, lp)
        g = torch.empty(part, dtype=torch.float32, device=dev)
        plan.reduce(0, sl, g, 1.0)
        out.append((g, plan_stats(plan)[:2]))
        plan.close()
    assert same_floats(out[0][0].cpu().numpy(), out[1][0].cpu().numpy())
    assert out[0][1] == out[1][1]


@pytest.mark.parametrize("lp", [0, 1])
def test_stage3_unit_by_unit_reduce_equals_partition_reduce(zlib, lp):
    # backward order: each unit reduce-scattered on its own, last unit first;
    # norm tiles restart per unit, so the bits equal one whole-partition call
    dev = torch.device("cuda")
    n = 4
    sizes, units = [70_000, 5, 33_000, 100_000, 7, TILE * 2], [0, 0, 1, 2, 3, 4]
    res = []
    for mode in ("partition", "units", "pairs", "buckets"):
        plan = _plan(-1, n, lp, stage=3, align=8, sizes=sizes, units=units)
        P = plan.part_len
        sl = [synth.grad_slice(P, lp, 1e-2, 1.0, 4, 1, j, 1, dev) for j in range(n)]
        g = torch.full((P,), float("nan"), dtype=torch.float32, device=dev)
        if mode == "partition":
            plan.reduce(1, sl, g, 1.0)
        elif mode == "units":
            for u in reversed(range(plan.n_units)):
                plan.reduce_units(1, u, 1, sl, g, 1.0)
        elif mode == "pairs":
            plan.reduce_units(1, 3, 2, sl, g, 1.0)
            plan.reduce_units(1, 1, 2, sl, g, 1.0)
            plan.reduce_units(1, 0, 1, sl, g, 1.0)
        else:
            plan.reduce(1, sl, g, 1.0, bucket_elems=3 * TILE + 5)
        res.append((g.cpu().numpy(), plan_stats(plan)[:2], [synth.to_numpy_codes(t) for t in sl]))
        plan.close()
    for other in res[1:]:
        assert same_floats(res[0][0], other[0])
        assert res[0][1] == other[1]
    og, oss, oof = oracle.reduce(res[0][2], lp, 1.0)
    assert same_floats(res[0][0], og) and oof == res[0][1][1]
    assert abs(res[0][1][0] - oss) <= 1e-9 * oss


@pytest.mark.parametrize("quant", [None, Z.ZERO_QUANT_INT8, Z.ZERO_QUANT_FP8_E4M3])
@pytest.mark.parametrize("prefetch", [True, False])
def test_stage3_prefetch_schedule_matches_the_oracle(zlib, quant, prefetch):
    # the benchmark's stage-3 call list (schedule module): forward gathers of
    # the 3 units, backward gathers in reverse order with bucketed reduces,
    # the decision, Adam (+ quantize); with prefetch the gathers alternate
    # between two streams and two layer buffers.  Every gathered layer buffer
    # (both streams, both buffers) is compared whole with the oracle's gather
    # of the shards as they stood before the step, and the step's state
    # with the oracle's, over 3 steps (the own shard changes every step).
    import dataclasses
    from zero_partitioned_mixed_flat_gb300.workloads import gpt2_block
    # the 7.5B layout in small: a rest unit and two transformer blocks, N = 64
    blocks = gpt2_block(512)
    w = dataclasses.replace(WORKLOADS["profile-zero3"], sizes=[8 << 20] + blocks + blocks,
                            unit_of_tensor=[0] + [1] * len(blocks) + [2] * len(blocks),
                            bucket_elems=60_000)   # units 2 and 1 share a bucket, unit 0 alone
    if quant is not None:
        w = dataclasses.replace(w, gather_quantized=True, quant_format=quant)
    h = Harness(w, full=True, threads=16, prefetch=prefetch)
    assert (h.side is not None) == prefetch
    for _ in range(3):
        h.step()
    assert h.gather_log == [2 * h.plan.n_units] * 3
    h.close()


def test_partly_reduced_partition_counts_only_its_part(zlib):
    # a unit reduced alone contributes only its own tiles to the step's norm
    dev = torch.device("cuda")
    n = 2
    plan = _plan(-1, n, 0, stage=3, align=8, sizes=[50_000, 60_000], units=[0, 1])
    P = plan.part_len
    sl = [synth.grad_slice(P, 0, 1e-2, 1.0, 6, 1, j, 0, dev) for j in range(n)]
    g = torch.zeros(P, dtype=torch.float32, device=dev)
    plan.reduce(0, sl, g, 1.0)                       # step 1: everything
    w = torch.zeros(P, device=dev); m = torch.zeros(P, device=dev); v = torch.zeros(P, device=dev)
    plan.adam(0, g, w, m, v, None, 1e-3, .9, .999, 1e-8, 0., 1, 1.0, 0.0)
    plan.reduce_units(0, 1, 1, sl, g, 1.0)          # step 2: unit 1 only
    ss, _, _ = plan_stats(plan)
    off = plan.unit_shard_offset(1)
    _, oss, _ = oracle.reduce([synth.to_numpy_codes(t[off:]) for t in sl], 0, 1.0)
    assert abs(ss - oss) <= 1e-9 * oss
    plan.close()
