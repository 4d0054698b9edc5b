"""Host-side checks of libzero (CPU only: no kernel is launched).

The library loads on a machine without a GPU (CUDA runtime linked
statically), exports every entry point include/zero.h declares, and its
partitioner and accounting agree with the independent oracle bit for bit.
Argument validation happens before any device call, so it is tested here.
"""
import ctypes as C
import os
import random
import re

import numpy as np
import pytest

import zero_partitioned_mixed_flat_gb300 as Z
from zero_partitioned_mixed_flat_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from zero_partitioned_mixed_flat_gb300 import build
    build.build()
    return Z.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "zero.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zero_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(Z.SIGNATURES) == names   # the binding covers exactly the ABI


def _prototypes():
    """name -> (return type, [parameter types]) of every function declared in
    include/zero.h, with the C types reduced to what a call passes."""
    text = open(os.path.join(ROOT, "include", "zero.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = {}
    for ret, name, args in re.findall(
            r"(zero_status|void|const char \*)\s*\b(zero_[a-z_]+)\s*\(([^)]*)\)\s*;", text):
        kinds = []
        for a in [x.strip() for x in args.split(",") if x.strip() and x.strip() != "void"]:
            a = re.sub(r"\[[^]]*\]", "*", a)              # array parameters are pointers
            if "*" in a:
                kinds.append("ptr")
            else:
                kinds.append(a.split()[0].replace("const", "").strip() or a.split()[1])
        protos[name] = (ret.replace(" ", ""), kinds)
    return protos


_CTYPES = {"ptr": (C.c_void_p,), "int32_t": (C.c_int32,), "int64_t": (C.c_int64,),
           "float": (C.c_float,), "double": (C.c_double,), "zero_lp": (C.c_int32,)}


def test_binding_signatures_match_the_header():
    protos = _prototypes()
    assert sorted(protos) == sorted(Z.SIGNATURES)
    for name, (ret, kinds) in protos.items():
        cret, cargs = Z.SIGNATURES[name]
        assert len(cargs) == len(kinds), name
        for i, (k, c) in enumerate(zip(kinds, cargs)):
            assert c in _CTYPES[k], (name, i, k, c)
        assert {"zero_status": C.c_int32, "void": None, "constchar*": C.c_char_p}[ret] == cret, name


def _cmp_layout(orc, sizes, n, align, stage, units):
    plan = Z.zero_plan_create(-1 if sizes else 0, n, sizes or None, align, stage, units, 0)
    try:
        lay = orc.layout(sizes or [0], n, align, stage, units)
        psi_p, part, offs = Z.zero_plan_query(plan, len(sizes))
        assert psi_p == lay["psi_padded"] and part == lay["part_len"]
        assert list(offs) == list(lay["tensor_offsets"])[:len(sizes)]
        nu, uoff, upad = Z.zero_plan_units(plan)
        assert nu == lay["n_units"]
        assert list(uoff) == list(lay["unit_offsets"]) and list(upad) == list(lay["unit_padded"])
        # each unit's shard: U_p / N (stage 0: U_p) at the running offset in a partition
        sl, so = Z.zero_plan_unit_shards(plan, nu)
        exp_len = [int(x) if stage == 0 else int(x) // n for x in lay["unit_padded"]]
        assert list(sl) == exp_len
        assert list(so) == [sum(exp_len[:u]) for u in range(nu)]
        assert sum(exp_len) == part
        for r in range(n):
            got = Z.zero_plan_fragments(plan, r)
            exp = orc.fragments(sizes or [0], n, align, stage, r, units)
            assert np.array_equal(got, exp), (sizes, n, align, stage, r)
    finally:
        Z.zero_plan_destroy(plan)


def test_plan_matches_oracle_random(lib, orc):
    rng = random.Random(23)
    for _ in range(300):
        nt = rng.randrange(1, 9)
        sizes = [rng.choice([0, 1, 7, 8, 100, 1000, 4097, 65536]) for _ in range(nt)]
        n = rng.choice([1, 2, 3, 4, 8, 64])
        align = rng.choice([8, 16, 128])
        stage = rng.choice([0, 1, 2, 3])
        units = None
        if stage == 3 and rng.random() < 0.8:
            units, u = [], 0
            for t in range(nt):
                if t and rng.random() < 0.5:
                    u += 1
                units.append(u)
        _cmp_layout(orc, sizes, n, align, stage, units)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_plan_matches_oracle_workloads(lib, orc, name):
    w = WORKLOADS[name]
    plan = Z.ZeroPlan(-1, w.n_ranks, w.sizes, w.align, w.stage, w.unit_of_tensor, w.lp)
    lay = orc.layout(w.sizes, w.n_ranks, w.align, w.stage, w.unit_of_tensor)
    assert plan.psi_padded == lay["psi_padded"] and plan.part_len == lay["part_len"]
    assert list(plan.tensor_offsets) == list(lay["tensor_offsets"])
    for r in sorted({0, w.n_ranks - 1}):
        assert np.array_equal(plan.fragments(r),
                              orc.fragments(w.sizes, w.n_ranks, w.align, w.stage, r,
                                            w.unit_of_tensor))
    plan.close()


def test_memory_report_matches_oracle(lib, orc):
    rng = random.Random(5)
    cases = [(7_500_000_000, 64, 1), (30_000_000_000, 64, 1), (1_000_000_000_000, 1024, 1),
             (13_000_000_000, 16, 128), (0, 1, 1)]
    cases += [(rng.randrange(0, 10 ** 13), rng.choice([1, 3, 8, 64, 1024]),
               rng.choice([1, 8, 128])) for _ in range(500)]
    for psi, n, al in cases:
        f1, a1, c1 = Z.zero_memory_report(psi, n, al)
        f2, a2, c2 = orc.memory(psi, n, al)
        assert np.array_equal(f1, f2) and np.array_equal(a1, a2) and np.array_equal(c1, c2)


@pytest.mark.parametrize("args", [
    dict(n_ranks=0), dict(n_ranks=1025), dict(align=4), dict(align=12), dict(stage=4),
    dict(stage=3, sizes=[4, 4], units=[0, 2]), dict(stage=3, sizes=[4, 4], units=[1, 1]),
    dict(sizes=[4, -1]), dict(psi=9, sizes=[4, 4]), dict(lp=2), dict(psi=-5, sizes=None),
])
def test_plan_create_rejects(lib, args):
    a = dict(psi=-1, n_ranks=2, sizes=[16, 16], align=8, stage=1, units=None, lp=0)
    a.update(args)
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_plan_create(a["psi"], a["n_ranks"], a["sizes"], a["align"], a["stage"],
                           a["units"], a["lp"])
    assert e.value.code == Z.ZERO_EINVAL


def test_step_calls_validate_before_touching_the_device(lib):
    plan = Z.zero_plan_create(1024, 2, None, 8, 1, None, 0)
    try:
        buf = 1 << 20  # a fake, 16-byte aligned address: never dereferenced
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partition(plan, 2, [buf, buf], buf, 1.0, 0, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # rank >= N
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partition(plan, 0, [buf, buf + 2], buf, 1.0, 0, stream=0)
        assert e.value.code == Z.ZERO_EALIGN                     # misaligned slice
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partition(plan, 0, [buf, buf], buf + 4, 1.0, 0, stream=0)
        assert e.value.code == Z.ZERO_EALIGN                     # misaligned output
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partition(plan, 0, [buf, buf], buf, 0.0, 0, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # loss scale <= 0
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partition(plan, 0, [buf, None], buf, 1.0, 0, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # NULL slice
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_adam_step(plan, 0, buf, buf, buf, buf, buf, 1e-3, .9, .999, 1e-8, 0., 1,
                             1.0, 1.0, stream=0)
        assert e.value.code == Z.ZERO_ESTATE                     # Adam before any reduce
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_adam_step(plan, 0, buf, buf + 8, buf, buf, buf, 1e-3, .9, .999, 1e-8, 0.,
                             1, 1.0, 1.0, stream=0)
        assert e.value.code == Z.ZERO_EALIGN
        for begin, length, code in [(-8, 8, Z.ZERO_EINVAL), (0, 520, Z.ZERO_EINVAL),
                                    (512, 8, Z.ZERO_EINVAL), (4, 8, Z.ZERO_EALIGN),
                                    (0, 12, Z.ZERO_EALIGN)]:   # P = 512
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_adam_step_range(plan, 0, begin, length, buf, buf, buf, buf, buf, 1e-3, .9,
                                       .999, 1e-8, 0., 1, 1.0, 1.0, stream=0)
            assert e.value.code == code, (begin, length)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_adam_step_range(plan, 0, 8, 8, buf, buf, buf, buf, buf, 1e-3, .9, .999, 1e-8,
                                   0., 1, 1.0, 1.0, stream=0)
        assert e.value.code == Z.ZERO_ESTATE                     # Adam before any reduce
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_gather_layer(plan, 0, [buf, buf], buf, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # not a stage-3 plan
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_allgather_params(plan, [buf, buf + 8], buf, 0, stream=0)
        assert e.value.code == Z.ZERO_EALIGN                     # misaligned partition
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_allgather_params(plan, [buf, None], buf, 0, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # NULL partition
        with pytest.raises(Z.ZeroError):
            Z.zero_plan_fragments(plan, 5)
        assert "rank" in Z.zero_last_error()
        # several partitions in one call: every argument checked before any CUDA call
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partitions(plan, [1, 1], [[buf, buf], [buf, buf]], [buf, buf], 1.0,
                                     stream=0)
        assert e.value.code == Z.ZERO_EINVAL and "twice" in Z.zero_last_error()
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partitions(plan, [0, 2], [[buf, buf], [buf, buf]], [buf, buf], 1.0,
                                     stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # rank >= N
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partitions(plan, [0, 1], [[buf, buf], [buf, buf + 8]], [buf, buf], 1.0,
                                     stream=0)
        assert e.value.code == Z.ZERO_EALIGN                     # misaligned slice of rank 1
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_reduce_partitions(plan, [0, 1, 1], [[buf, buf]] * 3, [buf] * 3, 1.0, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # more partitions than N
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_adam_step_partitions(plan, [0, 0], [buf] * 2, [buf] * 2, [buf] * 2, [buf] * 2,
                                        [buf] * 2, 1e-3, .9, .999, 1e-8, 0., 1, 1.0, 1.0, stream=0)
        assert e.value.code == Z.ZERO_EINVAL and "twice" in Z.zero_last_error()
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_adam_step_partitions(plan, [0, 1], [buf] * 2, [buf, buf + 4], [buf] * 2,
                                        [buf] * 2, [buf] * 2, 1e-3, .9, .999, 1e-8, 0., 1, 1.0, 1.0,
                                        stream=0)
        assert e.value.code == Z.ZERO_EALIGN
        # the statistics exchange: order and pointer checks
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_partition_stats(plan, buf, stream=0)
        assert e.value.code == Z.ZERO_ESTATE                     # nothing reduced yet
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_partition_stats(plan, buf + 4, stream=0)
        assert e.value.code == Z.ZERO_EALIGN
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_partition_stats(plan, None, stream=0)
        assert e.value.code == Z.ZERO_EINVAL
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_step_set_global_stats(plan, buf)
        assert e.value.code == Z.ZERO_ESTATE
    finally:
        Z.zero_plan_destroy(plan)
    p3 = Z.zero_plan_create(-1, 2, [64, 64], 8, 3, [0, 1], 0)
    try:
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_gather_layer(p3, 2, [1 << 20, 1 << 20], 1 << 20, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # unit out of range
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_gather_layer(p3, 0, [1 << 20, (1 << 20) + 8], 1 << 20, stream=0)
        assert e.value.code == Z.ZERO_EALIGN
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_allgather_params(p3, [1 << 20, 1 << 20], 1 << 20, 0, stream=0)
        assert e.value.code == Z.ZERO_EINVAL                     # stage 3: layer gathers
        Z.zero_plan_set_gather_quantization(p3, Z.ZERO_QUANT_FP8_E4M3)
        Z.zero_plan_set_gather_quantization(p3, Z.ZERO_QUANT_INT8)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_plan_set_gather_quantization(p3, 2)
        assert e.value.code == Z.ZERO_EINVAL                     # unknown code format
    finally:
        Z.zero_plan_destroy(p3)
