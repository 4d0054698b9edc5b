"""The step's call list (schedule.StepSchedule) on CPU.

A real plan gives the layout; the library's device calls are recorded instead
of run.  What is checked is the order "10.6 ZeRO 与 FSDP" §10.6.4 sets for
stage 3: the forward gathers visit every unit in order and the backward
gathers in reverse; each unit's gradients are reduced exactly once, after its
backward gather, in buckets of consecutive units that close as soon as they
hold reduce_bucket_size elements ("从'年糕切片'理解ZeRO" §2.2), the last one at
unit 0; with a prefetch stream (§10.6.4 预取, §10.6.6 overlap_comm) the gathers
alternate between two streams and two layer buffers and every reduce follows a
wait on the side stream; the decision comes after every reduce and before any
update; the quantized gather re-quantizes every updated shard.  For stages 1/2
(§10.6.2 Steps 2-4): the reduces, the exchange of a multi-rank job, the
decision, the updates.  The calls' byte counts are the per-element figures of
the step (2N + 4 B per reduced element, 30 B per updated element, 4 B per
gathered layer element).
"""
import pytest

import zero_partitioned_mixed_flat_gb300 as Z
from zero_partitioned_mixed_flat_gb300.schedule import Hyper, StepBuffers, StepSchedule

HP = Hyper(1e-4, 0.9, 0.999, 1e-8, 0.01, 1, 1.0)


@pytest.fixture(scope="module")
def lib():
    from zero_partitioned_mixed_flat_gb300 import build
    build.build()
    return Z.load()


class Stream:
    def __init__(self, handle):
        self.cuda_stream = handle


class Recorder:
    """The plan's layout, with every device call recorded as (kind, ...)."""

    def __init__(self, plan):
        self._plan = plan
        self.log = []

    def __getattr__(self, name):
        return getattr(self._plan, name)

    def gather(self, u, shards, out, stream=None):
        self.log.append(("gather", u, stream, out))

    def gather_quantized(self, u, codes, scales, out, stream=None):
        self.log.append(("gather", u, stream, out))

    def reduce_units(self, r, first, count, slices, g, scale, stream=None):
        self.log.append(("reduce", r, first, count))

    def reduce(self, r, slices, g, scale, bucket, stream=None):
        self.log.append(("reduce", r, bucket))

    def reduce_many(self, ranks, slices, g, scale, bucket, stream=None):
        self.log.append(("reduce", tuple(ranks), bucket))

    def adam_range(self, r, begin, length, *args):
        self.log.append(("decide", r, begin, length))

    def adam(self, r, *args):
        self.log.append(("adam", r))

    def adam_many(self, ranks, *args):
        self.log.append(("adam", tuple(ranks)))

    def quantize(self, shard, codes, scales, stream=None):
        self.log.append(("quantize", shard))


def _bufs(ranks, n, **kw):
    return StepBuffers(ranks=list(ranks), slices={r: ["s%d_%d" % (r, j) for j in range(n)] for r in ranks},
                       g={r: "g%d" % r for r in ranks}, master={r: "w%d" % r for r in ranks},
                       m={r: "m%d" % r for r in ranks}, v={r: "v%d" % r for r in ranks}, **kw)


def _run(calls):
    """Run every call but the stream waits (they need a device)."""
    for c in calls:
        if c.kind != "wait":
            c.fn()


SIZES = [70_000, 5, 33_000, 100_000, 7, 40_000, 12_345, 9]
UNITS = [0, 0, 1, 2, 2, 3, 4, 5]


@pytest.mark.parametrize("bucket", [0, 1, 30_000, 60_000, 10 ** 9])
@pytest.mark.parametrize("prefetch", [False, True])
@pytest.mark.parametrize("quantized", [False, True])
def test_stage3_call_order(lib, bucket, prefetch, quantized):
    n, ranks = 4, [0, 2]
    plan = Z.ZeroPlan(-1, n, SIZES, 128, 3, UNITS, Z.ZERO_FP16)
    rec = Recorder(plan)
    U = plan.n_units
    bufs = _bufs(ranks, n, shard={r: "shard%d" % r for r in ranks}, gather_shards=["x"] * n,
                 codes={r: "c%d" % r for r in ranks}, scales={r: "q%d" % r for r in ranks},
                 layer_bufs=["L0", "L1"])
    sched = StepSchedule(rec, bufs, HP, loss_scale=1.0, bucket_elems=bucket, gather=True,
                         quantized=quantized)
    main, side = Stream(11), Stream(22)
    calls = sched.calls(main, side=side if prefetch else None)
    _run(calls)
    log = rec.log
    kinds = [c.kind for c in calls if c.kind != "wait"]
    assert kinds == [e[0] for e in log]

    # gathers: forward in order, backward in reverse, alternating streams and buffers
    gathers = [e for e in log if e[0] == "gather"]
    assert [e[1] for e in gathers] == list(range(U)) + list(range(U))[::-1]
    streams = [11, 22] if prefetch else [11]
    bufs_used = ["L0", "L1"] if prefetch else ["L0"]
    for k, e in enumerate(gathers):
        assert e[2] == streams[k % len(streams)] and e[3] == bufs_used[k % len(streams)]

    # reduces: every unit once per rank, after its backward gather, in buckets
    # of consecutive units that close as soon as they are full
    seen_bwd = set()
    covered = {r: [] for r in ranks}
    groups = []
    fwd_left = U
    for e in log:
        if e[0] == "gather":
            if fwd_left:
                fwd_left -= 1
            else:
                seen_bwd.add(e[1])
        elif e[0] == "reduce":
            _, r, first, count = e
            assert all(u in seen_bwd for u in range(first, first + count))
            covered[r].extend(range(first, first + count))
            if r == ranks[0]:
                groups.append((first, count))
    for r in ranks:
        assert sorted(covered[r]) == list(range(U)) and len(covered[r]) == U
    assert groups[-1][0] == 0
    for first, count in groups:
        elems = sum(plan.shard_len(u) for u in range(first, first + count))
        if bucket:
            if first > 0:
                assert elems >= bucket
            # closed at the first unit that filled it: without its lowest unit it was not full
            assert count == 1 or elems - plan.shard_len(first) < bucket
        else:
            assert count == 1
    # with prefetch, each bucket's reduces follow one wait for the side stream
    if prefetch:
        for i, c in enumerate(calls):
            if c.kind == "reduce" and calls[i - 1].kind != "reduce":
                assert calls[i - 1].kind == "wait"
        assert calls[0].kind == "wait"   # the side stream waits for the previous step's update

    # the decision after the last reduce, then the updates (and re-quantization)
    last_reduce = max(i for i, e in enumerate(log) if e[0] == "reduce")
    assert log[last_reduce + 1] == ("decide", ranks[0], 0, 0)
    tail = log[last_reduce + 2:]
    if quantized:
        assert tail == [("adam", 0), ("quantize", "shard0"), ("adam", 2), ("quantize", "shard2")]
    else:
        assert tail == [("adam", 0), ("adam", 2)]

    # algorithmic bytes of the calls
    nb = {}
    for c in calls:
        nb[c.kind] = nb.get(c.kind, 0) + c.nbytes
    P = plan.part_len
    assert nb["reduce"] == (2 * n + 4) * P * len(ranks)
    assert nb["adam"] == 30 * P * len(ranks)
    per_elem = (3 + 4 / 128) if quantized else 4
    assert nb["gather"] == sum(int(per_elem * int(plan.unit_padded[u])) for u in range(U)) * 2
    plan.close()


@pytest.mark.parametrize("many", [False, True])
@pytest.mark.parametrize("exchange", [False, True])
def test_stage2_call_order(lib, many, exchange):
    n, ranks = 8, [1, 3, 4]
    plan = Z.ZeroPlan(-1, n, [1_000_003, 77], 128, 2, None, Z.ZERO_BF16)
    rec = Recorder(plan)
    bufs = _bufs(ranks, n, param="full", group=object() if exchange else None, stats="stats")
    sched = StepSchedule(rec, bufs, HP, loss_scale=1.0, bucket_elems=50_000, many=many)
    calls = sched.calls(Stream(5))
    kinds = [c.kind for c in calls]
    if many:
        expect = ["reduce"] + (["exchange"] if exchange else []) + ["decide", "adam"]
    else:
        expect = ["reduce"] * 3 + (["exchange"] if exchange else []) + ["decide"] + ["adam"] * 3
    assert kinds == expect
    for c in calls:
        if c.kind != "exchange":
            c.fn()
    if many:
        assert rec.log == [("reduce", (1, 3, 4), 50_000), ("decide", 1, 0, 0), ("adam", (1, 3, 4))]
    else:
        assert rec.log == [("reduce", 1, 50_000), ("reduce", 3, 50_000), ("reduce", 4, 50_000),
                           ("decide", 1, 0, 0), ("adam", 1), ("adam", 3), ("adam", 4)]
    P = plan.part_len
    assert sum(c.nbytes for c in calls if c.kind == "reduce") == (2 * n + 4) * P * 3
    assert sum(c.nbytes for c in calls if c.kind == "adam") == 30 * P * 3
    # one launch per bucket of whole norm tiles when each partition is its own call
    tile = Z.ZERO_NORM_TILE
    if not many:
        assert sched.reduce_launches == -(-P // (-(-50_000 // tile) * tile))
    plan.close()
