"""One ZeRO step as an ordered list of libzero calls, to run, time or capture.

Stages 1/2 ("10.6 ZeRO 与 FSDP" §10.6.2 Steps 2-4): every updated partition
is reduce-scattered (zero_reduce_partition, in buckets of reduce_bucket_size,
"从'年糕切片'理解ZeRO" §2.2), the step's one decision is taken, then every
partition is updated and cast into the full parameter layout.

Stage 3 (§10.6.4): the forward all-gather of every unit in order; then, unit
by unit in reverse order, its backward all-gather, its gradients joining the
reduce bucket and a full bucket (or the first unit) reduce-scattered
(zero_reduce_units); then the decision and the per-partition update, and
for the quantized gather (ZeRO++) the quantization of the new shard.

Prefetch (§10.6.4 预取, §10.6.6 overlap_comm): with a side stream, the gathers
alternate between the main and the side stream and between two layer
buffers, so the next unit's gather overlaps the current one; the reduce of a
bucket waits for the side stream (its units' gathers are done), and the side
stream's first gather of a step waits for the main stream (the previous
step's update of the shards).

A multi-rank job (several processes) adds the statistics exchange
(parallel_host.global_decision_inputs) between the reduces and the decision.

This module only orders calls; every step of the arithmetic runs in libzero.
"""
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence

from . import _abi as A


@dataclass
class Call:
    kind: str                 # gather, reduce, exchange, decide, adam, quantize, wait
    nbytes: int               # algorithmic HBM bytes of the call
    launches: int             # kernel launches of the library
    fn: Callable[[], None]
    stream: object            # torch.cuda.Stream, or None for "wait"
    unit: Optional[int] = None
    buf: object = None        # gathers: the layer buffer written


@dataclass
class StepBuffers:
    """The caller-owned buffers one process steps (see include/zero.h for the
    layouts).  slices[r]: the N lp gradient slices of partition r; g, master,
    m, v: per partition; param: the full lp layout (stages 1/2); shard[r]: the
    lp shard of partition r (stage 3).  Stage-3 gathers read gather_shards (N
    lp shard buffers, one of which is this rank's shard) or, quantized,
    codes/scales; layer_bufs holds one layer buffer per gather stream."""
    ranks: List[int]
    slices: Dict[int, Sequence]
    g: Dict[int, object]
    master: Dict[int, object]
    m: Dict[int, object]
    v: Dict[int, object]
    param: object = None
    shard: Dict[int, object] = field(default_factory=dict)
    gather_shards: Optional[List[object]] = None
    codes: Optional[List[object]] = None
    scales: Optional[List[object]] = None
    layer_bufs: List[object] = field(default_factory=list)
    stats: object = None      # 2N float64 (device) for a multi-rank exchange
    group: object = None      # torch.distributed group of that exchange


@dataclass
class Hyper:
    lr: float
    beta1: float
    beta2: float
    eps: float
    wd: float
    adamw: int
    clip: float


class StepSchedule:
    """Builds the call list of one step of `plan` over `bufs`.

    loss_scale is read when a call runs (set it from the previous step's
    result); bucket_elems is the reduce bucket (0: one per partition);
    gather: stage-3 forward/backward gathers; quantized: through codes/scales."""

    def __init__(self, plan, bufs: StepBuffers, hyper: Hyper, loss_scale: float,
                 bucket_elems: int = 0, gather: bool = False, quantized: bool = False,
                 many: Optional[bool] = None):
        self.plan, self.bufs, self.hp = plan, bufs, hyper
        self.loss_scale = loss_scale
        self.bucket_elems = bucket_elems
        self.gather = bool(gather and plan.stage == 3)
        self.quantized = bool(quantized and self.gather)
        # several partitions per process (stages 0-2): one reduce and one Adam
        # call for all of them (zero_reduce_partitions, zero_adam_step_partitions)
        if many is None:
            many = len(bufs.ranks) > 1
        self.many = bool(many and plan.stage != 3 and len(bufs.ranks) > 1)
        tile = A.ZERO_NORM_TILE   # buckets are rounded up to whole norm tiles
        if bucket_elems:
            b = -(-bucket_elems // tile) * tile
            self.reduce_launches = -(-plan.part_len // b) if plan.part_len else 0
        else:
            self.reduce_launches = 1 if plan.part_len else 0

    # ------------------------------------------------------------- the calls
    def calls(self, stream, side=None, slice_lists=None,
              on_gather: Optional[Callable] = None) -> List[Call]:
        """The step on `stream` (torch.cuda.Stream); `side`: second gather
        stream (prefetch); slice_lists: other gradient slices (e.g. host
        buffers) per partition; on_gather(unit, buf, stream) is called right
        after each gather is enqueued (e.g. to snapshot the layer buffer on
        that stream)."""
        import torch
        plan, b, n = self.plan, self.bufs, self.plan.n_ranks
        lists = slice_lists or b.slices
        sh = int(stream.cuda_stream)
        red_b = 2 * n + 4
        out: List[Call] = []
        if self.gather:
            streams = [stream, side] if side is not None else [stream]
            bufs = b.layer_bufs[:len(streams)]
            if len(bufs) < len(streams):
                raise ValueError("one layer buffer per gather stream is needed")
            gb = (3 + 4 / 128) if self.quantized else 4
            ev_main, ev_side = torch.cuda.Event(), torch.cuda.Event()
            if side is not None:
                out.append(Call("wait", 0, 0, lambda: (ev_main.record(stream), side.wait_event(ev_main)),
                                None))
            nth = [0]

            def add_gather(u):
                k = nth[0] % len(streams)
                nth[0] += 1
                st, buf = streams[k], bufs[k]

                def fn(u=u, st=st, buf=buf):
                    if self.quantized:
                        plan.gather_quantized(u, b.codes, b.scales, buf, int(st.cuda_stream))
                    else:
                        plan.gather(u, b.gather_shards, buf, int(st.cuda_stream))
                    if on_gather is not None:
                        on_gather(u, buf, st)
                out.append(Call("gather", int(gb * int(plan.unit_padded[u])), 1, fn, st, u, buf))

            units = list(range(plan.n_units))
            for u in units:                      # forward
                add_gather(u)
            pending = []
            for u in units[::-1]:                # backward
                add_gather(u)
                pending.append(u)
                elems = sum(plan.shard_len(x) for x in pending)
                if not self.bucket_elems or elems >= self.bucket_elems or u == 0:
                    if side is not None:
                        out.append(Call("wait", 0, 0,
                                        lambda: (ev_side.record(side), stream.wait_event(ev_side)), None))
                    first, cnt = min(pending), len(pending)
                    for r in b.ranks:
                        out.append(Call("reduce", red_b * elems, -(-cnt // 64),
                                        lambda first=first, cnt=cnt, r=r: plan.reduce_units(
                                            r, first, cnt, lists[r], b.g[r], self.loss_scale, sh),
                                        stream))
                    pending = []
        elif self.many:
            # every partition in one call (zero_reduce_partitions)
            rk = list(b.ranks)
            out.append(Call("reduce", red_b * plan.part_len * len(rk), self.many_reduce_launches(),
                            lambda: plan.reduce_many(rk, [lists[r] for r in rk], [b.g[r] for r in rk],
                                                     self.loss_scale, self.bucket_elems, sh), stream))
        else:
            launches = self.reduce_launches if plan.stage != 3 else -(-plan.n_units // 64)
            for r in b.ranks:
                out.append(Call("reduce", red_b * plan.part_len, launches,
                                lambda r=r: plan.reduce(r, lists[r], b.g[r], self.loss_scale,
                                                        self.bucket_elems, sh), stream))
        if b.group is not None:
            out.append(Call("exchange", 16 * n, 1, self._exchange, stream))
        for i, r in enumerate(b.ranks):
            if i == 0:
                # the step's one decision (norm of every reduced partition, clip,
                # skip, loss scale, t) as its own call: an empty Adam range
                out.append(Call("decide", 8 * self.tiles_per_partition() * len(b.ranks), 1,
                                lambda r=r: self._adam(r, sh, decide_only=True), stream))
            if self.many:
                if i == 0:
                    out.append(Call("adam", 30 * plan.part_len * len(b.ranks),
                                    -(-len(b.ranks) // 64), lambda: self._adam_many(sh), stream))
                continue
            out.append(Call("adam", 30 * plan.part_len, 1, lambda r=r: self._adam(r, sh), stream))
            if self.quantized:
                out.append(Call("quantize", int((3 + 4 / 128) * plan.part_len), 1,
                                lambda r=r: plan.quantize(b.shard[r], b.codes[r], b.scales[r], sh),
                                stream))
        return out

    @staticmethod
    def run(calls: List[Call]):
        for c in calls:
            c.fn()

    # --------------------------------------------------------------- helpers
    def _exchange(self):
        from .parallel_host import global_decision_inputs
        global_decision_inputs(self.plan, self.bufs.stats, self.bufs.group)

    def _adam(self, r, stream, decide_only=False):
        b, hp = self.bufs, self.hp
        out = b.shard[r] if self.plan.stage == 3 else b.param
        args = (b.g[r], b.master[r], b.m[r], b.v[r], out, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.wd,
                int(hp.adamw), self.loss_scale, hp.clip, 0.0, 0, stream)
        if decide_only:
            self.plan.adam_range(r, 0, 0, *args)
        else:
            self.plan.adam(r, *args)

    def _adam_many(self, stream):
        b, hp = self.bufs, self.hp
        rk = list(b.ranks)
        self.plan.adam_many(rk, [b.g[r] for r in rk], [b.master[r] for r in rk], [b.m[r] for r in rk],
                            [b.v[r] for r in rk], [b.param] * len(rk), hp.lr, hp.beta1, hp.beta2,
                            hp.eps, hp.wd, int(hp.adamw), self.loss_scale, hp.clip, 0.0, 0, stream)

    def many_reduce_launches(self) -> int:
        """Kernel launches of zero_reduce_partitions over this step's partitions
        (the library's grouping: consecutive pieces while a launch holds at most
        one bucket, at most 64 pieces and the slices of floor(512/N) partitions,
        floor(1024/N) when N > 64)."""
        P, n = self.plan.part_len, self.plan.n_ranks
        if P == 0:
            return 0
        tile = A.ZERO_NORM_TILE
        piece = -(-self.bucket_elems // tile) * tile if self.bucket_elems else 0
        per_table = max(1, (512 if n <= 64 else 1024) // n)
        pieces = [min(piece, P - b0) for b0 in range(0, P, piece)] if piece else [P]
        launches, elems, segs, parts = 0, 0, 0, 0
        for _ in self.bufs.ranks:
            new_part = True
            for length in pieces:
                need = 1 if new_part else 0
                if segs and ((piece and elems + length > piece) or segs == 64 or parts + need > per_table):
                    launches += 1
                    elems = segs = parts = 0
                    need = 1
                parts += need
                new_part = False
                segs += 1
                elems += length
        return launches + (1 if segs else 0)

    def tiles_per_partition(self) -> int:
        """Norm tiles of one partition (per unit shard in stage 3)."""
        t = A.ZERO_NORM_TILE
        if self.plan.stage == 3:
            return sum(-(-self.plan.shard_len(u) // t) for u in range(self.plan.n_units))
        return -(-self.plan.part_len // t)
