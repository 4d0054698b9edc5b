"""Test harness: run a workload's steps through libzero on the GPU and through
the CPU oracle on the same seeded inputs, and compare.

Used by the GPU parity tests.  The oracle never sees a value computed by the
CUDA path: it gets the synthetic inputs (gradient slices, initial master
weights, other ranks' parameter shards) and evolves its own state.

Comparison bars (from the task's parity statement):
  layout, padding, overflow flag, skip, loss scale, step: bit-exact;
  reduced fp32 gradient: bit-exact (fixed rank order on both sides);
  master / m / v: max relative error 1e-6 (denominator floored at 1e-30), and
      bit-exact whenever both sides took the same clip coefficient;
  global norm: 1e-5 relative;
  fp16/bf16 parameters: within 1 ulp (bit-exact when the coefficients agree).
"""
import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

import oracle
import zero_partitioned_mixed_flat_gb300 as Z
from zero_partitioned_mixed_flat_gb300 import synth
from zero_partitioned_mixed_flat_gb300.schedule import Hyper, StepBuffers, StepSchedule
from zero_partitioned_mixed_flat_gb300.workloads import Workload

SEED = 0
REL_TOL = 1e-6
NORM_TOL = 1e-5


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).view(np.uint32)


def same_floats(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equal, treating any two NaNs as equal."""
    eq = bits(a) == bits(b)
    return bool(np.all(eq | (np.isnan(a) & np.isnan(b))))


def max_rel_err(a: np.ndarray, b: np.ndarray) -> float:
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    den = np.maximum(np.abs(b64), 1e-30)
    if a64.size == 0:
        return 0.0
    return float(np.max(np.abs(a64 - b64) / den))


def lp_ulp_dist(a: np.ndarray, b: np.ndarray) -> int:
    """Largest distance in units in the last place between two lp code arrays."""
    def key(c):
        c = c.astype(np.int32)
        return np.where(c & 0x8000, -(c & 0x7FFF), c)
    if a.size == 0:
        return 0
    return int(np.max(np.abs(key(a) - key(b))))


def plan_stats(plan, stream=None):
    """The plan's exported statistics for the current step (zero_partition_stats):
    (exact sum of the per-partition sums of squares, any overflow, the 2N vector).
    The exact sum (math.fsum) is only the test's yardstick for the oracle's
    sequential sum; the library's own sum is the one inside the decision."""
    n = plan.n_ranks
    t = torch.full((2 * n,), float("nan"), dtype=torch.float64, device="cuda")
    plan.partition_stats(t, stream)
    torch.cuda.synchronize()
    v = t.cpu().numpy()
    return math.fsum(v[:n]), int(np.any(v[n:] != 0)), v


def coef_from_norm(norm: float, clip: float) -> float:
    if clip > 0:
        c = clip / (norm + 1e-6)
        if c < 1.0:
            return float(np.float32(c))
    return 1.0


@dataclass
class RankState:
    slices: List[torch.Tensor] = field(default_factory=list)
    g: Optional[torch.Tensor] = None
    master: Optional[torch.Tensor] = None
    m: Optional[torch.Tensor] = None
    v: Optional[torch.Tensor] = None
    shard: Optional[torch.Tensor] = None       # stage 3: this rank's lp shard
    idx: Optional[np.ndarray] = None           # compared positions
    idx_dev: Optional[torch.Tensor] = None
    o_master: Optional[np.ndarray] = None      # oracle state at idx
    o_m: Optional[np.ndarray] = None
    o_v: Optional[np.ndarray] = None
    keep: list = field(default_factory=list)
    pad_idx: Optional[torch.Tensor] = None


class Harness:
    """Runs `w` on the GPU through libzero and on the oracle; compares each step."""

    def __init__(self, w: Workload, ranks=None, full: bool = True, n_sample: int = 1 << 20,
                 threads: int = 8, chunk: int = 1 << 22, device="cuda", bucket=None,
                 stage=None, sub_group: int = 0, prefetch: bool = True,
                 gather_windows: Optional[bool] = None):
        self.w = w
        self.sub_group = sub_group  # > 0: Adam in sub-groups of this many elements
        self.dev = torch.device(device)
        self.full = full
        self.threads = threads
        self.chunk = chunk
        self.stage = w.stage if stage is None else stage
        self.bucket = w.bucket_elems if bucket is None else bucket
        self.plan = Z.ZeroPlan(-1, w.n_ranks, w.sizes, w.align, self.stage, w.unit_of_tensor,
                               w.lp, growth_interval=w.growth_interval)
        if w.reduce_lp_accum:
            self.plan.set_reduce_precision(1)
        self.o_reduce = oracle.reduce_lp_accum if w.reduce_lp_accum else oracle.reduce
        self.lay = oracle.layout(w.sizes, w.n_ranks, w.align, self.stage, w.unit_of_tensor)
        assert self.plan.psi_padded == self.lay["psi_padded"]
        assert self.plan.part_len == self.lay["part_len"]
        self.P = self.plan.part_len
        self.ranks = list(w.ranks if ranks is None else ranks)
        self.S = w.loss_scale
        self.o_step = 0
        self.o_good = 0
        self.step_no = 0
        self.log: List[Dict] = []
        gen = np.random.default_rng(1234)
        if self.stage == 3:
            self.param = None
        else:
            self.param = torch.zeros(self.plan.psi_padded, dtype=synth.LP_DTYPES[w.lp],
                                     device=self.dev)
        self.st: Dict[int, RankState] = {}
        self.o_param: Dict[int, np.ndarray] = {}
        for r in self.ranks:
            s = RankState()
            s.keep = self.plan.keep_ranges(r)
            s.master = synth.master_init(self.P, w.master_std, SEED, r, self.dev, s.keep)
            s.m = torch.zeros(self.P, dtype=torch.float32, device=self.dev)
            s.v = torch.zeros(self.P, dtype=torch.float32, device=self.dev)
            s.g = torch.full((self.P,), float("nan"), dtype=torch.float32, device=self.dev)
            if self.stage == 3:
                s.shard = torch.zeros(self.P, dtype=synth.LP_DTYPES[w.lp], device=self.dev)
            if full or self.P <= n_sample:
                s.idx = None          # every position is compared
            else:
                edges = [np.arange(0, min(4096, self.P)), np.arange(max(0, self.P - 4096), self.P)]
                tiles = np.arange(0, self.P, 32768)
                edges += [t + np.arange(-8, 8) for t in tiles[1:]]
                rnd = gen.integers(0, self.P, n_sample)
                s.idx = np.unique(np.clip(np.concatenate(edges + [rnd]), 0, self.P - 1))
            if s.idx is None:
                s.o_master = s.master.cpu().numpy().copy()
            else:
                s.idx_dev = torch.from_numpy(s.idx).to(self.dev)
                s.o_master = s.master[s.idx_dev].cpu().numpy().copy()
            s.o_m = np.zeros(s.o_master.size, np.float32)
            s.o_v = np.zeros(s.o_master.size, np.float32)
            # padding positions inside the partition
            mask = torch.ones(self.P, dtype=torch.bool, device=self.dev)
            for a, n in s.keep:
                mask[a:a + n] = False
            s.pad_idx = torch.nonzero(mask).flatten()
            self.st[r] = s
        # stage-3 gathers: whole layer buffers, or sampled windows of them
        self.gather_windows = (not full) if gather_windows is None else gather_windows
        self._build_schedule(gen, prefetch)

    # ------------------------------------------------------- the schedule
    def _build_schedule(self, gen, prefetch):
        """The benchmark's call list (zero_partitioned_mixed_flat_gb300.schedule)
        over this harness's buffers; stage-3 workloads with gathers add the
        other ranks' synthetic shards, two layer buffers and (prefetch) a side
        stream, and every gathered layer buffer is checked against the oracle."""
        w = self.w
        self.gathers = bool(self.stage == 3 and w.gather)
        self.quantized = bool(self.gathers and w.gather_quantized)
        self.side = None
        self.gather_log: List[Dict] = []
        bufs = StepBuffers(ranks=self.ranks, slices={}, g={r: self.st[r].g for r in self.ranks},
                           master={r: self.st[r].master for r in self.ranks},
                           m={r: self.st[r].m for r in self.ranks},
                           v={r: self.st[r].v for r in self.ranks}, param=self.param,
                           shard={r: self.st[r].shard for r in self.ranks} if self.stage == 3 else {})
        if self.gathers:
            lpd = synth.LP_DTYPES[w.lp]
            n = w.n_ranks
            bufs.gather_shards = [self.st[j].shard if j in self.st else
                                  synth.lp_shard(self.P, w.lp, w.master_std, 0, j, self.dev)
                                  for j in range(n)]
            biggest = max(self.plan.shard_len(u) for u in range(self.plan.n_units)) * n
            bufs.layer_bufs = [torch.full((biggest,), float("nan"), dtype=lpd, device=self.dev)
                               for _ in range(2)]
            if self.quantized:
                self.plan.set_gather_quantization(w.quant_format)
                bufs.codes = [torch.empty(self.P, dtype=torch.int8, device=self.dev) for _ in range(n)]
                bufs.scales = [torch.empty(self.P // 128, dtype=torch.float32, device=self.dev)
                               for _ in range(n)]
                for j in range(n):
                    self.plan.quantize(bufs.gather_shards[j], bufs.codes[j], bufs.scales[j])
            if prefetch:
                self.side = torch.cuda.Stream(self.dev)
            # compared positions of each unit's layer buffer: all of it, or
            # (sampled harness) block-aligned windows of every rank's segment
            self.g_windows, self.g_index = {}, {}
            host_pos = []
            for u in range(self.plan.n_units):
                sl, off = self.plan.shard_len(u), self.plan.unit_shard_offset(u)
                if not self.gather_windows:
                    wins = [(0, sl)]
                else:
                    L = min(2048, sl)
                    starts = {0, (sl - L) // 128 * 128}
                    starts |= {int(x) // 128 * 128 for x in gen.integers(0, max(1, sl - L), 6)}
                    wins = [(k0, min(L, sl - k0)) for k0 in sorted(starts)]
                self.g_windows[u] = wins
                idx = np.concatenate([j * sl + k0 + np.arange(L) for k0, L in wins for j in range(n)])
                self.g_index[u] = torch.from_numpy(idx).to(self.dev)
                host_pos += [off + k0 + np.arange(L) for k0, L in wins]
            self.g_host_pos = np.concatenate(host_pos)
            self.g_host_pos_dev = torch.from_numpy(self.g_host_pos).to(self.dev)
        self.bufs = bufs
        self.sched = StepSchedule(self.plan, bufs, Hyper(w.lr, w.beta1, w.beta2, w.eps, w.wd,
                                                         int(w.adamw), w.clip),
                                  self.S, self.bucket, gather=self.gathers, quantized=self.quantized)

    def _expected_gathers(self):
        """The oracle's gather of every unit (at the compared positions) from
        the shards as they stand before the step."""
        w, n = self.w, self.w.n_ranks
        host = [synth.to_numpy_codes(t[self.g_host_pos_dev]) for t in self.bufs.gather_shards]
        exp, pos = {}, 0
        for u in range(self.plan.n_units):
            parts = []
            for k0, L in self.g_windows[u]:
                win = [h[pos:pos + L] for h in host]
                pos += L
                if self.quantized:
                    qf = oracle.quantize_blocks_fp8 if w.quant_format else oracle.quantize_blocks
                    dq = oracle.dequant_gather_fp8 if w.quant_format else oracle.dequant_gather
                    qs = [qf(x, w.lp, 128) for x in win]
                    parts.append(dq([q for q, _ in qs], [c for _, c in qs], w.lp, 128))
                else:
                    parts.append(oracle.gather(win))
            exp[u] = np.concatenate(parts)
        return exp

    # ------------------------------------------------------------ inputs
    def make_slices(self, r: int):
        w = self.w
        scale = self.S if w.grads_times_scale else 1.0
        s = self.st[r]
        s.slices = [synth.grad_slice(self.P, w.lp, w.grad_std, scale, SEED, self.step_no, j, r,
                                     self.dev, s.keep) for j in range(w.n_ranks)]
        if w.inject_inf_step and self.step_no == w.inject_inf_step and r == self.ranks[0]:
            j, i = synth.inject_position(SEED, self.step_no, r, w.n_ranks, s.keep)
            s.slices[j][i] = float("inf")

    # ------------------------------------------------------------- GPU
    def gpu_step(self):
        w = self.w
        if not self.sub_group:
            # the benchmark's own call list for this step
            self.bufs.slices = {r: self.st[r].slices for r in self.ranks}
            self.sched.loss_scale = self.S
            stream = torch.cuda.current_stream(self.dev)
            snaps = []
            exp = None
            hook = None
            if self.gathers:
                exp = self._expected_gathers()

                def hook(u, buf, st):
                    with torch.cuda.stream(st):
                        snaps.append((u, buf[self.g_index[u]]))
            StepSchedule.run(self.sched.calls(stream, side=self.side, on_gather=hook))
            if self.side is not None:
                stream.wait_stream(self.side)
            res = self.plan.result()
            if self.gathers:
                torch.cuda.synchronize()
                assert len(snaps) == 2 * self.plan.n_units   # forward and backward
                for u, snap in snaps:
                    got = synth.to_numpy_codes(snap)
                    assert np.array_equal(got, exp[u]), "gathered layer %d differs from the oracle" % u
                self.gather_log.append(len(snaps))
            return res
        for r in self.ranks:
            s = self.st[r]
            self.plan.reduce(r, s.slices, s.g, self.S, self.bucket)
        for r in self.ranks:
            s = self.st[r]
            out = s.shard if self.stage == 3 else self.param
            # an empty range first (it only takes the decision), then the
            # sub-groups in reverse order, the last one ragged
            self.plan.adam_range(r, 0, 0, s.g, s.master, s.m, s.v, out, w.lr, w.beta1, w.beta2,
                                 w.eps, w.wd, int(w.adamw), self.S, w.clip)
            for b in reversed(range(0, self.P, self.sub_group)):
                n = min(self.sub_group, self.P - b)
                self.plan.adam_range(r, b, n, s.g, s.master, s.m, s.v, out, w.lr, w.beta1,
                                     w.beta2, w.eps, w.wd, int(w.adamw), self.S, w.clip)
        return self.plan.result()

    # ---------------------------------------------------------- oracle
    def _oracle_reduce(self, r: int):
        """Chunked oracle reduce of rank r; compares the GPU gradient bit for bit.
        Returns (sumsq, overflow, g at idx)."""
        w, s = self.w, self.st[r]
        chunks = [(c, min(self.P, c + self.chunk)) for c in range(0, self.P, self.chunk)]
        idx = s.idx

        def work(c0, c1, host_slices, host_g):
            g, ss, of = self.o_reduce(host_slices, w.lp, self.S)
            ok = same_floats(g, host_g)
            if idx is None:
                return ss, of, ok, g
            lo, hi = np.searchsorted(idx, [c0, c1])
            return ss, of, ok, g[idx[lo:hi] - c0]

        results = []
        with ThreadPoolExecutor(self.threads) as ex:
            pending = []
            for c0, c1 in chunks:
                hs = [synth.to_numpy_codes(t[c0:c1]) for t in s.slices]
                hg = s.g[c0:c1].cpu().numpy()
                pending.append(ex.submit(work, c0, c1, hs, hg))
                if len(pending) >= 2 * self.threads:
                    results.append(pending.pop(0).result())
            results += [f.result() for f in pending]
        ss = 0.0
        of = 0
        for r_ss, r_of, ok, _ in results:
            ss += r_ss
            of |= r_of
            assert ok, "reduced gradient differs from the oracle (rank %d)" % r
        g_idx = np.concatenate([x[3] for x in results]) if results else np.zeros(0, np.float32)
        return ss, of, g_idx

    def oracle_step(self):
        w = self.w
        tot, of, g_at = 0.0, 0, {}
        for r in self.ranks:
            ss, o, g_at[r] = self._oracle_reduce(r)
            tot += ss
            of |= o
        d = oracle.decide(tot, of, w.clip, self.S, self.o_step, self.o_good, w.growth_interval,
                          w.beta1, w.beta2)
        params = {}
        for r in self.ranks:
            s = self.st[r]
            args = (w.lp, d["coef"], d["skip"], w.lr, w.beta1, w.beta2, w.eps, w.wd, int(w.adamw),
                    d["bc1"], d["bc2"])
            n = s.o_master.size
            if n <= self.chunk:
                params[r] = oracle.adam(g_at[r], s.o_master, s.o_m, s.o_v, *args)
                continue
            # element-wise: the same update on contiguous pieces, on several host threads
            bounds = [(c, min(n, c + self.chunk)) for c in range(0, n, self.chunk)]
            with ThreadPoolExecutor(self.threads) as ex:
                parts = list(ex.map(lambda b: oracle.adam(g_at[r][b[0]:b[1]], s.o_master[b[0]:b[1]],
                                                          s.o_m[b[0]:b[1]], s.o_v[b[0]:b[1]], *args),
                                    bounds))
            params[r] = np.concatenate(parts)
        return d, params

    def _compare_state(self, r, exact, params_r, info):
        """master/m/v within REL_TOL of the oracle (bit for bit when the clip
        coefficients agree), the lp param within 0/1 ulp; piecewise on host
        threads for large partitions."""
        s = self.st[r]
        if s.idx is None:
            gm, gmm, gv = (t.cpu().numpy() for t in (s.master, s.m, s.v))
            src = s.shard if self.stage == 3 else self.param[r * self.P:(r + 1) * self.P]
            gp = synth.to_numpy_codes(src)
        else:
            gm = s.master[s.idx_dev].cpu().numpy()
            gmm = s.m[s.idx_dev].cpu().numpy()
            gv = s.v[s.idx_dev].cpu().numpy()
            if self.stage == 3:
                gp = synth.to_numpy_codes(s.shard[s.idx_dev])
            else:
                gp = synth.to_numpy_codes(self.param[r * self.P + s.idx_dev])
        n = gm.size
        bounds = [(c, min(n, c + self.chunk)) for c in range(0, n, self.chunk)] or [(0, 0)]

        def piece(b):
            a, z = b
            errs = (max_rel_err(gm[a:z], s.o_master[a:z]), max_rel_err(gmm[a:z], s.o_m[a:z]),
                    max_rel_err(gv[a:z], s.o_v[a:z]))
            same = (same_floats(gm[a:z], s.o_master[a:z]) and same_floats(gmm[a:z], s.o_m[a:z])
                    and same_floats(gv[a:z], s.o_v[a:z]))
            ulp = lp_ulp_dist(gp[a:z], params_r[a:z]) if params_r is not None else 0
            return errs, same, ulp
        with ThreadPoolExecutor(self.threads) as ex:
            res = list(ex.map(piece, bounds))
        errs = tuple(max(x[0][i] for x in res) for i in range(3))
        info.setdefault("rel_err", {})[r] = errs
        info.setdefault("compared", {})[r] = int(n)
        assert max(errs) <= REL_TOL, info
        if exact:
            assert all(x[1] for x in res), info
        if params_r is not None:
            # the param buffer holds the cast of the latest master
            assert max(x[2] for x in res) <= (0 if exact else 1), info

    # --------------------------------------------------------- compare
    def step(self):
        self.step_no += 1
        for r in self.ranks:
            self.make_slices(r)
        res = self.gpu_step()
        d, params = self.oracle_step()
        info = {"step": self.step_no, "gpu": res, "oracle": {k: d[k] for k in
                ("norm", "coef", "skip", "new_scale", "step")}}
        assert res["skipped"] == d["skip"], info
        assert res["step"] == d["step"], info
        assert res["loss_scale"] == d["new_scale"], info
        if d["skip"]:
            assert not math.isfinite(res["norm"]) or not math.isfinite(d["norm"]) or \
                abs(res["norm"] - d["norm"]) <= NORM_TOL * d["norm"], info
        else:
            assert abs(res["norm"] - d["norm"]) <= NORM_TOL * d["norm"], info
        gpu_coef = coef_from_norm(res["norm"], self.w.clip)
        exact = (gpu_coef == d["coef"]) or d["skip"]
        info["coef_equal"] = exact
        for r in self.ranks:
            s = self.st[r]
            if not d["skip"]:
                self.o_param[r] = params[r]
            self._compare_state(r, exact, self.o_param.get(r), info)
            # padding stays exactly zero
            if s.pad_idx.numel():
                for t in (s.master, s.m, s.v):
                    assert not t[s.pad_idx].any().item(), "padding became non-zero"
        self.S = d["new_scale"]
        self.o_step, self.o_good = d["step"], d["good_steps"]
        self.log.append(info)
        return info

    def close(self):
        self.plan.close()
