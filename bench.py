#!/usr/bin/env python3
"""Benchmark of the ZeRO partitioned mixed-precision Adam step on GB300.

One step = every row of the hot path for one batch of synthetic gradients:
for each simulated partition, the N-way bucketed reduce + unscale + overflow +
sum of squares, the global-norm/skip/loss-scale decision, the fused AdamW +
cast into the parameter layout, and (stage 3) the forward and backward
per-unit gathers of the N parameter shards.  All of it runs in libzero's
kernels through the C ABI; PyTorch only allocates memory and owns the stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl gb300|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload (the baseline arm).
"""
import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "13b-zero2"
METRIC = "partition elements/s per ZeRO step (with achieved HBM GB/s)"
UNIT = "elements/s"
L2_BYTES = 129 * 1000 * 1000
L2_FLUSH_BELOW = 4 * L2_BYTES     # steps touching less than this get an L2 flush
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time the step as one CUDA graph replay (launch-bound small workloads)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="stage 3: issue every gather on one stream (no prefetch)")
    ap.add_argument("--quantized-gather", action="store_true",
                    help="stage-3 workloads: int8 block-quantized gathers")
    ap.add_argument("--n-ranks", type=int, default=None,
                    help="override the workload's N (simulated data-parallel ranks), rank 0 only")
    ap.add_argument("--reduce-in-lp", action="store_true",
                    help="sum the gradient slices in the lp type (reduce_dtype=float16)")
    ap.add_argument("--quant-format", choices=["int8", "fp8"], default=None,
                    help="code format of the quantized gather (default: the workload's)")
    ap.add_argument("--dist-backend", choices=["nccl", "gloo"], default="nccl",
                    help="torch.distributed backend under torchrun (gloo: host-staged exchange, "
                         "e.g. several processes on one GPU)")
    ap.add_argument("--one-job", action="store_true",
                    help="take the multi-rank path (statistics exported, all-reduced and decided "
                         "from the sum) even in a world of one process")
    return ap.parse_args()


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def emit(line):
    """Print the JSON line as the last line of stdout: first write out what C
    libraries left in the C stdio buffer (nccl prints its version banner there
    at the first collective), then the line."""
    import ctypes
    try:
        ctypes.CDLL(None).fflush(None)
    except (OSError, AttributeError):
        pass
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- byte model

def bytes_per_element(n_ranks: int):
    """Algorithmic HBM bytes per partition element of one step.
    reduce: N lp reads (2N) + f32 grad write (4); Adam: grad, master, m, v
    reads (16) + master, m, v writes (12) + lp param write (2)."""
    return {"reduce": 2 * n_ranks + 4, "adam": 30, "step": 2 * n_ranks + 34,
            "floor": 2 * n_ranks + 26}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_SOURCES = {"reduce_unscale_stats": "kernels.cu", "norm_decide": "kernels.cu",
                  "adam_fused_cast": "kernels.cu", "gather_layer_tma": "kernels.cu",
                  "gather_dequant": "quant.cu", "quantize_shard_blocks": "quant.cu"}


def source_hash(fname):
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "zero_partitioned_mixed_flat_gb300", "csrc", fname), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """Per-launch DRAM bytes (read + write) from the committed ncu summary,
    only while the kernel's source file is unchanged since the counters were
    taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload][kernel]
        if e.get("source_sha256_16") != source_hash(KERNEL_SOURCES[kernel]):
            return None
        return e.get("dram_bytes_per_launch")
    except Exception:
        return None


# ------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, enabled=True):
        self.proc = None
        self.enabled = enabled

    def start(self):
        if not self.enabled:
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        want = vis.split(",")[0].strip() if vis and vis.split(",")[0].strip().isdigit() else None
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        if want is not None:
            rows = [r for r in rows if r[0].strip() == want] or rows
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() in ("active", "1")})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- the step

class Run:
    """Buffers and calls of one workload on this GPU."""

    def __init__(self, w, part_ranks, dev):
        import torch
        import zero_partitioned_mixed_flat_gb300 as Z
        from zero_partitioned_mixed_flat_gb300 import synth
        self.torch, self.Z, self.synth = torch, Z, synth
        self.w = w
        self.dev = dev
        self.ranks = part_ranks
        self.plan = Z.ZeroPlan(-1, w.n_ranks, w.sizes, w.align, w.stage, w.unit_of_tensor, w.lp,
                               growth_interval=w.growth_interval)
        if w.reduce_lp_accum:
            self.plan.set_reduce_precision(1)
        P = self.P = self.plan.part_len
        self.S = w.loss_scale
        lpd = synth.LP_DTYPES[w.lp]
        self.slices, self.g, self.master, self.m, self.v, self.shard = {}, {}, {}, {}, {}, {}
        scale = self.S if w.grads_times_scale else 1.0
        for r in self.ranks:
            keep = self.plan.keep_ranges(r)
            sl = torch.empty((w.n_ranks, P), dtype=lpd, device=dev)
            for j in range(w.n_ranks):
                synth.normal_(sl[j], w.grad_std * scale, 0, 1, j, r, synth.KINDS["grad"])
                synth.zero_outside(sl[j], keep)
            self.slices[r] = sl
            self.g[r] = torch.empty(P, dtype=torch.float32, device=dev)
            self.master[r] = synth.master_init(P, w.master_std, 0, r, dev, keep)
            self.m[r] = torch.zeros(P, dtype=torch.float32, device=dev)
            self.v[r] = torch.zeros(P, dtype=torch.float32, device=dev)
            if w.stage == 3:
                self.shard[r] = torch.zeros(P, dtype=lpd, device=dev)
        self.param = None if w.stage == 3 else torch.zeros(self.plan.psi_padded, dtype=lpd,
                                                           device=dev)
        self.gather_shards = None
        self.quantized = bool(w.stage == 3 and w.gather and w.gather_quantized)
        if w.stage == 3 and w.gather:
            r0 = self.ranks[0]
            others = [synth.lp_shard(P, w.lp, w.master_std, 0, j, dev)
                      for j in range(w.n_ranks) if j != r0]
            self.gather_shards = others[:r0] + [self.shard[r0]] + others[r0:]
            biggest = max(self.plan.shard_len(u) for u in range(self.plan.n_units)) * w.n_ranks
            self.gather_out = torch.empty(biggest, dtype=lpd, device=dev)
            self.gather_out2 = torch.empty(biggest, dtype=lpd, device=dev)
            if self.quantized:
                # every rank's 1-byte codes (int8 or E4M3) + block scales
                # (ZeRO++-style gather); the other ranks quantize their shards once here
                self.plan.set_gather_quantization(w.quant_format)
                self.codes = [torch.empty(P, dtype=torch.int8, device=dev) for _ in range(w.n_ranks)]
                self.scales = [torch.empty(P // 128, dtype=torch.float32, device=dev)
                               for _ in range(w.n_ranks)]
                for j in range(w.n_ranks):
                    self.plan.quantize(self.gather_shards[j], self.codes[j], self.scales[j])
                del others
                self.gather_shards = [None] * w.n_ranks
        self.slice_lists = {r: [self.slices[r][j] for j in range(w.n_ranks)] for r in self.ranks}
        from zero_partitioned_mixed_flat_gb300.schedule import Hyper, StepBuffers, StepSchedule
        self.bufs = StepBuffers(
            ranks=self.ranks, slices=self.slice_lists, g=self.g, master=self.master, m=self.m,
            v=self.v, param=self.param, shard=self.shard, gather_shards=self.gather_shards,
            codes=getattr(self, "codes", None), scales=getattr(self, "scales", None),
            layer_bufs=[self.gather_out, self.gather_out2] if w.stage == 3 and w.gather else [],
            stats=torch.zeros(2 * w.n_ranks, dtype=torch.float64, device=dev))
        self.sched = StepSchedule(self.plan, self.bufs,
                                  Hyper(w.lr, w.beta1, w.beta2, w.eps, w.wd, int(w.adamw), w.clip),
                                  self.S, w.bucket_elems, gather=w.stage == 3 and w.gather,
                                  quantized=self.quantized)

    def set_group(self, group):
        """One job over several GPUs: this process's statistics are all-reduced
        over `group` before the decision."""
        self.bufs.group = group

    def calls(self, stream, slice_lists=None, side=None):
        """The step's ordered call list (zero_partitioned_mixed_flat_gb300.schedule)."""
        return self.sched.calls(stream, side=side, slice_lists=slice_lists)

    def tiles_per_part(self):
        return self.sched.tiles_per_partition()

    def launches_per_step(self):
        import torch
        return sum(c.launches for c in self.calls(torch.cuda.current_stream()))

    def gather_bytes_per_element(self):
        # lp gather: 2 B in + 2 B out; quantized: 1 B code + 4/128 B scale in, 2 B out
        return (3 + 4 / 128) if self.quantized else 4

    def bytes_per_step(self):
        import torch
        return int(sum(c.nbytes for c in self.calls(torch.cuda.current_stream())))


def dist_setup(n_gpus, backend="nccl", force=False):
    """(world size, rank, device index, torch.distributed or None).  One process
    per GPU; with fewer visible GPUs than local ranks (a gloo run of several
    processes on one GPU) the ranks share devices round-robin.  force: a
    process group even for a world of one (outside torchrun: 127.0.0.1 on a
    free port)."""
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1 or force:
        import socket
        import torch.distributed as dist
        if "MASTER_PORT" not in os.environ:
            with socket.socket() as s:
                s.bind(("127.0.0.1", 0))
                os.environ["MASTER_PORT"] = str(s.getsockname()[1])
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("RANK", str(rank))
        os.environ.setdefault("WORLD_SIZE", str(ws))
        dev = local % max(1, torch.cuda.device_count())
        torch.cuda.set_device(dev)
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", dev))
        else:
            dist.init_process_group(backend)
        return ws, rank, dev, dist
    torch.cuda.set_device(0)
    return 1, 0, 0, None


def host_threads():
    return max(1, min(os.cpu_count() or 1, 64))


class OracleSample:
    """The oracle as it stands over a sample of one partition, split into T
    contiguous chunks run on T host threads (the oracle's C calls release the
    GIL): per step every chunk is reduced, the chunks' sums of squares are
    added in chunk order for the one decision, then every chunk is updated."""

    def __init__(self, w, slices, master, loss_scale, threads):
        import numpy as np
        from concurrent.futures import ThreadPoolExecutor
        self.w, self.S = w, loss_scale
        M = slices[0].size
        T = max(1, min(threads, M // 4096))
        bounds = [(M * i // T) // 8 * 8 for i in range(T)] + [M]
        self.chunks = [(bounds[i], bounds[i + 1]) for i in range(T) if bounds[i + 1] > bounds[i]]
        self.slices = slices
        self.master = master
        self.m = np.zeros(M, np.float32)
        self.v = np.zeros(M, np.float32)
        self.g = np.empty(M, np.float32)
        self.step_no = self.good = 0
        self.pool = ThreadPoolExecutor(len(self.chunks))
        self.threads = len(self.chunks)

    def step(self):
        import oracle
        w = self.w

        def red(c):
            c0, c1 = c
            _, ss, of = oracle.reduce([s[c0:c1] for s in self.slices], w.lp, self.S,
                                      out=self.g[c0:c1])
            return ss, of
        parts = list(self.pool.map(red, self.chunks))
        ss, of = 0.0, 0
        for p_ss, p_of in parts:
            ss += p_ss
            of |= p_of
        d = oracle.decide(ss, of, w.clip, self.S, self.step_no, self.good, w.growth_interval,
                          w.beta1, w.beta2)

        def upd(c):
            c0, c1 = c
            oracle.adam(self.g[c0:c1], self.master[c0:c1], self.m[c0:c1], self.v[c0:c1], w.lp,
                        d["coef"], d["skip"], w.lr, w.beta1, w.beta2, w.eps, w.wd, int(w.adamw),
                        d["bc1"], d["bc2"])
        list(self.pool.map(upd, self.chunks))
        self.step_no, self.good = d["step"], d["good_steps"]

    def close(self):
        self.pool.shutdown()


def cpu_baseline(run, seconds):
    """The oracle as it stands on a bounded sample of the same workload (the
    first M elements of the first simulated partition, all N slices), on all
    host cores."""
    from zero_partitioned_mixed_flat_gb300 import synth
    w = run.w
    r = run.ranks[0]
    T = host_threads()
    # up to 2^20 elements per thread, at most 512 MB of slices on the host
    M = min(run.P, T << 20, (256 << 20) // w.n_ranks)
    M -= M % 8
    if M == 0:
        return None
    sl = [synth.to_numpy_codes(run.slices[r][j, :M]) for j in range(w.n_ranks)]
    o = OracleSample(w, sl, run.master[r][:M].cpu().numpy().copy(), run.S, T)
    reps, t0 = 0, time.perf_counter()
    while True:
        o.step()
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or el >= 30.0:
            break
    o.close()
    return {"value": M * reps / el, "unit": UNIT, "cores": o.threads, "kind": "oracle",
            "sample": "first %d elements of partition %d (all %d slices): reduce + decide + "
                      "Adam, %d repetitions, %.1f s, %d host threads over contiguous chunks"
                      % (M, r, w.n_ranks, reps, el, o.threads)}


def run_reference(args):
    """Baseline arm: the CPU oracle, as it stands, timed per step on a bounded
    sample of the workload (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from zero_partitioned_mixed_flat_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    lay = oracle.layout(w.sizes, w.n_ranks, w.align, w.stage, w.unit_of_tensor)
    P = lay["part_len"]
    T = host_threads()
    M = min(P, T << 20, (256 << 20) // w.n_ranks)
    M -= M % 8
    rng = np.random.default_rng(0)
    scale = w.loss_scale if w.grads_times_scale else 1.0
    vals = (rng.standard_normal((w.n_ranks, M)) * w.grad_std * scale).astype(np.float32)
    if w.lp == 0:
        sl = list(vals.astype(np.float16).view(np.uint16))
    else:
        sl = list(oracle.float_to_lp(vals, 1).reshape(w.n_ranks, M))
    master = (rng.standard_normal(M) * w.master_std).astype(np.float32)
    o = OracleSample(w, sl, master, w.loss_scale, T)
    for _ in range(args.warmup):
        o.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.step()
    el = time.perf_counter() - t0
    o.close()
    value = M * args.steps / el
    sample = ("%d of the %d elements of one partition, all %d slices, per step "
              "(reduce + decide + Adam), %d host threads over contiguous chunks"
              % (M, P, w.n_ranks, o.threads))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "sample_elements": M, "part_len": P,
                       "n_ranks": w.n_ranks, "stage": w.stage},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": o.threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    emit(line)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import zero_partitioned_mixed_flat_gb300 as Z
    from zero_partitioned_mixed_flat_gb300.workloads import WORKLOADS
    Z.load()
    ws, rank, local, dist = dist_setup(args.gpus, args.dist_backend, force=args.one_job)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    if args.n_ranks:
        import dataclasses
        w = dataclasses.replace(w, n_ranks=args.n_ranks, ranks=[0],
                                name="%s-n%d" % (w.name, args.n_ranks))
    if args.reduce_in_lp:
        import dataclasses
        w = dataclasses.replace(w, reduce_lp_accum=True)
    if args.quantized_gather or args.quant_format:
        import dataclasses
        w = dataclasses.replace(w, gather_quantized=True)
        if args.quant_format:
            w = dataclasses.replace(w, quant_format=int(args.quant_format == "fp8"))
    # weak scaling: every GPU owns as many partitions as one GPU does.  When
    # the GPUs' partitions fit in the job without overlap (rank-r configs),
    # they form one job: GPU k owns partitions k*len .. (k+1)*len - 1 and the
    # step's statistics are all-reduced before the decision.  Otherwise
    # (configs that update every partition on one GPU) each GPU runs its own
    # replica of the job.
    per = len(w.ranks)
    one_job = (ws > 1 or args.one_job) and ws * per <= w.n_ranks
    if one_job:
        part_ranks = [rank * per + i for i in range(per)]
    else:
        part_ranks = [(r + rank) % w.n_ranks for r in w.ranks]
    t_setup = time.perf_counter()
    run = Run(w, part_ranks, dev)
    if one_job:
        run.set_group(dist.group.WORLD)
    torch.cuda.synchronize()
    log("setup %.1f s: workload %s, P=%d, N=%d, partitions %s" %
        (time.perf_counter() - t_setup, w.name, run.P, w.n_ranks, part_ranks))
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)

    side = torch.cuda.Stream() if (run.gather_shards is not None and not args.no_overlap) else None
    calls = run.calls(stream, side=side)
    timed_calls = [c for c in calls if c.kind != "wait"]
    kinds = sorted({c.kind for c in timed_calls})

    def step(evs=None):
        i = 0
        for c in calls:
            if c.kind == "wait":
                c.fn()
                continue
            if evs is not None:
                evs[i][0].record(c.stream)
            c.fn()
            if evs is not None:
                evs[i][1].record(c.stream)
            i += 1

    # a step that touches less than a few L2 sizes is timed step by step with a
    # 256 MB write between steps (outside the step's events) to flush the L2
    flush = None
    if run.bytes_per_step() < L2_FLUSH_BELOW:
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    K = args.steps
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in timed_calls] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(enabled=not args.no_clocks)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3 if not args.no_clocks else 0.0)
    # the timed steps: no event between a step's calls (an event record between
    # two kernels costs their programmatic-launch overlap); with the L2 flush,
    # one event pair per step keeps the flush out of the step's time
    start.record(stream)
    for k in range(K):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(float(k))
            step_ev[k][0].record(stream)
        step()
        if side is not None:
            stream.wait_stream(side)
        if flush is not None:
            step_ev[k][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    total_ms = (sum(a.elapsed_time(b_) for a, b_ in step_ev) if flush is not None
                else start.elapsed_time(end))
    if dist:
        t = torch.tensor([total_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    res = run.plan.result()
    if res["skipped"]:
        log("warning: a timed step was skipped (overflow)")
    # per-kind times: K more steps, now with an event pair around every call
    kstart = torch.cuda.Event(enable_timing=True)
    kstart.record(stream)
    for k in range(K):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.fill_(float(k))
        step(evs[k])
        if side is not None:
            stream.wait_stream(side)
    torch.cuda.synchronize()
    # per kind: time per step (sum of its calls), bytes per step, launches per step
    # time per kind and step = the union of its calls' intervals (calls of one
    # kind may overlap when gathers are prefetched on the second stream)
    t_kind = {k: 0.0 for k in kinds}
    for e in evs:
        spans = {k: [] for k in kinds}
        for i, c in enumerate(timed_calls):
            spans[c.kind].append((kstart.elapsed_time(e[i][0]), kstart.elapsed_time(e[i][1])))
        for k, iv in spans.items():
            iv.sort()
            cur0, cur1 = iv[0]
            for a, b_ in iv[1:]:
                if a > cur1:
                    t_kind[k] += cur1 - cur0
                    cur0, cur1 = a, b_
                else:
                    cur1 = max(cur1, b_)
            t_kind[k] += cur1 - cur0
    t_kind = {k: v / K for k, v in t_kind.items()}
    b_kind = {k: sum(c.nbytes for c in timed_calls if c.kind == k) for k in kinds}
    n_kind = {k: sum(1 for c in timed_calls if c.kind == k) for k in kinds}
    ms_per_step = total_ms / K
    graph_info = None
    if args.graph and run.bufs.group is not None:
        log("--graph: not taken with the multi-GPU exchange (its collective is not captured here)")
        args.graph = False
    if args.graph:
        # the same call list captured once into a CUDA graph and replayed K
        # times: the launches cost no host time; per-kind times stay the eager ones
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            gcalls = run.calls(cap, side=None)
            with torch.cuda.graph(g, stream=cap):
                for c in gcalls:
                    if c.kind != "wait":
                        c.fn()
        stream.wait_stream(cap)
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        gms = 0.0
        with torch.cuda.stream(stream):
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for k in range(K):
                if flush is not None:
                    flush.fill_(float(k))
                    step_ev[k][0].record(stream)
                g.replay()
                if flush is not None:
                    step_ev[k][1].record(stream)
            g1.record(stream)
            torch.cuda.synchronize()
        gms = (sum(a.elapsed_time(b_) for a, b_ in step_ev) if flush is not None
               else g0.elapsed_time(g1))
        if dist:
            t = torch.tensor([gms], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            gms = float(t.item())
        graph_info = {"eager_ms_per_step": ms_per_step, "graph_ms_per_step": gms / K}
        ms_per_step = gms / K
    elems = run.P * len(run.ranks)
    value = elems * ws / (ms_per_step / 1e3)
    peak, peak_kind = load_peaks()
    b = bytes_per_element(w.n_ranks)
    # dominant kernel = the one with the largest share of the step
    dom = max(t_kind, key=t_kind.get)
    kname = {"reduce": "reduce_unscale_stats", "adam": "adam_fused_cast", "decide": "norm_decide",
             "gather": "gather_dequant" if run.quantized else "gather_layer_tma",
             "quantize": "quantize_shard_blocks", "exchange": "norm_decide"}[dom]
    achieved = b_kind[dom] / (t_kind[dom] / 1e3) / 1e9
    step_gbs = run.bytes_per_step() / (ms_per_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": traffic_for(kname, w.name),
                "algorithmic_bytes_per_launch": b_kind[dom] / n_kind[dom],
                "avg_launch_ms": t_kind[dom] / n_kind[dom],
                "launches_per_step": n_kind[dom]}
    kernels = {k: {"calls_per_step": n_kind[k], "avg_ms": t_kind[k] / n_kind[k],
                   "ms_per_step": t_kind[k], "share": t_kind[k] / ms_per_step,
                   "GBps": b_kind[k] / (t_kind[k] / 1e3) / 1e9,
                   "frac_of_peak": b_kind[k] / (t_kind[k] / 1e3) / 1e9 / peak}
               for k in kinds}

    # ---- end to end through the ABI, host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(run, args.e2e_steps, stream, side, ws, dist, dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(run, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": w.name + ("-fp8" if run.quantized and w.quant_format and
                                                  not w.name.endswith("fp8") else ""),
                           "psi": int(sum(w.sizes)),
                           "n_ranks": w.n_ranks, "stage": w.stage,
                           "lp": ["fp16", "bf16"][w.lp], "part_len": run.P,
                           "reduce_dtype": ["fp32", "lp"][int(w.reduce_lp_accum)],
                           "partitions_per_gpu": len(run.ranks),
                           "bucket_elems": w.bucket_elems,
                           "gather_prefetch_streams": 2 if side is not None else (
                               1 if run.gather_shards is not None else 0),
                           "l2": ("L2 flushed between timed steps (%d MB write outside the "
                                  "step's events; %.1f MB touched per step)"
                                  % (L2_FLUSH_BYTES >> 20, run.bytes_per_step() / 1e6))
                                 if flush is not None else
                                 "inputs larger than L2 (%.1f GB touched per step vs 129 MB L2)"
                                 % (run.bytes_per_step() / 1e9),
                           "parallelism": ("dp%d job over %d GPUs: GPU k owns partitions %s of "
                                           "it, step statistics all-reduced (%s) before the "
                                           "decision; the other ranks' slices simulated on each "
                                           "GPU" % (w.n_ranks, ws, "k" if per == 1 else
                                                    "k*%d..k*%d+%d" % (per, per, per - 1),
                                                    dist.get_backend()))
                                          if run.bufs.group is not None else
                                          ("dp%d simulated on each GPU (ranks as device buffers)"
                                           % w.n_ranks) + (", one replica per GPU" if ws > 1 else "")},
                "step_hbm_gbs": step_gbs, "step_frac_of_peak": step_gbs / peak,
                "step_frac_of_nominal_8tbs": step_gbs / 8000.0,
                "bytes_per_element": b, "roofline": roofline, "kernels": kernels,
                "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "gpu_launches": run.launches_per_step() * K,
                "decision": res, "graph": graph_info}
        emit(line)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    run.plan.close()
    return 0


def host_mem_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def measure_e2e(run, steps, stream, side, ws, dist, dev):
    """Same metric through the public API with the step's gradient slices in
    pinned host memory, timed end to end on the host clock, every step ending
    with a synchronising device->host read of the step result.

    Two ways in: "direct" hands the pinned host slices to zero_reduce_partition,
    whose kernel reads them in place over NVLink-C2C (no staging buffer);
    "staged" first copies them host->device (one cudaMemcpyAsync per
    partition) and reduces from device memory.  The faster is reported as the
    e2e value; both are listed."""
    import torch
    torch.cuda.synchronize()
    need = sum(int(t.numel()) * t.element_size() for t in run.slices.values())
    avail = host_mem_available()
    if avail is not None:
        # the processes of this node share its memory
        avail //= max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))
    ok = avail is None or need * 2 <= avail
    if dist:  # every rank takes the same branch (the timed part has collectives)
        flag = torch.tensor([1.0 if ok else 0.0], device=dev, dtype=torch.float64)
        dist.all_reduce(flag, op=dist.ReduceOp.MIN)
        ok = bool(flag.item() > 0)
    if not ok:
        log("e2e skipped: %.1f GB of host buffers needed per process, %s GB available"
            % (need / 1e9, "%.1f" % (avail / 1e9) if avail is not None else "?"))
        return {"value": None, "unit": UNIT, "skipped": "host memory: %.1f GB needed per process"
                % (need / 1e9)}
    host = {}
    try:
        for r in run.ranks:
            host[r] = torch.empty(run.slices[r].shape, dtype=run.slices[r].dtype, pin_memory=True)
            host[r].copy_(run.slices[r])
        pinned = True
    except RuntimeError:
        host = {r: run.slices[r].cpu() for r in run.ranks}
        pinned = False
    h2d = sum(int(t.numel()) * t.element_size() for t in host.values())
    host_lists = {r: [host[r][j] for j in range(run.w.n_ranks)] for r in run.ranks}

    staged_calls = run.calls(stream, side=side)
    direct_calls = run.calls(stream, slice_lists=host_lists, side=side)

    def staged():
        for r in run.ranks:
            run.slices[r].copy_(host[r], non_blocking=True)
        for c in staged_calls:
            c.fn()
        return run.plan.result()          # synchronises and reads the record

    def direct():
        for c in direct_calls:
            c.fn()
        return run.plan.result()

    def timed(fn):
        fn()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            fn()
        el = time.perf_counter() - t0
        if dist:
            t = torch.tensor([el], device=dev, dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            el = float(t.item())
        return run.P * len(run.ranks) * ws * steps / el, el / steps * 1e3

    modes = {}
    modes["staged"] = timed(staged)
    if pinned:
        try:
            modes["direct"] = timed(direct)
        except Exception as e:   # the device cannot read this host memory
            log("e2e direct mode unavailable: %s" % e)
    del host, host_lists
    best = max(modes, key=lambda k: modes[k][0])
    return {"value": modes[best][0], "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": 64, "pinned": pinned, "steps": steps,
            "ms_per_step": modes[best][1], "mode": best,
            "modes": {k: {"value": v, "ms_per_step": ms} for k, (v, ms) in modes.items()}}


if __name__ == "__main__":
    sys.exit(main())
