"""The benchmark's own arm prints one JSON line with every key of its
contract, on a small workload (GB300)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("extra", [[], ["--graph"]])
def test_bench_json_line(zlib, extra):
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny-zero1", "--steps", "4",
                        "--warmup", "3", "--cpu-seconds", "0.5", "--e2e-steps", "2"] + extra,
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3 and d["value"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny-zero1" and "flushed" in d["config"]["l2"]
    rf = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rf, k
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["achieved"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # per step: one reduce launch for the 4 partitions, the decision, one Adam launch
    assert d["gpu_launches"] == 4 * 3
    assert set(d["kernels"]) == {"reduce", "decide", "adam"}
    if extra:
        assert d["graph"]["graph_ms_per_step"] == d["ms_per_step"]


def test_bench_one_job_over_two_ranks(zlib):
    # the multi-GPU path of the benchmark (one job, the per-partition statistics
    # all-reduced before every decision), run as two gloo ranks sharing this
    # GPU: the same code as under nccl on two GPUs except the exchange backend
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--workload", "gpt2-xl-zero2", "--steps", "3", "--warmup", "3", "--no-cpu-baseline",
           "--e2e-steps", "2", "--no-clocks", "--dist-backend", "gloo"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                       # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["value"] > 0 and d["scaling"] == "weak"
    assert "job over 2 GPUs" in d["config"]["parallelism"]
    assert d["config"]["partitions_per_gpu"] == 1
    # per step: the reduce, the statistics export, the decision, Adam
    assert d["gpu_launches"] == 3 * 4
    assert "exchange" in d["kernels"] and d["e2e"]["value"] > 0
    assert d["decision"]["skipped"] == 0 and d["decision"]["step"] == 3 + 3   # warm-up + timed


def test_bench_one_job_nccl_world_of_one(zlib):
    # the multi-GPU step's nccl exchange (statistics exported, all-reduced by
    # nccl, decided from the sum) in a world of one process: the decision must
    # be the one the local path takes, bit for bit, at one launch more per step
    def bench(*extra):
        cmd = [sys.executable, "bench.py", "--workload", "gpt2-xl-zero2", "--steps", "3", "--warmup",
               "3", "--no-cpu-baseline", "--no-e2e", "--no-clocks"] + list(extra)
        env = {k: v for k, v in os.environ.items()
               if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
        r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
        assert r.returncode == 0, r.stderr[-3000:]
        lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
        assert len(lines) == 1
        assert r.stdout.strip().splitlines()[-1] == lines[0]   # nccl's banner comes before it
        return json.loads(lines[0])

    local, job = bench(), bench("--one-job", "--dist-backend", "nccl")
    assert "job over 1 GPUs" in job["config"]["parallelism"] and "(nccl)" in job["config"]["parallelism"]
    assert job["n_gpus"] == 1 and job["value"] > 0
    assert "exchange" in job["kernels"] and "exchange" not in local["kernels"]
    assert local["gpu_launches"] == 3 * 3 and job["gpu_launches"] == 3 * 4
    assert job["decision"] == local["decision"]
    assert job["decision"]["step"] == 3 + 3
