"""The allocation-free reduce (zero_reduce_partition_noalloc).

Some callers cannot allocate device memory: a framework whose caching
allocator already owns the whole GPU (an extra cudaMalloc would fail or
fragment its pool), or a loop that must not pay cudaMalloc's implicit
synchronisation.  This entry point keeps its scratch in a fixed array inside
the library image instead of plan-owned memory.  These tests call it through
the C ABI and check, on several calls in a row that share that array (a later
call must not see an earlier call's overflow word or partial sums):
  - the reduced gradient and the overflow flag against the CPU oracle, bit for
    bit, and the sum of squares within 1e-6 of the oracle's sequential sum;
  - the sum of squares against the plan-based path's exported statistic for
    the same partition, bit for bit (both add the tile partials with the same
    fixed tree);
  - that a warm call allocates nothing: the device's free memory and torch's
    allocated bytes are unchanged across it;
and that sizes beyond the stated maximum are refused.  This file is collected
last on purpose.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import zero_partitioned_mixed_flat_gb300 as Z
from zero_partitioned_mixed_flat_gb300 import synth

TILE = Z.ZERO_NORM_TILE


def _plan_reduce(n, lp, slices, part, scale):
    plan = Z.ZeroPlan(n * part, n, None, 8, 2, None, lp)
    g = torch.empty(part, dtype=torch.float32, device="cuda")
    plan.reduce(0, slices, g, scale)
    stats = torch.empty(2 * n, dtype=torch.float64, device="cuda")
    plan.partition_stats(stats)
    torch.cuda.synchronize()
    plan.close()
    st = stats.cpu().numpy()
    return g, float(st[0]), int(st[n] != 0)


def _same_floats(a, b):
    eq = a.view(np.uint32) == b.view(np.uint32)
    return bool(np.all(eq | (np.isnan(a) & np.isnan(b))))


@pytest.mark.gpu
def test_noalloc_reduce_matches_the_oracle_and_the_plan_path(zlib):
    dev = torch.device("cuda")
    ss_out = torch.empty(1, dtype=torch.float64, device=dev)
    of_out = torch.empty(1, dtype=torch.int32, device=dev)
    # (N, len, lp, loss scale, injected +inf at (slice, index) or None):
    # 16 bf16 slices over 5 tiles + a ragged tail with an overflow; then 5 fp16
    # slices, fewer tiles, finite (must not inherit the overflow or the tail
    # tiles' partials); then one tile + 8 elements (the ragged last tile); then
    # 4097 tiles (two chunks of the fixed tree)
    calls = [(16, 5 * TILE + 136, 1, 1.0, (3, 4321)),
             (5, 2 * TILE + 64, 0, 1024.0, None),
             (3, TILE + 8, 1, 1.0, None),
             (2, 4097 * TILE + 16, 0, 256.0, None)]
    for k, (n, part, lp, scale, inject) in enumerate(calls):
        slices = [synth.grad_slice(part, lp, 1e-3, scale, 11, k, j, 0, dev) for j in range(n)]
        if inject is not None:
            slices[inject[0]][inject[1]] = float("inf")
        g = torch.full((part,), 7.0, dtype=torch.float32, device=dev)
        Z.zero_reduce_partition_noalloc(n, lp, slices, part, scale, g, ss_out, of_out)
        torch.cuda.synchronize()
        got_g = g.cpu().numpy()
        ss, of = float(ss_out.item()), int(of_out.item())
        og, oss, oof = oracle.reduce([synth.to_numpy_codes(t) for t in slices], lp, scale)
        assert _same_floats(got_g, og), k
        assert of == oof == (1 if inject is not None else 0), k
        if oof:
            assert not math.isfinite(ss)
        else:
            assert abs(ss - oss) <= 1e-6 * oss, (k, ss, oss)
        g_ref, ss_ref, of_ref = _plan_reduce(n, lp, slices, part, scale)
        assert _same_floats(got_g, g_ref.cpu().numpy()), k
        assert of == of_ref, k
        assert np.float64(ss).tobytes() == np.float64(ss_ref).tobytes(), (k, ss, ss_ref)


@pytest.mark.gpu
def test_noalloc_warm_call_allocates_nothing(zlib):
    dev = torch.device("cuda")
    n, part = 4, 3 * TILE + 24
    slices = [synth.grad_slice(part, 0, 1e-3, 64.0, 12, 1, j, 0, dev) for j in range(n)]
    g = torch.empty(part, dtype=torch.float32, device=dev)
    ss_out = torch.empty(1, dtype=torch.float64, device=dev)
    of_out = torch.empty(1, dtype=torch.int32, device=dev)
    # the first call may load the library's device code (module loading is lazy)
    Z.zero_reduce_partition_noalloc(n, 0, slices, part, 64.0, g, ss_out, of_out)
    torch.cuda.synchronize()
    first = (g.clone(), ss_out.clone())
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    Z.zero_reduce_partition_noalloc(n, 0, slices, part, 64.0, g, ss_out, of_out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert torch.equal(g, first[0]) and torch.equal(ss_out, first[1])


def test_noalloc_refuses_sizes_beyond_its_maximum():
    from zero_partitioned_mixed_flat_gb300 import build
    build.build()
    Z.load()
    assert Z.ZERO_NOALLOC_MAX_ELEMS == 65536 * TILE
    buf = 1 << 20   # never dereferenced: the size check comes first
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_reduce_partition_noalloc(2, 0, [buf, buf], Z.ZERO_NOALLOC_MAX_ELEMS + 8, 1.0,
                                        buf, buf, buf, stream=0)
    assert e.value.code == Z.ZERO_EINVAL
    assert "ZERO_NOALLOC_MAX_ELEMS" in Z.zero_last_error()
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_reduce_partition_noalloc(2, 0, [buf, buf + 4], 64, 1.0, buf, buf, buf, stream=0)
    assert e.value.code == Z.ZERO_EALIGN
