"""The allocation-free reduce (zero_reduce_partition_noalloc).

It is for callers that cannot allocate device memory (a framework whose
caching allocator owns the whole GPU, or a loop that must not pay
cudaMalloc's implicit synchronisation): its scratch is a fixed array in the
library image instead of plan-owned memory.  These tests check, through the C
ABI, that it gives what the plan-based zero_reduce_partition gives, on two
calls in a row that share that array (the second call must not see the first
call's overflow word or partial sums), and that sizes beyond its stated
maximum are refused.  This file is collected last on purpose.
"""
import math

import numpy as np
import pytest
import torch

import zero_partitioned_mixed_flat_gb300 as Z
from zero_partitioned_mixed_flat_gb300 import synth

TILE = 32768


def _plan_reduce(n, lp, slices, part, scale):
    plan = Z.ZeroPlan(n * part, n, None, 8, 2, None, lp)
    g = torch.empty(part, dtype=torch.float32, device="cuda")
    plan.reduce(0, slices, g, scale)
    ss, of = plan.stats()
    plan.close()
    return g, ss, of


def _same_floats(a, b):
    a, b = a.cpu().numpy(), b.cpu().numpy()
    eq = a.view(np.uint32) == b.view(np.uint32)
    return bool(np.all(eq | (np.isnan(a) & np.isnan(b))))


@pytest.mark.gpu
def test_noalloc_reduce_matches_the_plan_reduce_on_two_calls_in_a_row(zlib):
    dev = torch.device("cuda")
    ss_out = torch.empty(1, dtype=torch.float64, device=dev)
    of_out = torch.empty(1, dtype=torch.int32, device=dev)
    # call 1: 16 bf16 slices, 5 tiles + ragged tail, with an injected +inf;
    # call 2: 5 fp16 slices, fewer tiles, finite -- must not inherit call 1's state
    calls = [(16, 5 * TILE + 136, 1, 1.0, (3, 4321)),
             (5, 2 * TILE + 64, 0, 1024.0, None)]
    for k, (n, part, lp, scale, inject) in enumerate(calls):
        slices = [synth.grad_slice(part, lp, 1e-3, scale, 11, k, j, 0, dev) for j in range(n)]
        if inject is not None:
            slices[inject[0]][inject[1]] = float("inf")
        g = torch.full((part,), 7.0, dtype=torch.float32, device=dev)
        Z.zero_reduce_partition_noalloc(n, lp, slices, part, scale, g, ss_out, of_out)
        torch.cuda.synchronize()
        g_ref, ss_ref, of_ref = _plan_reduce(n, lp, slices, part, scale)
        assert _same_floats(g, g_ref), k
        assert int(of_out.item()) == of_ref == (1 if inject is not None else 0), k
        ss = float(ss_out.item())
        if of_ref:
            assert not math.isfinite(ss) and not math.isfinite(ss_ref)
        else:
            assert abs(ss - ss_ref) <= 1e-6 * ss_ref, (ss, ss_ref)


def test_noalloc_refuses_sizes_beyond_its_maximum():
    from zero_partitioned_mixed_flat_gb300 import build
    build.build()
    Z.load()
    buf = 1 << 20   # never dereferenced: the size check comes first
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_reduce_partition_noalloc(2, 0, [buf, buf], Z.ZERO_NOALLOC_MAX_ELEMS + 8, 1.0,
                                        buf, buf, buf, stream=0)
    assert e.value.code == Z.ZERO_EINVAL
    assert "ZERO_NOALLOC_MAX_ELEMS" in Z.zero_last_error()
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_reduce_partition_noalloc(2, 0, [buf, buf + 4], 64, 1.0, buf, buf, buf, stream=0)
    assert e.value.code == Z.ZERO_EALIGN
