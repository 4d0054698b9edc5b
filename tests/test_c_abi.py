"""The ABI from plain C (CPU only): a C11 program compiled against
include/zero.h and linked to libzero.so creates plans, reads their layout
(stage-3 unit shards included) and the memory report, checks the exchange
calls' state errors, and destroys the plans; the values must be the oracle's."""
import os
import subprocess
import tempfile

import pytest

import oracle
from zero_partitioned_mixed_flat_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "zero.h"

int main(void) {
    const int64_t sizes[3] = {1000, 24, 70000};
    zero_plan *plan = NULL;
    if (zero_plan_create(-1, 8, sizes, 3, 128, 2, NULL, ZERO_BF16, &plan) != ZERO_OK) {
        printf("create failed: %s\n", zero_last_error());
        return 1;
    }
    int64_t psi_p = 0, part = 0, offs[3];
    if (zero_plan_query(plan, &psi_p, &part, offs) != ZERO_OK) return 2;
    printf("%lld %lld %lld %lld %lld\n", (long long)psi_p, (long long)part,
           (long long)offs[0], (long long)offs[1], (long long)offs[2]);
    zero_plan_destroy(plan);
    double formula[4];
    int64_t actual[4], comm[4];
    if (zero_memory_report(7500000000LL, 64, 128, formula, actual, comm) != ZERO_OK) return 3;
    for (int k = 0; k < 4; ++k) printf("%.17g %lld %lld\n", formula[k], (long long)actual[k], (long long)comm[k]);
    if (zero_plan_create(-1, 0, sizes, 3, 128, 2, NULL, ZERO_BF16, &plan) != ZERO_EINVAL) return 4;
    printf("%s\n", zero_last_error()[0] ? "error-message" : "no-message");
    /* a stage-3 plan: each unit's shard, and the exchange calls out of order */
    const int32_t units[3] = {0, 0, 1};
    if (zero_plan_create(-1, 4, sizes, 3, 8, 3, units, ZERO_FP16, &plan) != ZERO_OK) return 5;
    int64_t shard_len[2], shard_off[2];
    if (zero_plan_unit_shards(plan, shard_len, shard_off) != ZERO_OK) return 6;
    printf("%lld %lld %lld %lld\n", (long long)shard_len[0], (long long)shard_len[1],
           (long long)shard_off[0], (long long)shard_off[1]);
    double stats[8];
    if (zero_partition_stats(plan, stats, NULL) != ZERO_ESTATE) return 7;
    if (zero_step_set_global_stats(plan, stats) != ZERO_ESTATE) return 8;
    zero_plan_destroy(plan);
    return 0;
}
"""


def test_c_program_uses_the_abi():
    lib = build.build()
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "use_zero.c")
        exe = os.path.join(tmp, "use_zero")
        with open(src, "w") as f:
            f.write(PROGRAM)
        libdir = os.path.dirname(lib)
        r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                            src, "-o", exe, "-L", libdir, "-lzero", "-Wl,-rpath," + libdir],
                           capture_output=True, text=True)
        if r.returncode != 0 and "cannot find -lzero" in r.stderr:
            pytest.skip("libzero.so not linkable as -lzero here")
        assert r.returncode == 0, r.stderr
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert out.returncode == 0, out.stdout + out.stderr
        lines = out.stdout.split("\n")
    lay = oracle.layout([1000, 24, 70000], 8, 128, 2)
    first = [int(x) for x in lines[0].split()]
    assert first == [lay["psi_padded"], lay["part_len"]] + list(lay["tensor_offsets"])[:3]
    formula, actual, comm = oracle.memory(7500000000, 64, 128)
    for k in range(4):
        f, a, c = lines[1 + k].split()
        assert float(f) == formula[k] and int(a) == actual[k] and int(c) == comm[k]
    assert lines[5] == "error-message"
    lay3 = oracle.layout([1000, 24, 70000], 4, 8, 3, [0, 0, 1])
    shard = [int(x) // 4 for x in lay3["unit_padded"]]
    assert [int(x) for x in lines[6].split()] == shard + [0, shard[0]]
