"""The pins must catch plausible mistakes in the oracle (CPU only).

Each case plants one mistake in a temporary copy of the oracle's C source
(a wrong sign, a dropped term, a transposed index, a misplaced eps, ...),
compiles it, and runs the pin suite against it: the suite has to fail.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

MUTANTS = {
    "reduce_minus": ("s = s + orc_lp_to_float(slices[j][i], lp);",
                     "s = s - orc_lp_to_float(slices[j][i], lp);"),
    "reduce_sum_not_mean": ("(double)loss_scale * (double)n", "(double)loss_scale"),
    "reduce_double_counts_rank0": ("for (int32_t j = 1; j < n; ++j)",
                                   "for (int32_t j = 0; j < n; ++j)"),
    "reduce_flag_on_g_inf_only": ("if (!isfinite(s))", "if (isinf(s))"),
    "sumsq_of_abs": ("sq = gi * gi;", "sq = gi < 0 ? -gi : gi;"),
    "skip_keeps_scale": ("fmaxf(loss_scale * 0.5f, 1.0f)", "loss_scale"),
    "skip_advances_step": ("        out->new_scale = growth_interval > 0 ? fmaxf",
                           "        t = step + 1;\n        out->new_scale = growth_interval > 0 ? fmaxf"),
    "no_bias_correction_m": ("mhat = mi / bc1;", "mhat = mi;"),
    "no_bias_correction_v": ("vhat = vi / bc2;", "vhat = vi;"),
    "eps_inside_sqrt": ("denom = sqrtf(vhat) + eps;", "denom = sqrtf(vhat + eps);"),
    "betas_swapped": ("mi = beta1 * m[i] + omb1 * gi;", "mi = beta2 * m[i] + omb2 * gi;"),
    "v_not_squared": ("vi = beta2 * v[i] + omb2 * (gi * gi);", "vi = beta2 * v[i] + omb2 * gi;"),
    "l2_wrong_sign": ("gi = gi + wd * w;", "gi = gi - wd * w;"),
    "no_decoupled_decay": ("w = w * decay;", "w = w;"),
    "coef_ignored": ("float gi = g[i] * coef;", "float gi = g[i];"),
    "update_sign": ("w = w - upd;", "w = w + upd;"),
    "pad_to_align_only": ("quantum = (int64_t)n_ranks * align;", "quantum = align;"),
    "partition_offset_off_by_one": ("int64_t start = unit_offsets[u] + (stage == 0 ? 0 : rank * shard);",
                                    "int64_t start = unit_offsets[u] + (stage == 0 ? 0 : rank * shard) + (k > 0);"),
    "gather_transposed": ("out[(int64_t)j * shard_len + k] = shards[j][k];",
                          "out[k * n + j] = shards[j][k];"),
    "half_ties_away": ("n = nearbyint(a / q);", "n = round(a / q);"),
    "memory_stage2_k": ("int_plus_ratio(2 * psi, 14 * psi, n_ranks)",
                        "int_plus_ratio(2 * psi, 12 * psi, n_ranks)"),
    "comm_stage3": ("comm[3] = 3 * psi;", "comm[3] = 2 * psi;"),
    "quant_scale_255": ("scale = amax / 127.0f;", "scale = amax / 255.0f;"),
    "quant_truncates": ("r = nearbyintf(orc_lp_to_float(x[b0 + k], lp) / scale);",
                        "r = truncf(orc_lp_to_float(x[b0 + k], lp) / scale);"),
    "dequant_wrong_block": ("scales[j][k / block]", "scales[j][k / block / 2]"),
    "e4m3_bias_8": ("mag = ldexpf((float)(8 + m), e - 10);", "mag = ldexpf((float)(8 + m), e - 11);"),
    "e4m3_truncates": ("r = nearbyintf(a / step) * step;", "r = floorf(a / step) * step;"),
    "fp8_scale_exponent_off": ("e = E - 1 - 7;", "e = E - 1 - 8;"),
    "fp8_dequant_one_scale": ("orc_e4m3_decode(q[j][k]) * scales[j][k / block]",
                              "orc_e4m3_decode(q[j][k]) * scales[j][0]"),
    "lp_accum_not_rounded": ("run = orc_float_to_lp(orc_lp_to_float(run, lp) +\n                                      orc_lp_to_float(slices[j][i], lp), lp);",
                             "run = orc_float_to_lp(orc_lp_to_float(run, lp), lp);"),
}


def _build_and_run(name, old, new, tmp):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new, 1)
    cpath = os.path.join(tmp, name + ".c")
    lib = os.path.join(tmp, name + ".so")
    with open(cpath, "w", encoding="utf-8") as f:
        f.write(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-I", os.path.join(ROOT, "oracle"), cpath, "-o", lib, "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, ZERO_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    return r.returncode


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            futs = {k: ex.submit(_build_and_run, k, o, n, tmp) for k, (o, n) in MUTANTS.items()}
            survived = [k for k, f in futs.items() if f.result() == 0]
    assert not survived, "mutants not caught by the oracle pins: %s" % survived


def test_unmutated_oracle_passes_the_pins():
    with tempfile.TemporaryDirectory() as tmp:
        assert _build_and_run("identity", "#include <math.h>", "#include <math.h>", tmp) == 0


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
