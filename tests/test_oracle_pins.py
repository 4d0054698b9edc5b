"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks one oracle function against what the pages print, a closed
form, a library routine (numpy / torch casts, math.fsum, np.concatenate) or
brute force on tiny inputs, chosen so that a dropped term, a wrong sign or
index, or a transposed operand fails at least one of them.
"""
import math
import os
import random

import numpy as np
import pytest
import torch

from zero_partitioned_mixed_flat_gb300.workloads import gpt2_tensors, zero3_7p5b_tensors

U32 = np.uint32
F16_MAX, F16_TINY = 0x7BFF, 0x0001


# ---------------------------------------------------------------- formats

def test_half_decode_exhaustive(orc):
    codes = np.arange(65536, dtype=np.uint16)
    ours = orc.lp_to_float(codes, 0)
    ref = codes.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(U32), ref[~nan].view(U32))


def test_bf16_decode_exhaustive(orc):
    codes = np.arange(65536, dtype=np.uint16)
    ours = orc.lp_to_float(codes, 1)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(U32), ref[~nan].view(U32))


def _encode_cases(lp):
    rng = np.random.default_rng(7 + lp)
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(U32)
    parts = [bits.view(np.float32)]
    parts.append((rng.standard_normal(200_000) * 10.0 ** rng.integers(-9, 6, 200_000))
                 .astype(np.float32))
    # exact ties between consecutive representable values (ties go to even)
    codes = np.arange(0, 0x7BFF if lp == 0 else 0x7F7F, dtype=np.uint16)
    lo = codes.view(np.float16).astype(np.float64) if lp == 0 else \
        torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    hi = (codes + 1).view(np.float16).astype(np.float64) if lp == 0 else \
        torch.from_numpy((codes + 1).view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # exact in f32
    parts += [mid, -mid]
    parts.append(np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 65504.0, 65519.996, 65520.0,
                           -65520.0, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001,
                           2.0 ** -14, 3.0e38, 3.3961e38, 3.4e38], np.float32))
    return np.concatenate(parts)


def test_half_encode_matches_numpy(orc):
    x = _encode_cases(0)
    ours = orc.float_to_lp(x, 0)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(orc.lp_to_float(ours[nan], 0)))


def test_bf16_encode_matches_torch(orc):
    x = _encode_cases(1)
    ours = orc.float_to_lp(x, 1)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(orc.lp_to_float(ours[nan], 1)))


# ---------------------------------------------------------- accounting

QIDX = {"ddp": 0, "os": 1, "os_g": 2, "os_g_p": 3}


def _golden_rows(path):
    rows = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split(None, 5)
            rows.append(parts)
    return rows


def test_memory_worked_examples(orc, golden_dir):
    rows = _golden_rows(os.path.join(golden_dir, "memory_worked_examples.txt"))
    assert len(rows) >= 12
    for psi, n, q, printed, dec, src in rows:
        formula, actual, _ = orc.memory(int(psi), int(n), 1)
        gb = formula[QIDX[q]] / 1e9
        tol = 0.5 * 10.0 ** (-int(dec)) + 1e-9
        assert abs(gb - float(printed)) <= tol, (psi, n, q, gb, printed, src)


def test_comm_volume(orc, golden_dir):
    rows = _golden_rows(os.path.join(golden_dir, "comm_volume.txt"))
    idx = {"ddp": 0, "1": 1, "2": 2, "3": 3}
    for psi in (1, 7, 1 << 20, 7_500_000_000):
        _, _, comm = orc.memory(psi, 8, 1)
        for row in rows:
            stage, mult = row[0], int(row[1])
            assert comm[idx[stage]] == mult * psi


def test_memory_exact_and_padded(orc):
    # N * align divides psi: padded layout equals the pages' formulas exactly
    f, a, _ = orc.memory(7_500_000_000, 64, 1)
    assert list(a) == [int(x) for x in f]
    assert list(a) == [120_000_000_000, 31_406_250_000, 16_640_625_000, 1_875_000_000]
    # N = 1: every stage is 16 psi
    f, a, _ = orc.memory(12345, 1, 1)
    assert set(f) == {16 * 12345.0} and set(a) == {16 * 12345}
    rng = random.Random(3)
    for _ in range(300):
        psi = rng.randrange(0, 10 ** 12)
        n = rng.choice([1, 2, 3, 7, 8, 64, 1000])
        al = rng.choice([1, 8, 128])
        f, a, _ = orc.memory(psi, n, al)
        # stages never grow, the padded actuals are never below the formula
        assert f[0] >= f[1] >= f[2] >= f[3]
        assert all(a[k] + 1e-3 * a[k] * 1e-9 >= f[k] - 1 for k in range(4))
        pad = (-psi) % (n * al)
        assert a[3] - f[3] <= 16 * pad / n + 1
        assert a[1] - f[1] <= 4 * pad + 12 * pad / n + 1


# --------------------------------------------------------------- layout

def _brute_layout(sizes, units, n, align, stage):
    if stage != 3 or units is None or not sizes:
        units = [0] * len(sizes)
    n_units = (max(units) + 1) if sizes else 1
    flat, offs, ustart, upad = [], [0] * len(sizes), [], []
    for u in range(n_units):
        start = len(flat)
        ustart.append(start)
        for t, s in enumerate(sizes):
            if units[t] != u:
                continue
            offs[t] = len(flat)
            flat += [(t, k) for k in range(s)]
        while (len(flat) - start) % (n * align):
            flat.append(None)
        upad.append(len(flat) - start)
    parts = []
    for r in range(n):
        p = []
        for u in range(n_units):
            shard = upad[u] if stage == 0 else upad[u] // n
            lo = ustart[u] + (0 if stage == 0 else r * shard)
            p += list(range(lo, lo + shard))
        parts.append(p)
    return flat, offs, parts


def _runs(flat, part):
    runs = []
    for pos, fi in enumerate(part):
        e = flat[fi]
        if e is None:
            continue
        t, k = e
        if runs and runs[-1][0] == t and runs[-1][1] + runs[-1][3] == k \
                and runs[-1][2] + runs[-1][3] == pos:
            runs[-1][3] += 1
        else:
            runs.append([t, k, pos, 1])
    return runs


def test_layout_brute_force(orc):
    rng = random.Random(11)
    for case in range(250):
        nt = rng.randrange(0, 7)
        sizes = [rng.choice([0, 1, 3, 8, 17, 100, 257]) for _ in range(nt)]
        n = rng.choice([1, 2, 3, 4, 8])
        align = rng.choice([8, 16, 128])
        stage = rng.choice([0, 1, 2, 3])
        units = None
        if stage == 3 and nt:
            units, u = [], 0
            for t in range(nt):
                if t and rng.random() < 0.5:
                    u += 1
                units.append(u)
        lay = orc.layout(sizes, n, align, stage, units)
        flat, offs, parts = _brute_layout(sizes, units, n, align, stage)
        assert lay["psi"] == sum(sizes)
        assert lay["psi_padded"] == len(flat)
        assert list(lay["tensor_offsets"]) == offs
        assert lay["part_len"] == len(parts[0])
        assert all(len(p) == len(parts[0]) for p in parts)
        if stage != 0:
            assert lay["part_len"] * n == lay["psi_padded"]
            # partitions tile the flat buffer exactly once
            assert sorted(i for p in parts for i in p) == list(range(len(flat)))
        for r in range(n):
            got = [orc.partition_to_flat(lay, r, k) for k in range(lay["part_len"])]
            assert got == parts[r]
            assert orc.partition_to_flat(lay, r, lay["part_len"]) == -1
            frags = orc.fragments(sizes, n, align, stage, r, units).tolist()
            assert frags == _runs(flat, parts[r]), (case, r)


def test_layout_rejects_bad_units(orc):
    with pytest.raises(ValueError):
        orc.layout([4, 4], 2, 8, 3, [0, 2])
    with pytest.raises(ValueError):
        orc.layout([4, 4], 2, 8, 3, [1, 1])
    with pytest.raises(ValueError):
        orc.layout([4, -1], 2, 8, 1)


def test_workload_sizes(orc):
    # GPT-2 small with biases and tied embeddings has 124,439,808 parameters
    assert sum(gpt2_tensors(768, 12)) == 124_439_808
    assert sum(gpt2_tensors(1600, 48)) == 1_557_611_200
    s, u = zero3_7p5b_tensors()
    assert sum(s) == 7_500_000_000 and u[-1] == 32
    lay = orc.layout(gpt2_tensors(768, 12), 8, 128, 1)
    assert lay["psi_padded"] == 124_440_576 and lay["part_len"] == 15_555_072
    lay = orc.layout(gpt2_tensors(1600, 48), 64, 128, 2)
    assert lay["psi_padded"] == 1_557_618_688 and lay["part_len"] == 24_337_792
    lay = orc.layout(s, 64, 128, 3, u)
    assert lay["n_units"] == 33 and lay["part_len"] == 117_189_632
    assert lay["unit_padded"][0] == 1_055_850_496 and lay["unit_padded"][1] == 201_383_936
    lay = orc.layout([13_000_000_000], 16, 128, 2)
    assert lay["psi_padded"] == 13_000_001_536 and lay["part_len"] == 812_500_096


# --------------------------------------------------------------- reduce

def _half(vals):
    return np.asarray(vals, np.float32).astype(np.float16).view(np.uint16)


def test_reduce_single_rank_is_exact_unscale(orc):
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(5000) * 1024).astype(np.float16)
    g, _, of = orc.reduce([x.view(np.uint16)], 0, 1024.0)
    assert of == 0
    assert np.array_equal(g, x.astype(np.float32) / np.float32(1024))


def test_reduce_is_mean_of_ranks(orc):
    ones = _half([1.0, -2.0, 0.5])
    g, _, _ = orc.reduce([ones] * 4, 0, 1.0)
    assert g.tolist() == [1.0, -2.0, 0.5]          # averaged, not summed
    g, _, _ = orc.reduce([ones] * 4, 0, 8.0)
    assert g.tolist() == [0.125, -0.25, 0.0625]    # and unscaled by S


def test_reduce_follows_rank_order(orc):
    a = np.array([F16_MAX], np.uint16)
    tiny = np.array([F16_TINY], np.uint16)
    neg = np.array([F16_MAX | 0x8000], np.uint16)
    g, _, _ = orc.reduce([a, tiny, neg], 0, 1.0)
    assert g[0] == 0.0                      # 65504 + 2^-24 rounds back to 65504
    g, _, _ = orc.reduce([a, neg, tiny], 0, 1.0)
    assert g[0] == np.float32(2.0 ** -24 / 3.0)


def test_reduce_error_bound_random(orc):
    rng = np.random.default_rng(5)
    for n in (1, 2, 3, 4, 8, 16):
        for lp in (0, 1):
            vals = rng.standard_normal((n, 4096)) * 10.0 ** rng.integers(-4, 3, (n, 4096))
            if lp == 0:
                codes = vals.astype(np.float16).view(np.uint16)
                exact_vals = codes.view(np.float16).astype(np.float64)
            else:
                t = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
                codes = t.view(torch.int16).numpy().view(np.uint16)
                exact_vals = t.double().numpy()
            s_exact = exact_vals.sum(axis=0)            # exact: few small-precision terms
            absum = np.abs(exact_vals).sum(axis=0)
            g, _, _ = orc.reduce(list(codes), lp, 1.0)
            inv = 1.0 / n
            bound = ((n - 1) * 2.0 ** -24 * absum) * inv + np.abs(g) * 2.0 ** -23
            assert np.all(np.abs(g.astype(np.float64) - s_exact * inv) <= bound + 1e-45)


def test_reduce_overflow_flag(orc):
    fine = _half([1.0, 2.0, 3.0])
    inf = fine.copy(); inf[1] = 0x7C00
    nan = fine.copy(); nan[2] = 0x7E00
    assert orc.reduce([fine, fine], 0, 2.0)[2] == 0
    assert orc.reduce([fine, inf], 0, 2.0)[2] == 1
    assert orc.reduce([nan, fine], 0, 2.0)[2] == 1
    big = np.array([0x7F7F, 0x3F80], np.uint16)   # bf16 max, 1.0
    assert orc.reduce([big, big], 1, 1.0)[2] == 1  # sum overflows float
    assert orc.reduce([big, big[::-1].copy()], 1, 1.0)[2] == 0


def test_sumsq_matches_fsum_and_runs_on(orc):
    rng = np.random.default_rng(9)
    codes = [(rng.standard_normal(100_003) * 3).astype(np.float16).view(np.uint16)
             for _ in range(3)]
    g, ss, _ = orc.reduce(codes, 0, 4.0)
    sq = (g * g).astype(np.float64)                 # float products, then exact sum
    ref = math.fsum(sq.tolist())
    assert abs(ss - ref) <= 1e-12 * ref
    # chunked calls continue the same running sum: identical to one pass
    acc, of = 0.0, 0
    for lo in range(0, 100_003, 17_000):
        _, acc, of = orc.reduce([c[lo:lo + 17_000] for c in codes], 0, 4.0, acc, of)
    assert acc == ss


def test_reduce_lp_accum_hand_cases(orc):
    # fp16: 2048 + 1 = 2049 is a tie between 2048 and 2050 -> even (2048), twice
    x = [_half([2048.0]), _half([1.0]), _half([1.0])]
    third = np.float32(1.0 / 3.0)                   # g = s * float(1/(S*N))
    g, _, of = orc.reduce_lp_accum(x, 0, 1.0)
    assert g[0] == np.float32(2048.0) * third and of == 0
    g, _, _ = orc.reduce(x, 0, 1.0)                 # float accumulation keeps both ones
    assert g[0] == np.float32(2050.0) * third
    # bf16: 256 + 1 ties to 256 the same way
    b = [np.array([0x4380], np.uint16), np.array([0x3F80], np.uint16), np.array([0x3F80], np.uint16)]
    g, _, _ = orc.reduce_lp_accum(b, 1, 1.0)
    assert g[0] == np.float32(256.0) * third
    # fp16: 65504 + 16 = 65520 rounds up to 65536, which overflows to inf
    o = [_half([65504.0]), _half([16.0])]
    assert orc.reduce_lp_accum(o, 0, 1.0)[2] == 1
    assert orc.reduce(o, 0, 1.0)[2] == 0            # finite in float


def test_reduce_lp_accum_matches_library_sequential_sums(orc):
    rng = np.random.default_rng(12)
    for n in (2, 3, 8, 17):
        vals = rng.standard_normal((n, 20_000)) * 10.0 ** rng.integers(-6, 4, (n, 20_000))
        h = vals.astype(np.float16)
        with np.errstate(over="ignore"):
            acc = h[0].copy()
            for j in range(1, n):
                acc = (acc + h[j]).astype(np.float16)   # numpy half add: rounded to half
        g, _, _ = orc.reduce_lp_accum(list(h.view(np.uint16)), 0, 1.0)
        ref = acc.astype(np.float32) * np.float32(1.0 / n)
        fin = np.isfinite(ref)
        assert np.array_equal(g[fin].view(U32), ref[fin].view(U32))
        t = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
        acc = t[0].clone()
        for j in range(1, n):
            acc = acc + t[j]                            # torch bf16 add: rounded to bf16
        g, _, _ = orc.reduce_lp_accum(list(t.view(torch.int16).numpy().view(np.uint16)), 1, 1.0)
        ref = acc.float().numpy() * np.float32(1.0 / n)
        assert np.array_equal(g.view(U32), ref.view(U32))


# ----------------------------------------------------- decision (clip/scale)

def test_clip_coefficient_closed_form(orc):
    half = _half([0.5] * 1024)
    g, ss, _ = orc.reduce([half], 0, 1.0)
    assert ss == 256.0                             # 1024 * 0.25
    d = orc.decide(ss, 0, 1.0, 1.0, 0)
    assert d["norm"] == 16.0
    assert d["coef"] == np.float32(1.0 / (16.0 + 1e-6))
    d = orc.decide(ss, 0, 100.0, 1.0, 0)
    assert d["coef"] == 1.0                        # below the clip: untouched
    d = orc.decide(ss, 0, 0.0, 1.0, 0)
    assert d["coef"] == 1.0                        # clip <= 0 disables
    d = orc.decide(ss, 0, 1.0, 1.0, 0, remote_sumsq=144.0)
    assert d["norm"] == 20.0                       # sqrt(256 + 144): global norm


def test_loss_scale_sequence_with_injected_overflow(orc):
    # dynamic scale 2^16, overflow on step 2 of 3: S 65536 -> 32768, t = 1, 1, 2
    s, t, good, seen = 65536.0, 0, 0, []
    for step, of in enumerate([0, 1, 0], start=1):
        d = orc.decide(1.0, of, 1.0, s, t, good, 1000)
        assert d["skip"] == of
        s, t, good = d["new_scale"], d["step"], d["good_steps"]
        seen.append((s, t))
    assert seen == [(65536.0, 1), (32768.0, 1), (32768.0, 2)]


def test_loss_scale_growth_floor_and_static(orc):
    d = orc.decide(1.0, 0, 1.0, 8.0, 5, 1, 2)      # second good step of interval 2
    assert (d["new_scale"], d["good_steps"], d["step"]) == (16.0, 0, 6)
    d = orc.decide(1.0, 1, 1.0, 1.0, 5, 1, 2)      # overflow at the floor
    assert (d["new_scale"], d["good_steps"], d["step"], d["skip"]) == (1.0, 0, 5, 1)
    d = orc.decide(1.0, 1, 1.0, 1024.0, 5, 0, 0)   # static scale keeps S
    assert (d["new_scale"], d["step"], d["skip"]) == (1024.0, 5, 1)
    d = orc.decide(1.0, 0, 1.0, 1.0, 0, 0, 0, remote_overflow=1)
    assert d["skip"] == 1 and d["step"] == 0


def test_bias_corrections(orc):
    d = orc.decide(1.0, 0, 1.0, 1.0, 0, beta1=0.9, beta2=0.999)
    assert d["step"] == 1
    assert d["bc1"] == np.float32(1.0) - np.float32(0.9)     # exact (Sterbenz)
    assert d["bc2"] == np.float32(1.0) - np.float32(0.999)
    d = orc.decide(1.0, 0, 1.0, 1.0, 1, beta1=0.9, beta2=0.999)
    b1 = float(np.float32(0.9))
    # 1 - b^2 = (1 - b)(1 + b)
    assert abs(d["bc1"] - (1 - b1) * (1 + b1)) <= 2.0 ** -24 * 0.19


# ------------------------------------------------------------------ adam

HP = dict(beta1=0.9, beta2=0.999)


def _run_adam(orc, g_seq, w0, lr, eps, wd, adamw, coef=1.0, lp=0, b1=0.9, b2=0.999):
    n = len(w0)
    master = np.array(w0, np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    hist = []
    for t, g in enumerate(g_seq, start=1):
        d = orc.decide(0.0, 0, 0.0, 1.0, t - 1, beta1=b1, beta2=b2)
        prev = master.copy()
        p = orc.adam(np.array(g, np.float32), master, m, v, lp, coef, 0, lr, b1, b2, eps,
                     wd, adamw, d["bc1"], d["bc2"])
        hist.append((prev, master.copy(), m.copy(), v.copy(), p))
    return hist


@pytest.mark.parametrize("eps", [1e-8, 0.5])
def test_adam_constant_gradient_closed_form(orc, eps):
    # with a constant gradient m_hat = g and v_hat = g^2 at every step, so each
    # step moves the weight by lr * g / (|g| + eps) (eps outside the sqrt)
    g = [1.5, -0.75, 3.0, -2.0 ** -10]
    lr = 1e-3
    hist = _run_adam(orc, [g] * 6, [0.25, -0.5, 0.0, 1.0], lr, eps, 0.0, 1)
    ga = np.array(g, np.float64)
    expected = lr * ga / (np.abs(ga) + eps)
    for t, (prev, cur, m, v, _) in enumerate(hist, start=1):
        step = prev.astype(np.float64) - cur.astype(np.float64)
        ulp = np.spacing(np.abs(cur).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(step - expected) <= 16 * 2.0 ** -24 * np.abs(expected) + ulp)
        b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))  # the betas as passed
        assert np.allclose(m, (1 - b1 ** t) * ga, rtol=8 * t * 2.0 ** -24, atol=0)
        assert np.allclose(v, (1 - b2 ** t) * ga * ga, rtol=40 * t * 2.0 ** -24, atol=0)


def test_adam_two_step_hand_values(orc):
    # g1 = 1, g2 = -1: m2 = b1(1-b1) - (1-b1) = -(1-b1)^2 and 1 - b1^2 = (1-b1)(1+b1),
    # so m_hat = -(1-b1)/(1+b1) (= -0.1/1.9); v2 = (1-b2)(b2+1) = 1 - b2^2, so v_hat = 1.
    lr, eps = 1e-2, 1e-8
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))  # the betas as passed
    hist = _run_adam(orc, [[1.0], [-1.0]], [0.0], lr, eps, 0.0, 1)
    prev, cur, m, v, _ = hist[1]
    assert abs(m[0] + (1 - b1) ** 2) <= 4 * 2.0 ** -24 * (1 - b1) ** 2 * 10
    assert abs(v[0] - (1 - b2 * b2)) <= 8 * 2.0 ** -24 * (1 - b2 * b2) * 10
    upd = float(prev[0]) - float(cur[0])
    exp = lr * (-(1 - b1) / (1 + b1)) / (1.0 + eps)
    assert abs(upd - exp) <= 1e-6 * abs(exp)
    assert abs(exp - lr * (-0.1 / 1.9)) <= 1e-6 * lr


def test_adamw_pure_decay(orc):
    # zero gradient: the moments stay 0 and AdamW only decays the weight
    lr, wd = 1e-2, 0.1
    w0 = [1.0, -3.0, 0.0, 2.0 ** -20]
    hist = _run_adam(orc, [[0.0] * 4] * 5, w0, lr, 1e-8, wd, 1)
    for t, (_, cur, m, v, _) in enumerate(hist, start=1):
        exp = np.array(w0) * (1 - lr * wd) ** t
        assert np.all(np.abs(cur - exp) <= 2 * t * 2.0 ** -24 * np.abs(exp))
        assert not m.any() and not v.any()


def test_adam_l2_differs_from_adamw(orc):
    # L2 Adam folds wd * w into the gradient: with g = 0 the first step moves
    # the weight by about lr * sign(w); AdamW instead scales it by (1 - lr wd)
    lr, wd = 1e-3, 0.1
    l2 = _run_adam(orc, [[0.0, 0.0]], [2.0, -4.0], lr, 1e-8, wd, 0)[0]
    w = _run_adam(orc, [[0.0, 0.0]], [2.0, -4.0], lr, 1e-8, wd, 1)[0]
    step = l2[0].astype(np.float64) - l2[1].astype(np.float64)
    ulp = float(np.spacing(np.float32(4.0)))          # rounding of the stored weight
    assert np.allclose(step, [lr, -lr], rtol=1e-6, atol=ulp)
    assert np.allclose(w[1], [2.0 * (1 - lr * wd), -4.0 * (1 - lr * wd)], rtol=0, atol=ulp)


def test_adam_coef_scales_gradient_and_skip_writes_nothing(orc):
    lr, eps = 1e-3, 0.5
    a = _run_adam(orc, [[2.0]], [0.0], lr, eps, 0.0, 1, coef=0.5)[0]
    # g' = 1: update = lr * 1 / (1 + 0.5)
    assert abs((a[0] - a[1])[0] - lr / 1.5) <= 4 * 2.0 ** -24 * lr
    master = np.ones(3, np.float32); m = np.ones(3, np.float32); v = np.ones(3, np.float32)
    p = orc.adam(np.ones(3, np.float32), master, m, v, 0, 1.0, 1, lr, 0.9, 0.999, 1e-8,
                 0.01, 1, 0.1, 0.001)
    assert master.tolist() == [1.0] * 3 and m.tolist() == [1.0] * 3 and v.tolist() == [1.0] * 3
    assert p is not None  # the buffer exists but is untouched by a skipped step


def test_adam_param_is_rounded_master(orc):
    rng = np.random.default_rng(2)
    w0 = (rng.standard_normal(10_000) * 0.02).astype(np.float32)
    g = rng.standard_normal(10_000).astype(np.float32) * 1e-3
    for lp in (0, 1):
        hist = _run_adam(orc, [g], w0, 1e-4, 1e-8, 0.01, 1, lp=lp)
        _, cur, _, _, p = hist[0]
        if lp == 0:
            ref = cur.astype(np.float16).view(np.uint16)
        else:
            ref = torch.from_numpy(cur).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(p, ref)


# ---------------------------------------------------------------- gather

def test_gather_is_concatenation(orc):
    rng = np.random.default_rng(4)
    shards = [rng.integers(0, 65536, 1000, dtype=np.uint16) for _ in range(7)]
    assert np.array_equal(orc.gather(shards), np.concatenate(shards))


# ------------------------------------------ invariant: sharded step == DDP

def _ddp_vs_sharded(orc, sizes, units, n, stage, lp, steps, clip, seed):
    align = 8
    lay = orc.layout(sizes, n, align, stage, units)
    psi_p = lay["psi_padded"]
    P = lay["part_len"] if stage != 0 else psi_p // n
    rng = np.random.default_rng(seed)
    pad_mask = np.ones(psi_p, bool)
    for t, off in enumerate(lay["tensor_offsets"]):
        pad_mask[off:off + sizes[t]] = False
    w0 = (rng.standard_normal(psi_p) * 0.02).astype(np.float32)
    w0[pad_mask] = 0
    # DDP: every rank holds everything; all-reduce = the same reduce on all of psi_p
    dm, dmm, dv = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    sm, smm, sv = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    s_param = np.zeros(psi_p, np.uint16)
    t_ddp = t_sh = 0
    idx = [np.array([orc.partition_to_flat(lay, r, k) for k in range(P)], np.int64)
           for r in range(n)] if stage != 0 else None
    for step in range(steps):
        grads = []
        for j in range(n):
            x = (rng.standard_normal(psi_p) * 1e-2 * 64).astype(np.float32)
            x[pad_mask] = 0
            codes = x.astype(np.float16).view(np.uint16) if lp == 0 else \
                torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            grads.append(codes)
        S = 64.0
        g, ss, of = orc.reduce(grads, lp, S)
        d = orc.decide(ss, of, clip, S, t_ddp)
        p_ddp = orc.adam(g, dm, dmm, dv, lp, d["coef"], d["skip"], 1e-3, 0.9, 0.999, 1e-8,
                         0.01, 1, d["bc1"], d["bc2"])
        t_ddp = d["step"]
        # sharded: each rank reduces its partition from the N ranks' slices
        parts, tot, oft = [], 0.0, 0
        for r in range(n):
            gi, ssr, ofr = orc.reduce([gr[idx[r]] for gr in grads], lp, S)
            parts.append(gi)
            tot += ssr
            oft |= ofr
        ds = orc.decide(tot, oft, clip, S, t_sh)
        assert ds["coef"] == d["coef"] and ds["skip"] == d["skip"]
        assert abs(ds["norm"] - d["norm"]) <= 1e-12 * d["norm"]
        for r in range(n):
            mm, m1, v1 = sm[idx[r]], smm[idx[r]], sv[idx[r]]
            p = orc.adam(parts[r], mm, m1, v1, lp, ds["coef"], ds["skip"], 1e-3, 0.9, 0.999,
                         1e-8, 0.01, 1, ds["bc1"], ds["bc2"])
            sm[idx[r]], smm[idx[r]], sv[idx[r]] = mm, m1, v1
            s_param[idx[r]] = p          # all-gather destination: the full layout
        t_sh = ds["step"]
        assert np.array_equal(sm.view(U32), dm.view(U32))
        assert np.array_equal(smm.view(U32), dmm.view(U32))
        assert np.array_equal(sv.view(U32), dv.view(U32))
        assert np.array_equal(s_param, p_ddp)
        assert not sm[pad_mask].any() and not smm[pad_mask].any()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("stage", [1, 2])
def test_sharded_step_equals_ddp(orc, n, stage):
    _ddp_vs_sharded(orc, [1000, 37, 5, 2048], None, n, stage, stage - 1, 3, 1.0, n)


@pytest.mark.parametrize("n", [2, 3, 8])
def test_sharded_stage3_units_equals_ddp(orc, n):
    _ddp_vs_sharded(orc, [300, 17, 64, 64, 1, 999], [0, 0, 1, 2, 2, 3], n, 3, 0, 2, 0.05, 10 + n)


# ------------------------------------------------ quantized gather (ZeRO++)

def test_quantize_hand_block(orc):
    # one 8-element block with amax 127: scale 1, codes are x rounded to even
    x = _half([127.0, -127.0, 0.5, 1.5, 2.5, -0.5, -3.5, 0.0])
    q, sc = orc.quantize_blocks(x, 0, block=8)
    assert sc.tolist() == [1.0]
    assert q.tolist() == [127, -127, 0, 2, 2, 0, -4, 0]
    y = orc.dequant_gather([q], [sc], 0, block=8)
    assert orc.lp_to_float(y, 0).tolist() == [127.0, -127.0, 0.0, 2.0, 2.0, 0.0, -4.0, 0.0]
    # an all-zero block: scale 0, codes 0, values 0
    q, sc = orc.quantize_blocks(_half([0.0] * 8), 0, block=8)
    assert sc.tolist() == [0.0] and not q.any()


def test_quantize_matches_numpy_rint_and_bounds(orc):
    rng = np.random.default_rng(21)
    for lp in (0, 1):
        x = (rng.standard_normal(128 * 400) * 10.0 ** rng.integers(-3, 2, 128 * 400)).astype(np.float32)
        codes = orc.float_to_lp(x, lp)
        xf = orc.lp_to_float(codes, lp).reshape(-1, 128)
        q, sc = orc.quantize_blocks(codes, lp, 128)
        amax = np.abs(xf).max(axis=1)
        assert np.array_equal(sc, (amax / np.float32(127)).astype(np.float32))
        ref = np.rint(xf / sc[:, None]).astype(np.int8)          # numpy: RN-even
        assert np.array_equal(q.reshape(-1, 128), ref)
        # the block maximum maps to +-127 and every code is within the range
        assert np.all(np.abs(q.reshape(-1, 128)).max(axis=1) == 127)
        # dequantized error within half a step (plus the lp rounding)
        y = orc.lp_to_float(orc.dequant_gather([q], [sc], lp, 128), lp).reshape(-1, 128)
        lp_ulp = 2.0 ** (-10 if lp == 0 else -7)
        assert np.all(np.abs(y - xf) <= sc[:, None] * 0.5 * (1 + 1e-6) + np.abs(y) * lp_ulp)


def test_dequant_gather_layout(orc):
    rng = np.random.default_rng(22)
    shards = [orc.float_to_lp(rng.standard_normal(256).astype(np.float32), 0) for _ in range(3)]
    qs = [orc.quantize_blocks(s, 0, 128) for s in shards]
    out = orc.dequant_gather([q for q, _ in qs], [c for _, c in qs], 0, 128)
    for j in range(3):
        one = orc.dequant_gather([qs[j][0]], [qs[j][1]], 0, 128)
        assert np.array_equal(out[j * 256:(j + 1) * 256], one)


# ------------------------------------------ fp8 (E4M3) variant of the gather

def test_e4m3_decode_definition_and_library(orc):
    # the format's definition at hand-picked codes ...
    d = orc.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0xb8, 0x7e, 0x70, 0x77, 0x80],
                                 np.uint8))
    assert d.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, -1.0, 448.0, 128.0, 240.0,
                          -0.0]
    assert math.copysign(1.0, d[-1]) == -1.0
    assert np.isnan(orc.e4m3_decode(np.array([0x7f, 0xff], np.uint8))).all()
    # ... and every one of the 256 codes against torch's float8_e4m3fn
    c = np.arange(256, dtype=np.uint8)
    d = orc.e4m3_decode(c)
    t = torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(d), np.isnan(t))
    assert np.array_equal(d[~np.isnan(d)], t[~np.isnan(t)])


def test_e4m3_encode_rounds_to_nearest_even_and_saturates(orc):
    c = np.arange(0x7f, dtype=np.uint8)
    vals = orc.e4m3_decode(c)
    assert np.array_equal(orc.e4m3_encode(vals), c)                    # exact values
    assert np.array_equal(orc.e4m3_encode(-vals), c | 0x80)
    mids = ((vals[1:].astype(np.float64) + vals[:-1]) / 2).astype(np.float32)   # exact ties
    even = np.where((c[:-1] & 1) == 0, c[:-1], c[1:])
    assert np.array_equal(orc.e4m3_encode(mids), even)
    rng = np.random.default_rng(31)
    v = np.concatenate([rng.uniform(-463, 463, 50000),
                        rng.uniform(-1, 1, 50000) * 2.0 ** rng.integers(-14, 9, 50000)]).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    t = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(v), t)
    # saturation (finite and infinite), NaN, signed zero
    big = np.array([464.0, 1e30, np.inf, -464.0, -np.inf, np.nan, -0.0], np.float32)
    assert orc.e4m3_encode(big).tolist() == [0x7e, 0x7e, 0x7e, 0xfe, 0xfe, 0x7f, 0x80]


def test_quantize_fp8_scale_and_error(orc):
    rng = np.random.default_rng(32)
    for lp in (0, 1):
        x = (rng.standard_normal(128 * 300) * 10.0 ** rng.integers(-3, 3, 128 * 300)).astype(np.float32)
        codes = orc.float_to_lp(x, lp)
        xf = orc.lp_to_float(codes, lp).reshape(-1, 128).astype(np.float64)
        q, sc = orc.quantize_blocks_fp8(codes, lp, 128)
        amax = np.abs(xf).max(axis=1)
        # the scale is the power of two that puts amax in [128, 256)
        e = np.log2(sc.astype(np.float64))
        assert np.array_equal(e, np.round(e))
        assert np.all((amax / sc >= 128) & (amax / sc < 256))
        # codes are the nearest-even encoding of x / scale (computed in float64:
        # a power-of-two scaling is exact)
        ref = torch.from_numpy((xf / sc[:, None]).astype(np.float32).reshape(-1)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q, ref)
        # dequantized error: half an E4M3 step (2^-4 relative, 2^-10 * scale for
        # subnormal codes), plus the lp rounding
        y = orc.lp_to_float(orc.dequant_gather_fp8([q], [sc], lp, 128), lp).reshape(-1, 128)
        lp_ulp = 2.0 ** (-10 if lp == 0 else -7)
        bound = np.maximum(np.abs(xf) * 2.0 ** -4, sc[:, None] * 2.0 ** -10) + np.abs(y) * lp_ulp
        assert np.all(np.abs(y - xf) <= bound * (1 + 1e-6))


def test_quantize_fp8_exact_round_trip_and_zero_block(orc):
    # values that are E4M3 codes times 2^e come back bit for bit
    rng = np.random.default_rng(33)
    c = rng.integers(0, 0x70, 128).astype(np.uint8) | (rng.integers(0, 2, 128) << 7).astype(np.uint8)
    c[5] = 0x75                                            # 208: the block maximum, in [128, 256)
    for e in (-15, -3, 0, 4, 7):     # every value stays an fp16 number
        x = orc.e4m3_decode(c) * np.float32(2.0 ** e)
        codes = orc.float_to_lp(x, 0)
        assert np.array_equal(orc.lp_to_float(codes, 0), x)  # representable in fp16
        q, sc = orc.quantize_blocks_fp8(codes, 0, 128)
        assert sc.tolist() == [2.0 ** e]
        assert np.array_equal(q, c)
        assert np.array_equal(orc.dequant_gather_fp8([q], [sc], 0, 128), codes)
    q, sc = orc.quantize_blocks_fp8(np.zeros(128, np.uint16), 0, 128)
    assert sc.tolist() == [0.0] and not q.any()


def test_dequant_gather_fp8_layout(orc):
    rng = np.random.default_rng(34)
    shards = [orc.float_to_lp(rng.standard_normal(384).astype(np.float32), 1) for _ in range(3)]
    qs = [orc.quantize_blocks_fp8(s, 1, 128) for s in shards]
    out = orc.dequant_gather_fp8([q for q, _ in qs], [c for _, c in qs], 1, 128)
    for j in range(3):
        one = orc.dequant_gather_fp8([qs[j][0]], [qs[j][1]], 1, 128)
        assert np.array_equal(out[j * 384:(j + 1) * 384], one)
