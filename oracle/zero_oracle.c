/*
 * zero_oracle.c -- plain, slow CPU oracle of the ZeRO partitioned
 * mixed-precision Adam step (see zero_oracle.h for the sources).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product library.
 *
 * Every floating-point operation below is a separate IEEE operation rounded
 * to nearest-even.  The file must be compiled without FMA contraction and
 * without fast-math (-ffp-contract=off, see oracle/build.py), so that each
 * `a * b + c` is two roundings, as written.
 *
 * Parity status per function (what pins it is in tests/test_oracle_pins.py):
 *   formats, layout, fragments, memory, reduce, decide, adam, gather: pinned.
 *   No page prints an Adam trajectory; Adam is pinned by closed forms
 *   (constant-gradient steps, pure decay, first-step moments) rather than by
 *   printed values.
 */
#include "zero_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------
 * Number formats.
 *
 * Decoding is the IEEE definition: value = (-1)^s * 2^(e-bias) * 1.f for
 * normal codes, (-1)^s * 2^(1-bias) * 0.f for subnormal codes.
 * Encoding rounds the exact value to the nearest representable one, ties to
 * the even significand, with overflow to infinity (IEEE 754 §4.3.1, §7.4).
 * ---------------------------------------------------------------------- */

/* Round a >= 0 (finite) to a binary format with p significand bits and
 * minimum normal exponent emin; the result is exact in double. */
static double round_to_format(double a, int p, int emin)
{
    int e;
    double q, n;
    if (a == 0.0)
        return 0.0;
    e = ilogb(a);
    if (e < emin)
        e = emin; /* subnormals share the spacing of the first binade */
    q = ldexp(1.0, e - (p - 1));
    n = nearbyint(a / q); /* a / q is exact; default mode is to-nearest-even */
    return n * q;
}

static float half_decode_definition(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0x1f)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -24);           /* 2^(1-15) * f / 2^10 */
    else
        v = ldexp((double)(1024 + f), e - 25); /* 2^(e-15) * (1024+f) / 2^10 */
    return (float)(sign ? -v : v);
}

/* decoding table: built once, at load, from the definition above */
static float g_half_table[65536];

__attribute__((constructor)) static void build_half_table(void)
{
    for (int c = 0; c < 65536; ++c)
        g_half_table[c] = half_decode_definition((uint16_t)c);
}

float orc_half_to_float(uint16_t h) { return g_half_table[h]; }

uint16_t orc_float_to_half(float f)
{
    double x = (double)f, a, v;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7e00u);
    a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7c00u);
    v = round_to_format(a, 11, -14);
    if (v > 65504.0) /* largest finite binary16 */
        return (uint16_t)(sign | 0x7c00u);
    if (v < ldexp(1.0, -14)) /* subnormal (or zero): code = v / 2^-24 */
        return (uint16_t)(sign | (uint16_t)(v * ldexp(1.0, 24)));
    {
        int e = ilogb(v);
        int frac = (int)(ldexp(v, 10 - e)) - 1024;
        return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)frac);
    }
}

float orc_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t orc_float_to_bf16(float f)
{
    double x = (double)f, a, v;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    float r;
    uint32_t u;
    if (isnan(x))
        return (uint16_t)(sign | 0x7fc0u);
    a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | 0x7f80u);
    v = round_to_format(a, 8, -126);
    if (v > ldexp(2.0 - ldexp(1.0, -7), 127)) /* largest finite bfloat16 */
        return (uint16_t)(sign | 0x7f80u);
    r = (float)v; /* exact: bfloat16 values are a subset of binary32 */
    memcpy(&u, &r, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

float orc_lp_to_float(uint16_t x, int32_t lp)
{
    return lp ? orc_bf16_to_float(x) : orc_half_to_float(x);
}

uint16_t orc_float_to_lp(float f, int32_t lp)
{
    return lp ? orc_float_to_bf16(f) : orc_float_to_half(f);
}

void orc_lp_array_to_float(int64_t n, const uint16_t *x, int32_t lp, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_lp_to_float(x[i], lp);
}

void orc_float_array_to_lp(int64_t n, const float *x, int32_t lp, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_float_to_lp(x[i], lp);
}

/* ------------------------------------------------------------------------
 * Layout.  The flat buffer is the tensors concatenated in the given order
 * with no per-tensor padding ([P3] §2.1 item 3: gradients fused into one flat
 * buffer; [P4] §10.6.6 contiguous_gradients).  The tail of the buffer (of
 * every unit, in stage 3) is zero padding up to a multiple of N * align, so
 * that N equal partitions exist ([P4] §10.6.2: each GPU owns 1/N).  Stage 3
 * shards every unit on its own ([P4] §10.6.7: each FSDP unit is flattened and
 * sharded as a whole).
 * ---------------------------------------------------------------------- */

static int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

static int32_t count_units(int32_t n_tensors, const int32_t *unit_of_tensor,
                           int32_t stage)
{
    if (stage != 3 || unit_of_tensor == NULL || n_tensors == 0)
        return 1;
    if (unit_of_tensor[0] != 0)
        return -1;
    for (int32_t t = 1; t < n_tensors; ++t) {
        int32_t d = unit_of_tensor[t] - unit_of_tensor[t - 1];
        if (d != 0 && d != 1)
            return -1;
    }
    return unit_of_tensor[n_tensors - 1] + 1;
}

int32_t orc_layout(int32_t n_tensors, const int64_t *sizes,
                   const int32_t *unit_of_tensor, int32_t n_ranks,
                   int32_t align, int32_t stage,
                   int64_t *psi, int64_t *psi_padded, int64_t *part_len,
                   int32_t *n_units, int64_t *tensor_offsets,
                   int64_t *unit_offsets, int64_t *unit_padded)
{
    int64_t quantum, flat = 0, total = 0;
    int32_t nu, t = 0;
    if (n_tensors < 0 || n_ranks < 1 || align < 1 || stage < 0 || stage > 3)
        return -1;
    if (n_tensors > 0 && sizes == NULL)
        return -1;
    for (int32_t i = 0; i < n_tensors; ++i)
        if (sizes[i] < 0)
            return -1;
    nu = count_units(n_tensors, unit_of_tensor, stage);
    if (nu < 1)
        return -1;
    quantum = (int64_t)n_ranks * align;
    for (int32_t u = 0; u < nu; ++u) {
        int64_t fill = 0;
        if (unit_offsets)
            unit_offsets[u] = flat;
        /* every tensor of unit u, in list order */
        while (t < n_tensors &&
               (nu == 1 || unit_of_tensor[t] == u)) {
            if (tensor_offsets)
                tensor_offsets[t] = flat + fill;
            fill += sizes[t];
            ++t;
        }
        total += fill;
        if (unit_padded)
            unit_padded[u] = round_up(fill, quantum);
        flat += round_up(fill, quantum);
    }
    if (unit_offsets)
        unit_offsets[nu] = flat;
    if (psi)
        *psi = total;
    if (psi_padded)
        *psi_padded = flat;
    if (part_len)
        *part_len = stage == 0 ? flat : flat / n_ranks;
    if (n_units)
        *n_units = nu;
    return 0;
}

int64_t orc_partition_to_flat(int32_t n_units, const int64_t *unit_offsets,
                              const int64_t *unit_padded, int32_t n_ranks,
                              int32_t stage, int32_t rank, int64_t k)
{
    if (k < 0 || rank < 0 || rank >= n_ranks)
        return -1;
    for (int32_t u = 0; u < n_units; ++u) {
        int64_t shard = stage == 0 ? unit_padded[u] : unit_padded[u] / n_ranks;
        int64_t start = unit_offsets[u] + (stage == 0 ? 0 : rank * shard);
        if (k < shard)
            return start + k;
        k -= shard;
    }
    return -1;
}

int64_t orc_fragments(int32_t n_tensors, const int64_t *sizes,
                      const int32_t *unit_of_tensor, int32_t n_ranks,
                      int32_t align, int32_t stage, int32_t rank,
                      int64_t max_frag, int64_t *frag)
{
    int64_t psi, psi_p, part;
    int32_t nu;
    int64_t *toff, *uoff, *upad, count = 0, part_pos = 0;
    if (rank < 0 || rank >= n_ranks)
        return -1;
    toff = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_tensors + 1));
    uoff = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_tensors + 2));
    upad = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_tensors + 1));
    if (!toff || !uoff || !upad ||
        orc_layout(n_tensors, sizes, unit_of_tensor, n_ranks, align, stage,
                   &psi, &psi_p, &part, &nu, toff, uoff, upad) != 0) {
        free(toff); free(uoff); free(upad);
        return -1;
    }
    for (int32_t u = 0; u < nu; ++u) {
        int64_t shard = stage == 0 ? upad[u] : upad[u] / n_ranks;
        int64_t lo = uoff[u] + (stage == 0 ? 0 : rank * shard);
        int64_t hi = lo + shard;
        for (int32_t t = 0; t < n_tensors; ++t) {
            int32_t tu = (nu == 1) ? 0 : unit_of_tensor[t];
            int64_t a, b;
            if (tu != u)
                continue;
            a = toff[t] > lo ? toff[t] : lo;
            b = toff[t] + sizes[t] < hi ? toff[t] + sizes[t] : hi;
            if (a >= b)
                continue;
            if (count < max_frag && frag) {
                frag[4 * count + 0] = t;
                frag[4 * count + 1] = a - toff[t];
                frag[4 * count + 2] = part_pos + (a - lo);
                frag[4 * count + 3] = b - a;
            }
            ++count;
        }
        part_pos += shard;
    }
    free(toff); free(uoff); free(upad);
    return count;
}

/* ------------------------------------------------------------------------
 * Accounting.  [P4] Table 10-2 (and §10.6.2–§10.6.4): per-GPU model-state
 * bytes DDP 16Ψ, stage 1 4Ψ + 12Ψ/N, stage 2 2Ψ + 14Ψ/N, stage 3 16Ψ/N;
 * communication DDP 2Ψ, stages 1/2 2Ψ, stage 3 3Ψ.  [P3] §2.2: 2Ψ fp16
 * params + 2Ψ fp16 grads + KΨ optimizer state with K = 12.
 * ---------------------------------------------------------------------- */

/* base + num / n as one rounding (num, base >= 0). */
static double int_plus_ratio(int64_t base, int64_t num, int64_t n)
{
    return (double)(base + num / n) + (double)(num % n) / (double)n;
}

int32_t orc_memory(int64_t psi, int32_t n_ranks, int32_t align,
                   double formula[4], int64_t actual[4], int64_t comm[4])
{
    int64_t psi_p, part;
    if (psi < 0 || n_ranks < 1 || align < 1)
        return -1;
    formula[0] = (double)(16 * psi);
    formula[1] = int_plus_ratio(4 * psi, 12 * psi, n_ranks);
    formula[2] = int_plus_ratio(2 * psi, 14 * psi, n_ranks);
    formula[3] = int_plus_ratio(0, 16 * psi, n_ranks);
    psi_p = round_up(psi, (int64_t)n_ranks * align);
    part = psi_p / n_ranks;
    actual[0] = 16 * psi;
    actual[1] = 4 * psi_p + 12 * part;
    actual[2] = 2 * psi_p + 14 * part;
    actual[3] = 16 * part;
    comm[0] = 2 * psi;
    comm[1] = 2 * psi;
    comm[2] = 2 * psi;
    comm[3] = 3 * psi;
    return 0;
}

/* ------------------------------------------------------------------------
 * Reduce.  [P4] §10.6.1: reduce-scatter sums every rank's data and leaves
 * each rank one 1/N slice of the result; [P1] ZeRO-2: each rank receives the
 * average of all ranks' gradients for its 1/N.  Mean and loss-scale removal
 * ([P2] §4.3) are one multiplication by 1/(S*N).  The sum runs in float, in
 * rank order 0..N-1 (the accumulation precision is fixed as float because
 * the pages keep every optimizer-side quantity in fp32, [P4] §10.6 table).
 * ---------------------------------------------------------------------- */
void orc_reduce(int32_t n, const uint16_t *const *slices, int32_t lp,
                int64_t len, float loss_scale, float *g, double *sumsq,
                int32_t *overflow)
{
    const float inv = (float)(1.0 / ((double)loss_scale * (double)n));
    double acc = *sumsq; /* running sum: chunked calls equal one pass */
    int32_t of = *overflow;
    for (int64_t i = 0; i < len; ++i) {
        float s = orc_lp_to_float(slices[0][i], lp);
        float gi, sq;
        for (int32_t j = 1; j < n; ++j)
            s = s + orc_lp_to_float(slices[j][i], lp);
        if (!isfinite(s))
            of = 1;
        gi = s * inv;
        g[i] = gi;
        sq = gi * gi;
        acc = acc + (double)sq;
    }
    *sumsq = acc;
    *overflow = of;
}

/* The low-precision accumulation: the exact sum of the running lp value and
 * the next rank's lp value, rounded to the lp type.  The float addition is
 * that exact sum rounded to 24 bits; a second rounding to 11 (fp16) or 8
 * (bf16) bits then equals one direct rounding, because 24 >= 2p + 2
 * (Figueroa, "When is double rounding innocuous?", 1995). */
void orc_reduce_lp_accum(int32_t n, const uint16_t *const *slices, int32_t lp,
                         int64_t len, float loss_scale, float *g, double *sumsq,
                         int32_t *overflow)
{
    const float inv = (float)(1.0 / ((double)loss_scale * (double)n));
    double acc = *sumsq;
    int32_t of = *overflow;
    for (int64_t i = 0; i < len; ++i) {
        uint16_t run = slices[0][i];
        float s, gi, sq;
        for (int32_t j = 1; j < n; ++j)
            run = orc_float_to_lp(orc_lp_to_float(run, lp) +
                                      orc_lp_to_float(slices[j][i], lp), lp);
        s = orc_lp_to_float(run, lp);
        if (!isfinite(s))
            of = 1;
        gi = s * inv;
        g[i] = gi;
        sq = gi * gi;
        acc = acc + (double)sq;
    }
    *sumsq = acc;
    *overflow = of;
}

/* ------------------------------------------------------------------------
 * Decision.  [P2] §4.2: "gradient_clipping": 1.0 -- clip by the global L2
 * norm of the (unscaled, averaged) gradient, coef = clip / (norm + 1e-6)
 * when that is below 1.  [P2] §4.3: fp16 needs loss scaling -- the dynamic
 * rule: an overflow skips the step and halves S (floor 1), the step counter
 * does not advance; after growth_interval good steps S doubles.
 * growth_interval <= 0 keeps S static (the step is still skipped).
 * ---------------------------------------------------------------------- */
void orc_decide(double sumsq, double remote_sumsq, int32_t overflow,
                int32_t remote_overflow, float clip, float loss_scale,
                int64_t step, int32_t good_steps, int32_t growth_interval,
                float beta1, float beta2, orc_decision *out)
{
    double norm = sqrt(sumsq + remote_sumsq);
    int32_t skip = (overflow != 0) || (remote_overflow != 0);
    float coef = 1.0f;
    int64_t t = step;
    if (clip > 0.0f) {
        double c = (double)clip / (norm + 1e-6);
        if (c < 1.0)
            coef = (float)c;
    }
    out->norm = norm;
    out->coef = coef;
    out->skip = skip;
    if (skip) {
        out->new_scale = growth_interval > 0 ? fmaxf(loss_scale * 0.5f, 1.0f)
                                             : loss_scale;
        out->good_steps = 0;
    } else {
        int32_t good = good_steps + 1;
        float s = loss_scale;
        if (growth_interval > 0 && good >= growth_interval) {
            s = loss_scale * 2.0f;
            good = 0;
        }
        out->new_scale = s;
        out->good_steps = good;
        t = step + 1;
    }
    out->step = t;
    out->bc1 = (float)(1.0 - pow((double)beta1, (double)t));
    out->bc2 = (float)(1.0 - pow((double)beta2, (double)t));
}

/* ------------------------------------------------------------------------
 * Adam (Kingma & Ba, bias-corrected, eps outside the square root), AdamW
 * decoupled decay (Loshchilov & Hutter), on the fp32 master / m / v of one
 * partition ([P1], [P4] §10.6.2 Step 3), then the new weights rounded to the
 * low-precision parameter ([P4] §10.6.2 Step 4 destination).
 * Per element, in this order, each op rounded on its own:
 *   g'   = g * coef                 (+ wd * w first when adamw == 0: L2)
 *   m    = b1 * m + (1 - b1) * g'
 *   v    = b2 * v + (1 - b2) * (g' * g')
 *   upd  = (lr * (m / bc1)) / (sqrt(v / bc2) + eps)
 *   w    = w * (1 - lr * wd)        (adamw == 1; factor rounded once)
 *   w    = w - upd
 * ---------------------------------------------------------------------- */
void orc_adam(int64_t len, const float *g, float *master, float *m, float *v,
              uint16_t *param_lp, int32_t lp, float coef, int32_t skip,
              float lr, float beta1, float beta2, float eps, float wd,
              int32_t adamw, float bc1, float bc2)
{
    const float omb1 = 1.0f - beta1;
    const float omb2 = 1.0f - beta2;
    const float decay = (float)(1.0 - (double)lr * (double)wd);
    if (skip)
        return;
    for (int64_t i = 0; i < len; ++i) {
        float gi = g[i] * coef;
        float w = master[i];
        float mi, vi, mhat, vhat, denom, upd;
        if (!adamw)
            gi = gi + wd * w;
        mi = beta1 * m[i] + omb1 * gi;
        vi = beta2 * v[i] + omb2 * (gi * gi);
        mhat = mi / bc1;
        vhat = vi / bc2;
        denom = sqrtf(vhat) + eps;
        upd = (lr * mhat) / denom;
        if (adamw)
            w = w * decay;
        w = w - upd;
        master[i] = w;
        m[i] = mi;
        v[i] = vi;
        if (param_lp)
            param_lp[i] = orc_float_to_lp(w, lp);
    }
}

/* ------------------------------------------------------------------------
 * Gather.  [P4] §10.6.1 All-Gather: the N slices are concatenated in rank
 * order so every rank holds the whole; §10.6.4 forward step 1 applies it to
 * one layer.
 * ---------------------------------------------------------------------- */
void orc_gather(int32_t n, const uint16_t *const *shards, int64_t shard_len,
                uint16_t *out)
{
    for (int32_t j = 0; j < n; ++j)
        for (int64_t k = 0; k < shard_len; ++k)
            out[(int64_t)j * shard_len + k] = shards[j][k];
}

/* ------------------------------------------------------------------------
 * Quantized all-gather.  [P1] "ZeRO++": ZeRO++ quantizes the parameters that
 * the all-gather moves.  Symmetric int8 with one scale per block (the pages
 * give no block size or rounding rule; the readings are listed in the design
 * notes): the largest magnitude of the block maps to 127.
 * ---------------------------------------------------------------------- */
void orc_quantize_blocks(int64_t len, const uint16_t *x, int32_t lp, int32_t block,
                         int8_t *q, float *scales)
{
    for (int64_t b0 = 0; b0 < len; b0 += block) {
        float amax = 0.0f, scale;
        for (int32_t k = 0; k < block; ++k) {
            float a = fabsf(orc_lp_to_float(x[b0 + k], lp));
            if (a > amax)
                amax = a;
        }
        scale = amax / 127.0f;
        scales[b0 / block] = scale;
        for (int32_t k = 0; k < block; ++k) {
            float r = 0.0f;
            if (scale > 0.0f) {
                r = nearbyintf(orc_lp_to_float(x[b0 + k], lp) / scale);
                if (r > 127.0f)
                    r = 127.0f;
                if (r < -127.0f)
                    r = -127.0f;
            }
            q[b0 + k] = (int8_t)r;
        }
    }
}

void orc_dequant_gather(int32_t n, const int8_t *const *q, const float *const *scales,
                        int64_t shard_len, int32_t block, int32_t lp, uint16_t *out)
{
    for (int32_t j = 0; j < n; ++j)
        for (int64_t k = 0; k < shard_len; ++k) {
            float y = (float)q[j][k] * scales[j][k / block];
            out[(int64_t)j * shard_len + k] = orc_float_to_lp(y, lp);
        }
}

/* ------------------------------------------------------------------------
 * fp8 (OCP E4M3) variant of the quantized all-gather.  The format follows
 * its definition: code s.eeee.mmm is (-1)^s * m/8 * 2^-6 when eeee = 0 and
 * (-1)^s * (1 + m/8) * 2^(eeee - 7) otherwise; eeee.mmm = 1111.111 is NaN.
 * ---------------------------------------------------------------------- */
float orc_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    float mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexpf((float)m, -9);
    else
        mag = ldexpf((float)(8 + m), e - 10);
    return s ? -mag : mag;
}

/* Nearest code, ties to even: the magnitude is rounded on the grid of its
 * binade (step 2^(E-3) for a normal binade 2^E, E >= -6; step 2^-9 below
 * 2^-6), then the code whose value it is is looked up among the 127
 * non-negative finite codes. */
uint8_t orc_e4m3_encode(float v)
{
    uint8_t s = signbit(v) ? 0x80 : 0x00;
    float a, step, r;
    int E, c;
    if (isnan(v))
        return 0x7f;
    a = fabsf(v);
    if (a >= 464.0f)          /* past the midpoint between 448 and 480: saturate */
        return s | 0x7e;
    if (a == 0.0f)
        return s;
    frexpf(a, &E);            /* a = f * 2^E, f in [0.5, 1): binade 2^(E-1) */
    E = E - 1;
    if (E < -6)
        E = -6;
    step = ldexpf(1.0f, E - 3);
    r = nearbyintf(a / step) * step;   /* a / step is exact (power of two) */
    for (c = 0; c < 0x7f; ++c)
        if (orc_e4m3_decode((uint8_t)c) == r)
            return s | (uint8_t)c;
    return 0xff;              /* unreachable: every rounded magnitude is a code */
}

void orc_e4m3_decode_array(int64_t n, const uint8_t *c, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_decode(c[i]);
}

void orc_e4m3_encode_array(int64_t n, const float *v, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_quantize_blocks_fp8(int64_t len, const uint16_t *x, int32_t lp, int32_t block,
                             uint8_t *q, float *scales)
{
    for (int64_t b0 = 0; b0 < len; b0 += block) {
        float amax = 0.0f, inv;
        int e, E;
        for (int32_t k = 0; k < block; ++k) {
            float a = fabsf(orc_lp_to_float(x[b0 + k], lp));
            if (a > amax)
                amax = a;
        }
        if (amax == 0.0f) {
            scales[b0 / block] = 0.0f;
            for (int32_t k = 0; k < block; ++k)
                q[b0 + k] = 0;
            continue;
        }
        if (isinf(amax)) {
            e = 120;
        } else {
            frexpf(amax, &E);     /* floor(log2 amax) = E - 1 */
            e = E - 1 - 7;
            if (e < -126)
                e = -126;
            if (e > 120)
                e = 120;
        }
        scales[b0 / block] = ldexpf(1.0f, e);
        inv = ldexpf(1.0f, -e);
        for (int32_t k = 0; k < block; ++k)
            q[b0 + k] = orc_e4m3_encode(orc_lp_to_float(x[b0 + k], lp) * inv);
    }
}

void orc_dequant_gather_fp8(int32_t n, const uint8_t *const *q, const float *const *scales,
                            int64_t shard_len, int32_t block, int32_t lp, uint16_t *out)
{
    for (int32_t j = 0; j < n; ++j)
        for (int64_t k = 0; k < shard_len; ++k) {
            float y = orc_e4m3_decode(q[j][k]) * scales[j][k / block];
            out[(int64_t)j * shard_len + k] = orc_float_to_lp(y, lp);
        }
}
