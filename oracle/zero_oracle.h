/*
 * zero_oracle.h -- plain, slow CPU oracle of the ZeRO partitioned
 * mixed-precision Adam step over a flat, padded parameter buffer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * calls it.
 *
 * Sources (web pages on ZeRO; each function below names the passage it
 * follows):
 *   [P1] "ZeRO-1/2/3 分别优化了什么？和普通 DDP 有什么区别？" (interview note)
 *   [P2] "从'年糕切片'理解ZeRO的核心思想" (blog; §2.2 reduce_bucket_size,
 *        §4.2 gradient_clipping, §4.3 loss scaling)
 *   [P3] "第13篇 · ZeRO" reading notes of arXiv:1910.02054 (§2.2 16Ψ,
 *        §3.2 stage formulas, §3.3 Figure 1 / Table 1 worked numbers,
 *        §3.4 communication volume, §3.7 self-test answers)
 *   [P4] "10.6 ZeRO 与 FSDP" (§10.6.1 collectives, §10.6.2–10.6.4 stage
 *        flows, §10.6.5 Table 10-2, §10.6.7 FSDP units)
 * The pages do not write out Adam, the clipping rule or the loss-scale rule;
 * those follow Kingma & Ba (Adam, bias-corrected, eps outside the sqrt) and
 * Loshchilov & Hutter (decoupled weight decay), as listed in the design notes.
 *
 * Low-precision values travel as raw 16-bit codes (uint16_t): lp = 0 is IEEE
 * binary16 (fp16), lp = 1 is bfloat16.
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats (IEEE 754 binary16; bfloat16 = top half of binary32) */
float    orc_half_to_float(uint16_t h);
uint16_t orc_float_to_half(float f);
float    orc_bf16_to_float(uint16_t b);
uint16_t orc_float_to_bf16(float f);
float    orc_lp_to_float(uint16_t x, int32_t lp);
uint16_t orc_float_to_lp(float f, int32_t lp);
/* whole-array conversions (tests and input preparation) */
void orc_lp_array_to_float(int64_t n, const uint16_t *x, int32_t lp, float *out);
void orc_float_array_to_lp(int64_t n, const float *x, int32_t lp, uint16_t *out);

/* ---- flat layout and partitions ([P3] §2.1 item 3 flat buffer,
 *      [P4] §10.6.2 "1/N 分片", §10.6.7 FSDP units) ---------------------
 * stage 0 (DDP) / 1 / 2: one unit holding every tensor.
 * stage 3: tensors grouped into units by unit_of_tensor (non-decreasing,
 *          starting at 0, no gaps); each unit padded on its own.
 * Returns 0 on success, -1 on invalid arguments.
 * tensor_offsets[n_tensors]: flat offset of each tensor.
 * unit_offsets[n_units + 1], unit_padded[n_units]: where each padded unit
 * starts in the flat buffer and its padded length U_p.               */
int32_t orc_layout(int32_t n_tensors, const int64_t *sizes,
                   const int32_t *unit_of_tensor, int32_t n_ranks,
                   int32_t align, int32_t stage,
                   int64_t *psi, int64_t *psi_padded, int64_t *part_len,
                   int32_t *n_units, int64_t *tensor_offsets,
                   int64_t *unit_offsets, int64_t *unit_padded);

/* Flat-buffer index of element k of rank r's partition (-1 if out of range).
 * Needs the unit table from orc_layout.                                   */
int64_t orc_partition_to_flat(int32_t n_units, const int64_t *unit_offsets,
                              const int64_t *unit_padded, int32_t n_ranks,
                              int32_t stage, int32_t rank, int64_t k);

/* Fragments of rank r's partition: each maximal run of partition elements
 * that lies inside one tensor, in partition order, as 4 int64 per fragment:
 * (tensor id, offset inside the tensor, offset inside the partition, length).
 * Writes at most max_frag fragments; returns how many exist.             */
int64_t orc_fragments(int32_t n_tensors, const int64_t *sizes,
                      const int32_t *unit_of_tensor, int32_t n_ranks,
                      int32_t align, int32_t stage, int32_t rank,
                      int64_t max_frag, int64_t *frag);

/* ---- model-state accounting ([P4] Table 10-2; [P3] §3.2, §3.4) --------
 * formula[4]: the pages' per-GPU bytes 16Ψ, 4Ψ+12Ψ/N, 2Ψ+14Ψ/N, 16Ψ/N
 *             (exact rational value, rounded once to double).
 * actual[4] : the same with the padded layout (Ψ_p = Ψ rounded up to N·align,
 *             P = Ψ_p/N): 16Ψ, 4Ψ_p+12P, 2Ψ_p+14P, 16P.
 * comm[4]   : elements moved per step: 2Ψ (DDP), 2Ψ, 2Ψ, 3Ψ.             */
int32_t orc_memory(int64_t psi, int32_t n_ranks, int32_t align,
                   double formula[4], int64_t actual[4], int64_t comm[4]);

/* ---- reduce of N ranks' gradient slices into one partition -----------
 * [P4] §10.6.1 Reduce-Scatter (sum), [P1] ZeRO-2 (average), [P2] §4.3 loss
 * scale.  For each i: s = g_0[i] + g_1[i] + ... + g_{N-1}[i] in float, in
 * rank order; g[i] = s * inv, inv = float(1 / (S * N)); overflow if any s is
 * not finite; sumsq = sum over i of double(float(g*g)), index order.      */
void orc_reduce(int32_t n, const uint16_t *const *slices, int32_t lp,
                int64_t len, float loss_scale, float *g, double *sumsq,
                int32_t *overflow);

/* Same, with the sum kept in the low-precision type: each partial sum is
 * rounded to fp16/bf16 (nearest, ties to even) before the next rank's value
 * is added -- the reduce_dtype=float16 mixed-precision setting of "10.6 ZeRO
 * 与 FSDP" §10.6.7.  Rank order 0..N-1; the final lp sum is widened to float,
 * multiplied by float(1/(S*N)); overflow if that sum is not finite.        */
void orc_reduce_lp_accum(int32_t n, const uint16_t *const *slices, int32_t lp,
                         int64_t len, float loss_scale, float *g,
                         double *sumsq, int32_t *overflow);

/* ---- global-norm clip, skip and loss-scale decision -------------------
 * [P2] §4.2 "gradient_clipping": 1.0, §4.3 loss scaling.                  */
typedef struct {
    double  norm;        /* sqrt(sumsq + remote_sumsq)                  */
    float   coef;        /* clip / (norm + 1e-6) when < 1, else 1       */
    int32_t skip;        /* overflow seen on any rank                   */
    float   new_scale;   /* loss scale for the next step                */
    int32_t good_steps;  /* consecutive non-skipped steps since growth  */
    int64_t step;        /* Adam step counter t after this step         */
    float   bc1, bc2;    /* 1 - beta1^t, 1 - beta2^t (rounded to float) */
} orc_decision;

void orc_decide(double sumsq, double remote_sumsq, int32_t overflow,
                int32_t remote_overflow, float clip, float loss_scale,
                int64_t step, int32_t good_steps, int32_t growth_interval,
                float beta1, float beta2, orc_decision *out);

/* ---- Adam / AdamW on the fp32 master, m, v of one partition ----------
 * [P1] 优化器状态 (fp32 master + m + v = 12Ψ); [P4] §10.6.2 Step 3 local
 * update, Step 4 all-gather destination.  param_lp (nullable) receives the
 * new master rounded to fp16/bf16.  No writes at all when skip != 0.      */
void orc_adam(int64_t len, const float *g, float *master, float *m, float *v,
              uint16_t *param_lp, int32_t lp, float coef, int32_t skip,
              float lr, float beta1, float beta2, float eps, float wd,
              int32_t adamw, float bc1, float bc2);

/* ---- stage-3 layer gather ([P4] §10.6.4 forward step 1, all-gather) ---
 * out[j * shard_len + k] = shards[j][k].                                  */
void orc_gather(int32_t n, const uint16_t *const *shards, int64_t shard_len,
                uint16_t *out);

/* ---- quantized all-gather ([P1] "ZeRO++": the all-gathered parameters are
 * quantized to cut the traffic) ------------------------------------------
 * Blocks of `block` consecutive elements share one float scale:
 *   amax  = max |x| over the block (x = the lp parameter widened to float)
 *   scale = amax / 127                               (float division)
 *   q     = nearest integer to x / scale, ties to even, in [-127, 127]
 *           (q = 0 when scale == 0)
 * and the receiver's value is lp(q * scale) (float product, rounded to lp).
 * len must be a multiple of block.                                        */
void orc_quantize_blocks(int64_t len, const uint16_t *x, int32_t lp, int32_t block,
                         int8_t *q, float *scales);
/* out[j * shard_len + k] = lp(q_j[k] * scale_j[k / block]) */
void orc_dequant_gather(int32_t n, const int8_t *const *q, const float *const *scales,
                        int64_t shard_len, int32_t block, int32_t lp, uint16_t *out);

/* ---- fp8 variant of the quantized all-gather ---------------------------
 * Codes are OCP FP8 E4M3 ("e4m3fn": 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448;
 * subnormals m * 2^-9).  Encoding rounds to nearest, ties to even, and
 * saturates finite values beyond 448 (and infinities) to +-448; NaN -> 0x7f.
 * Blocks of `block` elements share a power-of-two scale 2^e with
 *   e = floor(log2 amax) - 7, clamped to [-126, 120]  (amax finite > 0),
 *   e = 120 when amax is infinite,
 * so amax / 2^e lies in [128, 256) and no finite value saturates:
 *   code = e4m3(x * 2^-e)   (one float multiply, then the encoding)
 *   scale = 2^e (0 and every code 0 when amax == 0)
 * and the receiver's value is lp(decode(code) * scale).                   */
float orc_e4m3_decode(uint8_t c);
uint8_t orc_e4m3_encode(float v);
void orc_e4m3_decode_array(int64_t n, const uint8_t *c, float *out);
void orc_e4m3_encode_array(int64_t n, const float *v, uint8_t *out);
void orc_quantize_blocks_fp8(int64_t len, const uint16_t *x, int32_t lp, int32_t block,
                             uint8_t *q, float *scales);
/* out[j * shard_len + k] = lp(decode(q_j[k]) * scale_j[k / block]) */
void orc_dequant_gather_fp8(int32_t n, const uint8_t *const *q, const float *const *scales,
                            int64_t shard_len, int32_t block, int32_t lp, uint16_t *out);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_ORACLE_H */
