/*
 * zero.h -- C ABI of libzero: the ZeRO partitioned mixed-precision Adam step
 * over a flat, padded parameter buffer, on one NVIDIA GB300 (sm_103a).
 *
 * What the library computes (the sources are web pages on ZeRO):
 *  - "10.6 ZeRO 与 FSDP" §10.6.2–§10.6.4: per step, each of N data-parallel
 *    ranks reduce-scatters the gradients so it holds the reduced 1/N slice
 *    of its partition (Step 2), updates its 1/N of the fp32 optimizer state
 *    and parameters locally (Step 3) and all-gathers the new parameters into
 *    the full layout (Step 4, stages 1/2); stage 3 instead all-gathers each
 *    layer's parameter shards when the layer is needed (§10.6.4).
 *  - Table 10-2 of the same page: per-GPU bytes 16Ψ, 4Ψ+12Ψ/N, 2Ψ+14Ψ/N,
 *    16Ψ/N and communication 2Ψ, 2Ψ, 2Ψ, 3Ψ.
 *  - "从'年糕切片'理解ZeRO" §4.2–§4.3: gradient clipping 1.0 and fp16 loss
 *    scaling.
 *  - "第13篇 · ZeRO" §2.1 item 3: gradients live in one flat buffer.
 * On one GPU, the N ranks' gradient slices and parameter shards are N
 * separate device buffers supplied by the caller.
 *
 * Conventions for every call:
 *  - Device pointers are caller-owned CUDA device memory on the current
 *    device and must be 16-byte aligned; lengths are element counts.
 *    The library never frees or retains caller memory after a call returns
 *    (kernels launched by the call may still be reading/writing it on
 *    `stream`).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *    device work of a call is enqueued on it; calls return without waiting,
 *    except the ones documented as synchronising.  A synchronising call waits
 *    for the plan's own device work only (an event recorded after each of its
 *    calls on each stream it used), never for other streams or other plans;
 *    it reads and writes the plan's record on a private non-blocking stream.
 *  - Errors are returned as zero_status codes; nothing is thrown.
 *    zero_last_error() gives a message for the last failure on the calling
 *    thread.  On an argument or state error, no device work has been
 *    enqueued by that call (a call that launches several kernels and meets a
 *    CUDA launch failure part-way may have enqueued the earlier ones).
 *  - A plan holds host-side step state: calls on one plan must not run
 *    concurrently from several host threads; different plans are independent.
 *  - CUDA graphs: once a plan has run one step eagerly (its first device call
 *    allocates its scratch), the asynchronous calls of a step (reduces,
 *    zero_adam_step / _range, gathers, quantize) can be captured on a stream
 *    and the graph replayed; each replay is one step with the arguments of
 *    capture time (the step counter, loss scale and skip logic stay on the
 *    device).  The synchronising calls are not capturable.  Once any call of
 *    a plan has been captured, the plan cannot know where its graph is
 *    replayed, so its synchronising calls wait for the whole device from then
 *    on (cudaDeviceSynchronize).
 *  - Low-precision ("lp") values are IEEE binary16 (ZERO_FP16) or bfloat16
 *    (ZERO_BF16), chosen per plan.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct zero_plan zero_plan; /* opaque, owned by the library */

typedef enum {
    ZERO_OK = 0,
    ZERO_EINVAL = 1,   /* bad argument: NULL, negative size, rank >= N ... */
    ZERO_EALIGN = 2,   /* a device pointer is not 16-byte aligned           */
    ZERO_ENOMEM = 3,   /* host or device allocation of plan scratch failed */
    ZERO_ECUDA = 4,    /* a CUDA runtime call failed (see zero_last_error) */
    ZERO_ETIMEOUT = 5, /* a bounded device wait ran out (Adam or gather)   */
    ZERO_ESTATE = 6    /* call out of order (e.g. Adam before any reduce)  */
} zero_status;

typedef enum { ZERO_FP16 = 0, ZERO_BF16 = 1 } zero_lp;

#define ZERO_MAX_RANKS 1024

/* Elements per norm tile: the reduce writes one fp64 partial sum of squares
 * per tile of each partition (per unit shard in stage 3); buckets are rounded
 * up to whole tiles. */
#define ZERO_NORM_TILE 4096

/* ----------------------------------------------------------------------
 * Plan: the flat-buffer partitioner.
 *
 * The flat buffer holds the tensors back to back in list order with no
 * per-tensor padding ("第13篇 · ZeRO" §2.1 item 3), then zero padding up to
 * a multiple of n_ranks * align so that N equal partitions of length
 * P = Ψ_p / N exist ("10.6 ZeRO 与 FSDP" §10.6.2).  Rank r owns
 * [r*P, (r+1)*P).  Padding elements are not parameters: their gradients
 * must be zero, and then their master/m/v/param stay exactly zero.
 *
 * stage 0 = DDP (no partitioning: one replica, rank must be 0, P = Ψ_p),
 * stage 1/2 = ZeRO-1/2 (same arithmetic on the rank's partition; the stages
 * differ only in what the caller keeps, see zero_memory_report),
 * stage 3 = ZeRO-3: tensors are grouped into units (unit_of_tensor:
 * non-decreasing, starting at 0, no gaps; NULL = one unit).  Each unit is
 * padded on its own to a multiple of N*align and sharded N ways ("10.6" §10.6.7
 * FSDP units); rank r's partition is the concatenation, in unit order, of
 * its shard of every unit.
 *
 * psi: total parameter count; with tensor_sizes == NULL the buffer is one
 * tensor of psi elements; with a tensor list, psi must equal the sum of the
 * sizes, or be -1 to take the sum.  align: elements, a positive multiple of
 * 8 (so every partition starts on a 16-byte boundary).  n_ranks in
 * [1, ZERO_MAX_RANKS].
 * Allocates no device memory (scratch is allocated on the first device call).
 */
zero_status zero_plan_create(int64_t psi, int32_t n_ranks,
                             const int64_t *tensor_sizes, int32_t n_tensors,
                             int32_t align, int32_t stage,
                             const int32_t *unit_of_tensor, zero_lp lp,
                             zero_plan **out);

/* Padded length Ψ_p, partition length P, and (nullable) the flat offset of
 * each tensor: n_tensors entries, or one entry (0) for a plan created from psi
 * alone, whose buffer is one tensor.  Host only. */
zero_status zero_plan_query(const zero_plan *plan, int64_t *psi_padded,
                            int64_t *part_len, int64_t *tensor_offsets);

/* Stage-3 unit table (one unit in stages 0-2): n_units, unit_offsets
 * (n_units + 1 entries: flat start of each padded unit, then Ψ_p) and
 * unit_padded (U_p per unit).  Either array may be NULL.  Host only. */
zero_status zero_plan_units(const zero_plan *plan, int32_t *n_units,
                            int64_t *unit_offsets, int64_t *unit_padded);

/* Each unit's shard within a rank's partition (the same for every rank):
 * shard_len[u] = U_p / N (stage 0: U_p) and shard_offset[u] = the sum of the
 * shard lengths of units 0 .. u-1.  n_units entries each; either array may be
 * NULL.  Host only. */
zero_status zero_plan_unit_shards(const zero_plan *plan, int64_t *shard_len,
                                  int64_t *shard_offset);

/* Fragments of rank r's partition: maximal runs of partition elements lying
 * in one tensor, in partition order, 4 int64 each: (tensor id, offset in the
 * tensor, offset in the partition, length).  Writes min(count, max_frag)
 * fragments into frag (nullable when max_frag == 0); *count gets the total.
 * Partition positions covered by no fragment are padding.  Host only. */
zero_status zero_plan_fragments(const zero_plan *plan, int32_t rank,
                                int64_t max_frag, int64_t *frag,
                                int64_t *count);

/* Dynamic loss-scale rule ("从'年糕切片'理解ZeRO" §4.3): on overflow the step
 * is skipped and S halves (floor 1); after growth_interval consecutive good
 * steps S doubles.  growth_interval <= 0 keeps S static (overflowing steps
 * are still skipped).  Default 1000.  Host only. */
zero_status zero_plan_set_loss_scaler(zero_plan *plan, int32_t growth_interval);

/* Reduce precision ("10.6 ZeRO 与 FSDP" §10.6.7: MixedPrecision with
 * reduce_dtype=float16, gradients communicated and summed in fp16).
 * accumulate_in_lp = 0 (default): the N slices are summed in float.
 * accumulate_in_lp = 1: every partial sum is rounded to the plan's lp type
 * (nearest, ties to even) before the next rank's value is added, in rank
 * order; the final lp sum is then widened, unscaled and checked as usual
 * (an lp overflow shows up as an overflow).  Host only. */
zero_status zero_plan_set_reduce_precision(zero_plan *plan, int32_t accumulate_in_lp);

/* Resume: set the device step counter t and the good-step count (e.g. from a
 * checkpoint).  Synchronising: waits for the plan's own device work first. */
zero_status zero_plan_set_state(zero_plan *plan, int64_t step,
                                int32_t good_steps);

/* Bound on the polls of each device-side pipeline wait (mbarrier try_wait)
 * of the calls launched after it: zero_adam_step / _range, zero_gather_layer
 * and zero_allgather_params.  Default 2^22; 0 makes every such wait give up
 * at once (used to test the timeout path).  A wait that gives up sets the
 * plan's error word and the kernel stops early: zero_adam_step then leaves
 * every 1024-element tile it had not yet stored untouched (master, m, v and
 * param keep their old values there), a gather leaves part of its output
 * unwritten.  Bulk loads already issued are always waited for (with a fixed
 * bound) before a CTA exits.  The next synchronising call (zero_step_result
 * or zero_plan_check) returns ZERO_ETIMEOUT.  The decision of the step is
 * taken before Adam runs, so after a timed-out zero_adam_step the step
 * counter has advanced; restore it with zero_plan_set_state before redoing
 * the step.  Host only. */
zero_status zero_plan_set_spin_limit(zero_plan *plan, int64_t polls);

/* ----------------------------------------------------------------------
 * Reduce ("10.6 ZeRO 与 FSDP" §10.6.1 Reduce-Scatter, §10.6.2 Step 2; average
 * over ranks per "ZeRO-1/2/3 vs DDP" ZeRO-2; unscale per "年糕切片" §4.3).
 *
 * grad_slices: N pointers; grad_slices[j] holds P lp elements, rank j's
 * gradient over rank `rank`'s partition.  They may be device memory of the
 * current device, managed memory, pinned host memory (cudaHostAlloc /
 * cudaHostRegister: the kernel then reads it in place, over NVLink-C2C on
 * Grace systems, with no staging copy), or pageable host memory where the
 * device reads host page tables; anything else is ZERO_EINVAL.  For i < P:
 *   s = g_0[i] + g_1[i] + ... + g_{N-1}[i]   (float, in rank order)
 *   grad_out[i] = s * float(1 / (loss_scale * N))
 * and, over the partition, the overflow flag (any s not finite) and the
 * partial sums of grad_out^2 that feed the global norm.
 * grad_out: P floats (device).  bucket_elems: reduce in buckets of this many
 * elements (rounded up to a whole number of 4096-element norm tiles, so
 * results are bit-identical for every bucket size); 0 = one bucket.  In
 * stage 3 buckets and tiles are counted within each unit's shard.
 * The first reduce after a step's Adam call starts a new step; every
 * partition reduced before the next zero_adam_step joins that step's norm
 * and overflow decision.  Stage 0: rank must be 0, slices hold Ψ_p elements.
 */
zero_status zero_reduce_partition(zero_plan *plan, int32_t rank,
                                  const void *const *grad_slices,
                                  float *grad_out, float loss_scale,
                                  int64_t bucket_elems, void *stream);

/* Several partitions in one call (one process simulating several ranks, or
 * owning several partitions): exactly the results of calling
 * zero_reduce_partition for ranks[0], ..., ranks[n_parts-1] in that order,
 * bit for bit, in fewer kernel launches.  grad_slices: n_parts * N pointers,
 * partition-major (the N slices of ranks[i] at [i*N, (i+1)*N)); grad_out:
 * n_parts pointers.  The ranks must be distinct (ZERO_EINVAL).  The pieces of
 * every partition (bucket_elems as for zero_reduce_partition) share launches:
 * a launch takes consecutive pieces while they hold at most bucket_elems
 * elements in total (all of them when bucket_elems is 0), at most 64 pieces
 * and the slice pointers of floor(512/N) partitions when N <= 64, of
 * floor(1024/N) when N > 64.  Every argument is validated before any launch. */
zero_status zero_reduce_partitions(zero_plan *plan, int32_t n_parts, const int32_t *ranks,
                                   const void *const *grad_slices, float *const *grad_out,
                                   float loss_scale, int64_t bucket_elems, void *stream);

/* Stage 3: reduce only units [first_unit, first_unit + n_units) of rank
 * `rank`'s partition ("10.6 ZeRO 与 FSDP" §10.6.4 backward step 4: each
 * layer's gradients are reduce-scattered once its backward is done, in
 * reverse layer order; "年糕切片" §2.2 reduce_bucket_size: a bucket collects
 * several layers before it is reduced).  Same arguments and arithmetic as
 * zero_reduce_partition (the slices and grad_out are whole-partition
 * buffers; only the units' range is read and written), in one kernel launch
 * per 64 units; the units join the current step like a partition.  The
 * norm's tiles restart at every unit, so reducing the units in any grouping
 * and order gives exactly the bits of one zero_reduce_partition call. */
zero_status zero_reduce_units(zero_plan *plan, int32_t rank, int32_t first_unit,
                              int32_t n_units, const void *const *grad_slices,
                              float *grad_out, float loss_scale, void *stream);

/* Multi-rank use (one process per rank; "10.6 ZeRO 与 FSDP" §10.6.1: the
 * global norm and overflow need an all-reduce over the ranks; "年糕切片" §4.2
 * global clipping).  Each rank reduces the partitions it owns, then exports
 * its per-partition statistics:
 *   stats: 2*N doubles (N = n_ranks), device memory of the current device,
 *   managed or pinned host memory, 8-byte aligned.  Written on `stream`:
 *     stats[p]     = sum over partition p's reduced gradient of g^2, added in
 *                    the library's fixed order (one fp64 partial per norm
 *                    tile, a fixed tree over chunks of tiles), if partition p
 *                    was reduced in the current step (stage 0: p = 0), else +0;
 *     stats[N + p] = 1.0 if one of partition p's sums was not finite, else 0.
 * Asynchronous; valid after the step's reduces, before its first Adam call.
 * A partition is reduced by exactly one rank, so the element-wise sum of every
 * rank's vector (an all-reduce with sum, in any order) adds only exact zeros:
 * it equals, bit for bit, the vector of a single process that reduced every
 * partition. */
zero_status zero_partition_stats(zero_plan *plan, double *stats, void *stream);

/* Make this step's decision use an all-reduced statistics vector (2*N
 * doubles, the layout of zero_partition_stats; same memory kinds) instead of
 * the plan's own partitions and the remote_* arguments:
 *   sumsq = the per-partition sums added in partition order by the fixed
 *           tree the single-process decision uses;  skip = any stats[N + p] != 0.
 * Every rank holding the same vector takes the bit-identical decision, equal
 * to the single-process decision over all N partitions.  Host only: the vector
 * is read by the decision kernel that the step's first zero_adam_step (or
 * _range) launches, on that call's stream, so it must hold the summed values
 * by then (e.g. all-reduced on the same stream) and stay unchanged until that
 * kernel has run.  Valid after the step's reduces and before its first Adam
 * call (ZERO_ESTATE otherwise). */
zero_status zero_step_set_global_stats(zero_plan *plan, const double *stats);

/* ----------------------------------------------------------------------
 * Decision + fused Adam/AdamW + cast ("10.6 ZeRO 与 FSDP" §10.6.2 Steps 3-4;
 * "年糕切片" §4.2 clipping, §4.3 loss scaling).
 *
 * The first zero_adam_step of a step decides, on the device:
 *   norm = sqrt(sum of squares of every reduced partition + remote_sumsq)
 *   coef = clip / (norm + 1e-6) if clip > 0 and that is < 1, else 1
 *   skip = overflow of any reduced partition or remote_overflow != 0
 *   skip:  S' = max(S/2, 1) (dynamic) or S (static); t unchanged
 *   else:  t = t + 1; after growth_interval good steps S' = 2S
 * Later zero_adam_step calls of the same step (other ranks) reuse that
 * decision (their loss_scale, clip and remote_* arguments are ignored).
 * Then, unless skip, for each i < P of rank `rank`'s partition, each float
 * op rounded to nearest on its own (no fused multiply-add):
 *   g' = grad[i] * coef;  adamw == 0: g' = g' + wd * master[i]   (L2 Adam)
 *   m  = b1*m + (1-b1)*g';   v = b2*v + (1-b2)*(g'*g')
 *   upd = (lr * (m / bc1)) / (sqrt(v / bc2) + eps),
 *         bc1 = float(1 - b1^t), bc2 = float(1 - b2^t)  (power and difference in
 *         double, then rounded once)
 *   adamw != 0: master = master * float(1 - lr*wd)   (decoupled decay)
 *   master = master - upd;  param = round-to-nearest-even lp(master)
 * grad, master, m, v: P floats (device).  param_out: lp, device; stages 0-2:
 * the full Ψ_p-element layout (the all-gather destination; this rank writes
 * [rank*P, (rank+1)*P)); stage 3: rank's own P-element shard buffer (there
 * is no step-end all-gather, "10.6" §10.6.4).  param_out may be NULL (no
 * cast).  loss_scale: the S used by this step's reduces.
 */
zero_status zero_adam_step(zero_plan *plan, int32_t rank, const float *grad,
                           float *master, float *m, float *v, void *param_out,
                           float lr, float beta1, float beta2, float eps,
                           float wd, int32_t adamw, float loss_scale,
                           float clip, double remote_sumsq,
                           int32_t remote_overflow, void *stream);

/* Optimizer sub-groups ("10.6 ZeRO 与 FSDP" §10.6.6, the ds_config key
 * sub_group_size: the flat partition is stepped a sub-group of elements at a
 * time).  zero_adam_step restricted to partition elements [begin, begin +
 * len): the same decision (taken by the first call of the step, range or
 * whole), the same per-element arithmetic, so stepping a partition in
 * sub-groups, in any order and grouping, gives exactly the bits of one
 * zero_adam_step call.  grad, master, m, v and param_out are the same
 * whole-partition (or whole-layout) pointers as for zero_adam_step; only the
 * range is read and written.  begin and len must be multiples of 8
 * (ZERO_EALIGN otherwise) with begin + len <= P (ZERO_EINVAL otherwise);
 * len = 0 only takes the decision if it is still due.  Each element must be
 * stepped once per step: the library does not track which ranges were done. */
zero_status zero_adam_step_range(zero_plan *plan, int32_t rank, int64_t begin,
                                 int64_t len, const float *grad, float *master,
                                 float *m, float *v, void *param_out, float lr,
                                 float beta1, float beta2, float eps, float wd,
                                 int32_t adamw, float loss_scale, float clip,
                                 double remote_sumsq, int32_t remote_overflow,
                                 void *stream);

/* Several partitions' updates in one call: exactly the results of calling
 * zero_adam_step for ranks[0], ..., ranks[n_parts-1] in that order with
 * these arguments, bit for bit (the first call of a step takes the decision),
 * in one kernel launch per 64 partitions.  grad, master, m, v, param_out:
 * n_parts pointers each, entry i as zero_adam_step takes it for ranks[i]
 * (param_out[i] may be NULL; stages 0-2: the full layout, to which the
 * library adds ranks[i]*P; stage 3: ranks[i]'s shard).  The ranks must be
 * distinct (ZERO_EINVAL).  Every argument is validated before any launch. */
zero_status zero_adam_step_partitions(zero_plan *plan, int32_t n_parts, const int32_t *ranks,
                                      const float *const *grad, float *const *master,
                                      float *const *m, float *const *v,
                                      void *const *param_out, float lr, float beta1,
                                      float beta2, float eps, float wd, int32_t adamw,
                                      float loss_scale, float clip, double remote_sumsq,
                                      int32_t remote_overflow, void *stream);

/* Decision of the last decided step: global norm, skipped flag, loss scale
 * for the next step, and the step counter t.  Any pointer may be NULL.
 * Synchronising: waits for the plan's own device work (not for other streams'
 * work).  Returns ZERO_ETIMEOUT (and clears it) if a bounded device wait gave
 * up since the last check. */
zero_status zero_step_result(zero_plan *plan, double *norm, int32_t *skipped,
                             float *new_loss_scale, int64_t *step);

/* Waits for the plan's own device work and reports (then clears) the plan's
 * device error word: ZERO_OK or ZERO_ETIMEOUT. */
zero_status zero_plan_check(zero_plan *plan);

/* ----------------------------------------------------------------------
 * Stage-3 layer gather ("10.6 ZeRO 与 FSDP" §10.6.4 forward/backward step 1:
 * All-Gather of one layer's parameters; §10.6.7 FSDP unit).
 * shards: N device pointers, shards[j] = rank j's P-element lp shard buffer
 * (the buffer zero_adam_step writes in stage 3).  out: U_p lp elements
 * (device) receiving unit `unit` in full layout:
 *   out[j * (U_p/N) + k] = shards[j][unit_shard_offset + k],  k < U_p/N.
 * Copies with TMA bulk transfers staged through shared memory; every device
 * wait is bounded (zero_plan_set_spin_limit).  Stage 3 plans only.
 */
zero_status zero_gather_layer(zero_plan *plan, int32_t unit,
                              const void *const *shards, void *out,
                              void *stream);

/* ----------------------------------------------------------------------
 * Stage-1/2 parameter all-gather after the update ("10.6 ZeRO 与 FSDP"
 * §10.6.2 Step 4: every rank's updated partition is all-gathered into the
 * full parameter layout), in buckets ("从'年糕切片'理解ZeRO" §4.2, the
 * ds_config key allgather_bucket_size).
 * partitions: N device pointers, partitions[j] = rank j's P updated lp
 * parameters (e.g. its range of its own full-layout buffer: out may be one
 * of them, partitions[j] == out + j*P gathers in place).  out: the Ψ_p-element
 * full layout (device):  out[j*P + k] = partitions[j][k],  k < P.
 * bucket_elems <= 0: one launch; else launches of N runs of
 * max(8, floor(bucket_elems / N / 8) * 8) elements each (one bucket of about
 * bucket_elems elements), in partition order.  Same TMA bulk copies and
 * bounded waits as zero_gather_layer.  Stage-1/2 plans only (ZERO_EINVAL);
 * pointers must be 16-byte aligned (ZERO_EALIGN).  Asynchronous on stream.
 */
zero_status zero_allgather_params(zero_plan *plan, const void *const *partitions,
                                  void *out, int64_t bucket_elems, void *stream);

/* ----------------------------------------------------------------------
 * Quantized stage-3 gather ("ZeRO-1/2/3 vs DDP" note, ZeRO++: the
 * all-gathered parameters are quantized to cut the traffic).  Stage-3 plans
 * whose align is a multiple of ZERO_QUANT_BLOCK.
 *
 * zero_quantize_shard: shard (P lp elements, this rank's own shard buffer)
 * -> codes (P bytes) and scales (P / ZERO_QUANT_BLOCK floats), per block of
 * ZERO_QUANT_BLOCK elements:
 *   amax = max |x|,  scale = amax / 127 (float division),
 *   code = nearest integer (ties to even) to x / scale, clamped to
 *          [-127, 127]; 0 when scale == 0.
 * zero_gather_layer_quantized: like zero_gather_layer, from every rank's
 * codes/scales (the buffers zero_quantize_shard wrote, whole-partition
 * pointers; the library adds the unit's offset):
 *   out[j * (U_p/N) + k] = lp(code_j[o + k] * scale_j[(o + k) / BLOCK])
 * with o the unit's shard offset; the product is a float multiply rounded to
 * the lp type (nearest even).  1 B + 4/128 B read per element instead of 2 B.
 * All pointers 16-byte aligned, device memory, asynchronous on `stream`.
 *
 * zero_plan_set_gather_quantization selects the code format of both calls
 * (the pages name no format; host only, default ZERO_QUANT_INT8):
 *  - ZERO_QUANT_INT8: the int8 codes above.
 *  - ZERO_QUANT_FP8_E4M3: each code byte is an OCP FP8 E4M3 value (bias 7,
 *    3 mantissa bits, largest 448, no infinities); per block the scale is the
 *    power of two 2^e with e = floor(log2 amax) - 7, clamped to [-126, 120]
 *    (120 when amax is infinite), so amax / 2^e is in [128, 256):
 *      code = E4M3(x * 2^-e), nearest even, finite overflow and infinities
 *             saturated to +-448 (never reached by finite blocks);
 *      scale = 2^e, or 0 with every code 0 when amax == 0;
 *    and the gather writes lp(decode(code) * scale).  Relative error up to
 *    2^-4 instead of int8's amax/254, with a wider dynamic range per block.
 *    Codes of non-finite elements are the hardware conversion's.
 */
#define ZERO_QUANT_BLOCK 128
#define ZERO_QUANT_INT8 0
#define ZERO_QUANT_FP8_E4M3 1
zero_status zero_plan_set_gather_quantization(zero_plan *plan, int32_t format);
zero_status zero_quantize_shard(zero_plan *plan, const void *shard, int8_t *codes,
                                float *scales, void *stream);
zero_status zero_gather_layer_quantized(zero_plan *plan, int32_t unit,
                                        const int8_t *const *codes,
                                        const float *const *scales, void *out,
                                        void *stream);

/* ----------------------------------------------------------------------
 * Allocation-free reduce.  The paper has no counterpart: this is a service
 * for callers that cannot allocate device memory -- e.g. code whose device
 * memory is entirely owned by a framework's caching allocator (an extra
 * cudaMalloc would fail or fragment that pool), or a latency-critical loop
 * that must not pay cudaMalloc's implicit synchronisation.
 *
 * Computes exactly what zero_reduce_partition computes for one partition in
 * one bucket (same kernel, same bits): grad_out[i] = (sum over j of
 * grad_slices[j][i]) * float(1/(loss_scale*n_ranks)) for i < len, plus
 * *sumsq_out (device double) = the partition's sum of grad_out^2, added in
 * the same fixed order, so it equals zero_partition_stats' entry for that
 * partition bit for bit, and *overflow_out (device int32) = 1 if any sum is
 * not finite, else 0.  No plan is involved and no step state is touched.
 *
 * Scratch: one fixed array of ZERO_NOALLOC_SCRATCH_BYTES in device memory
 * that belongs to the library image (present on every GPU that loads the
 * library until the process exits); no cudaMalloc/cudaFree or other
 * allocating call is made.  len is limited to ZERO_NOALLOC_MAX_ELEMS (a
 * multiple of 8); larger len returns ZERO_EINVAL.  Devices 0-63 only (the
 * array's address is kept per device; ZERO_EINVAL beyond).  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.
 * All calls share the array and it keeps the last call's contents (the
 * overflow word is cleared by every call); calls whose device work overlaps
 * in time (other streams or host threads) race on it and must be serialised
 * by the caller.  Inputs and outputs are caller-owned device memory, as for
 * every other call.  Asynchronous on `stream`.
 */
/* 65,536 norm tiles of ZERO_NORM_TILE elements */
#define ZERO_NOALLOC_MAX_ELEMS (65536LL * ZERO_NORM_TILE)
/* one double per tile + a 256-byte tail (chunk sums, overflow word) */
#define ZERO_NOALLOC_SCRATCH_BYTES (65536 * 8 + 256)
zero_status zero_reduce_partition_noalloc(int32_t n_ranks, zero_lp lp,
                                          const void *const *grad_slices,
                                          int64_t len, float loss_scale,
                                          float *grad_out, double *sumsq_out,
                                          int32_t *overflow_out, void *stream);

/* ----------------------------------------------------------------------
 * Accounting ("10.6 ZeRO 与 FSDP" Table 10-2; "第13篇 · ZeRO" §3.2, §3.4).
 * formula_bytes: per-GPU model-state bytes from the closed forms
 *   [0] DDP 16Ψ, [1] stage 1 4Ψ+12Ψ/N, [2] stage 2 2Ψ+14Ψ/N, [3] stage 3 16Ψ/N
 *   (exact rational values rounded once to double).
 * actual_bytes: the same for the padded layout (Ψ_p = Ψ rounded up to a
 *   multiple of N*align, P = Ψ_p/N): 16Ψ, 4Ψ_p+12P, 2Ψ_p+14P, 16P.
 * comm_elems: elements moved per step: DDP 2Ψ, stage 1 2Ψ, stage 2 2Ψ,
 *   stage 3 3Ψ.
 * Pure host arithmetic; align >= 1.  Any output array may be NULL.
 */
zero_status zero_memory_report(int64_t psi, int32_t n_ranks, int32_t align,
                               double formula_bytes[4], int64_t actual_bytes[4],
                               int64_t comm_elems[4]);

/* Frees the plan and its device scratch, after waiting for the plan's own
 * device work (the whole device once one of its calls was captured into a
 * graph).  NULL is allowed. */
void zero_plan_destroy(zero_plan *plan);

/* Message for the last failing call on this thread ("" if none). */
const char *zero_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_H */
