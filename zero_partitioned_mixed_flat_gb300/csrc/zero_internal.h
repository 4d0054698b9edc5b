// zero_internal.h -- shared between the host plan (plan.cpp) and the CUDA
// kernels (kernels.cu) of libzero.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace zk {

// Elements per norm tile.  Each tile's sum of squares is one fp64 partial,
// computed by one CTA in a fixed order, so the global norm is the same for
// every grid size and every bucket size (buckets are whole tiles).  Small
// enough that one stage-3 unit shard spans several hundred tiles (one CTA
// each), so a per-unit reduce fills the GPU.
constexpr int64_t kTile = 4096;
// Partials summed per first-level block of the norm (fixed, so the summation
// tree of the norm is a function of the partition only).
constexpr int64_t kPartialChunk = 4096;

// Default bound on the polls of a device pipeline wait (zero_plan_set_spin_limit).
constexpr int64_t kDefaultSpinLimit = int64_t(1) << 22;

// Per-plan device record of the step decision and the optimizer step state.
struct StepRecord {
    double norm;          // global gradient norm of the decided step
    double sumsq;         // the global sum of squares it is the root of
    float coef;           // clip coefficient (1 when not clipping)
    float loss_scale;     // S for the next step
    float bc1, bc2;       // 1 - beta1^t, 1 - beta2^t
    long long step;       // Adam step counter t
    int skip;             // 1: overflow, the update is skipped
    int good_steps;       // consecutive non-skipped steps since the last growth
    int error;            // set when a bounded device wait gives up
    unsigned arrivals;    // blocks of the decision kernel done (0 between launches)
    unsigned arrivals_x;  // the same for the statistics export
    int pad_;
};
static_assert(sizeof(StepRecord) == 64, "one 64-byte record");

int sm_count();

// message for zero_last_error() on the calling thread
void set_last_error(const char *msg);

// One run of whole norm tiles for the reduce kernel: elements [off, off + len)
// of one partition (off and len multiples of 8; the run starts a tile), whose
// first tile's partial sum goes to partials[pbase].  The partition's N slices
// are table entries src0 .. src0 + N - 1 (pointers to the partition start),
// its output starts at g, its overflow word is *overflow.
struct ReduceSegment {
    int64_t off, len, pbase;
    float *g;
    double *partials;
    unsigned *overflow;
    int32_t src0;
};
constexpr int kMaxReduceSegments = 64;
// Slice pointers one reduce launch can carry: enough for
// kReduceSrcTable / N partitions when N <= 64, one partition beyond.
constexpr int kReduceSrcTable = 512;
inline int reduce_src_table(int n) { return n > 64 ? 1024 : kReduceSrcTable; }

// Reduce the segments (at most kMaxReduceSegments) in one launch; slices is the
// table of slice pointers the segments index (n_src entries, at most
// reduce_src_table(n)); every slice holds the same lp type.
cudaError_t launch_reduce(const void *const *slices, int n_src, int n, int lp, int acc_lp,
                          const ReduceSegment *segs, int n_segs, float inv, cudaStream_t stream);

// Bias corrections computed on the host for the step counters the decision
// is likely to reach: entry i is for t = bc_t0 - i (1 - beta^t in fp64, then
// rounded to float).  A counter outside the table is computed on the device.
constexpr int kBcTable = 8;

// What a launch of the norm kernel does with the step's partials.
enum NormMode {
    kDecideLocal = 0,   // the step's partitions (+ remote terms) -> the decision
    kExportStats = 1,   // the step's partitions -> per-partition stats vector
    kDecideGlobal = 2,  // an all-reduced stats vector -> the decision
};

struct NormLaunch {
    int mode;
    const double *partials;     // n_slots x tiles_per_slot (local, export)
    double *level2;             // active x chunks doubles of scratch (local, export)
    unsigned *arrivals;         // 0 between launches (local, export)
    const unsigned *overflow;   // per slot (local, export)
    double *stats_out;          // export: 2 * n_slots doubles
    const double *stats_in;     // global: 2 * n_slots doubles
    int64_t tiles_per_slot;
    const uint64_t *active_mask;
    int n_slots;                // N (the stats vector has 2N entries)
    double remote_sumsq;        // local mode only
    int remote_overflow;        // local mode only
    float clip, loss_scale, beta1, beta2;
    int growth_interval;
    int64_t bc_t0;
    const float *bc1_tab, *bc2_tab;
    StepRecord *rec;
};

cudaError_t launch_norm(const NormLaunch &a, cudaStream_t stream);

// One run of the Adam kernel: len elements (a multiple of 8) at these
// pointers (param may be NULL: no cast).
struct AdamSegment {
    const float *g;
    float *master, *m, *v;
    void *param;
    int64_t len;
};
constexpr int kMaxAdamSegments = 64;

// Adam + cast over the segments (at most kMaxAdamSegments) in one launch.
cudaError_t launch_adam(const AdamSegment *segs, int n_segs, int lp,
                        const StepRecord *rec, int *error, int64_t spin_limit,
                        float lr, float beta1, float beta2, float omb1, float omb2,
                        float eps, float wd, float decay, int adamw,
                        cudaStream_t stream);

// out + j * dst_stride_bytes + [0, shard_bytes) <- shards[j] + src_offset_bytes + [0, shard_bytes)
cudaError_t launch_gather(const void *const *shards, int n, int64_t src_offset_bytes,
                          int64_t shard_bytes, void *out, int64_t dst_stride_bytes,
                          int64_t spin_limit, int *error, cudaStream_t stream);

// quantized all-gather (block = 128 elements): shard -> 1-byte codes (int8,
// or E4M3 when fp8) + float scales; codes/scales of N ranks at a unit's
// offset -> lp layer buffer
cudaError_t launch_quantize(const void *shard, int lp, int fp8, int64_t len, int8_t *codes,
                            float *scales, cudaStream_t stream);

cudaError_t launch_dequant_gather(const int8_t *const *codes, const float *const *scales,
                                  int n, int lp, int fp8, int64_t offset, int64_t shard_len,
                                  void *out, cudaStream_t stream);

}  // namespace zk
