// kernels.cu -- the device side of libzero (sm_103a).
//
// K1 reduce_unscale_stats  N-way reduce of lp gradient slices into one fp32
//                          partition, unscale, overflow flag, per-tile sum of
//                          squares ("10.6 ZeRO 与 FSDP" §10.6.1 Reduce-Scatter,
//                          §10.6.2 Step 2).
// K2 norm_decide           global norm, clip coefficient, skip and loss-scale
//                          decision, step counter ("年糕切片" §4.2-§4.3).
// K3 adam_fused_cast       Adam/AdamW on fp32 master/m/v + lp cast into the
//                          all-gather destination (§10.6.2 Steps 3-4); a
//                          warp-specialised TMA bulk-copy pipeline.
// K4 gather_layer_tma      stage-3 per-layer all-gather of N shards
//                          (§10.6.4 step 1) and the bucketed stage-1/2
//                          parameter all-gather (§10.6.2 Step 4): TMA bulk
//                          copies through shared memory with bounded
//                          mbarrier waits.
//
// Everything here is bandwidth-bound streaming: no tensor cores.  All float
// arithmetic of the step uses explicit round-to-nearest intrinsics so that no
// multiply-add is fused and the op order is the one the ABI documents.  Every
// kernel starts with pdl_enter() (launch.h): it waits for the previous grid of
// the stream before touching global memory.
#include "launch.h"
#include "norm_tree.cuh"
#include "zero_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <mutex>

namespace zk {
namespace {

constexpr int kReduceThreads = 128;
constexpr int kVec = 8;  // lp elements per 16-byte vector
constexpr int kBatch = 16;  // loads (slices x vectors) a thread issues before it adds
// vectors of 8 elements a thread takes from each slice per round: 4 makes a
// warp's load from one slice one contiguous 2 KB run and covers a 4096-element
// tile in one round (faster than 1 or 2 at N = 8, 16 and 64 on GB300)
constexpr int kReduceVpt = 4;
// Few slices give a thread few loads to keep in flight (N x 4), so up to
// kSmallN slices a tile goes to 64 threads taking 8 vectors each instead
// (13B-sized partitions on GB300: N = 2 from 73 % to 86 % of the copy peak,
// N = 3 from 85 % to 97 %; no gain from N = 4 on).
constexpr int kSmallN = 3;
constexpr int kSmallThreads = 64;
constexpr int kSmallVpt = 8;
constexpr int kMaxSegments = kMaxReduceSegments;  // tile runs per reduce launch
constexpr int kGatherStages = 3;
constexpr unsigned kGatherChunk = 32768;  // bytes per bulk copy
constexpr long long kDrainPolls = 1ll << 21;
static_assert(kTile % (kReduceVpt * kReduceThreads * kVec) == 0, "tile must be whole rounds");
static_assert(kTile % (kSmallVpt * kSmallThreads * kVec) == 0, "tile must be whole rounds");
static_assert(kBatch % kSmallVpt == 0, "a batch holds whole slices");
static_assert(kBatch % kReduceVpt == 0, "a batch holds whole slices");

// ---------------------------------------------------------------- memory ops

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream_f4(float4 *p, float4 v) { __stcs(p, v); }

// 8 lp values -> 8 floats (exact conversions)
template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &q, float f[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if constexpr (BF16) {
            f[2 * k] = __uint_as_float(w[k] << 16);
            f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        } else {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[k]);
            float2 t = __half22float2(h);
            f[2 * k] = t.x;
            f[2 * k + 1] = t.y;
        }
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (BF16) {
        uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
        uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
        return lo | (hi << 16);
    } else {
        uint32_t lo = __half_as_ushort(__float2half_rn(a));
        uint32_t hi = __half_as_ushort(__float2half_rn(b));
        return lo | (hi << 16);
    }
}

// ------------------------------------------------------------------ K1 reduce

// hi + lo += x, error-free (Knuth's TwoSum: the rounding error of hi + x is
// recovered exactly with round-to-nearest adds and kept in lo)
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float x) {
    const float s = __fadd_rn(hi, x);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(x, bp));
    hi = s;
    lo = __fadd_rn(lo, err);
}

template <int MAXN>
struct ReduceParams {
    static constexpr int kSrc = MAXN > kReduceSrcTable ? MAXN : kReduceSrcTable;
    const uint4 *src[kSrc];              // slice pointers (partition starts)
    long long seg_off[kMaxSegments];     // first element of each segment (multiple of 8)
    long long seg_end[kMaxSegments];     // one past its last element (multiple of 8)
    long long seg_pbase[kMaxSegments];   // partial index of its first tile
    float4 *seg_g[kMaxSegments];         // its partition's output (partition start)
    double *seg_partials[kMaxSegments];  // its partition's tile partials
    unsigned *seg_overflow[kMaxSegments];
    int seg_src0[kMaxSegments];          // its partition's slice j is src[seg_src0 + j]
    int seg_cta0[kMaxSegments + 1];      // first CTA of each segment; [n_seg] = grid
    float inv;                           // float(1 / (S * N))
    int n;
    int n_seg;
};

// round a float to the lp type and back (nearest, ties to even)
template <bool BF16>
__device__ __forceinline__ void round_lp_pair(float &a, float &b) {
    if constexpr (BF16) {
        const float2 t = __bfloat1622float2(__floats2bfloat162_rn(a, b));
        a = t.x;
        b = t.y;
    } else {
        const float2 t = __half22float2(__floats2half2_rn(a, b));
        a = t.x;
        b = t.y;
    }
}

// ACC_LP: every partial sum is rounded to the lp type before the next rank's
// value is added (reduce in the low-precision dtype).  The float add of two lp
// values followed by that rounding equals the correctly rounded lp sum (24
// float bits >= 2p + 2, so the double rounding is innocuous).
// VPT: vectors (of 8 elements) per thread per round, kBatch / VPT slices per
// batch of loads, so a thread keeps kBatch loads in flight.  Each warp's 1 KB
// of float output per vector goes through shared memory so that it leaves as
// two contiguous 512-byte stores instead of 32 lanes writing 32-byte strided
// halves.
template <int MAXN, bool BF16, bool ACC_LP, int VPT, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS == 64 ? 6 : 4)
reduce_unscale_stats(const __grid_constant__ ReduceParams<MAXN> p) {
    pdl_enter();
    constexpr int BATCH = kBatch / VPT;
    constexpr int kTileIters = int(kTile / (THREADS * kVec));
    __shared__ double warp_sq[THREADS / 32];
    __shared__ float4 stage[THREADS / 32][64];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    bool bad = false;
    // this CTA's tile: tile t of segment seg
    int seg = 0;
    while (seg + 1 < p.n_seg && (int)blockIdx.x >= p.seg_cta0[seg + 1]) ++seg;
    const long long t = (long long)blockIdx.x - p.seg_cta0[seg];
    const long long e0 = p.seg_off[seg] + t * kTile;
    const long long e1 = e0 + kTile < p.seg_end[seg] ? e0 + kTile : p.seg_end[seg];
    const long long v_end = e1 / kVec;
    const int s0 = p.seg_src0[seg];
    float4 *const gout = p.seg_g[seg];
    {
        // per-thread sum of squares as an unevaluated float pair (hi + lo):
        // compensated, so the tile sum is accurate to ~1e-13 relative and the
        // clip coefficient derived from it matches a sequential fp64 sum
        float sq_hi = 0.0f, sq_lo = 0.0f;
        const long long v0 = e0 / kVec;
#pragma unroll 1
        for (int it = 0; it < kTileIters / VPT; ++it) {
            const long long vb = v0 + (long long)it * VPT * THREADS + warp * 32;
            if (vb >= v_end) break;  // the whole warp is past the end
            long long vi[VPT];
            bool ok[VPT];
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                vi[v] = vb + (long long)v * THREADS + lane;
                ok[v] = vi[v] < v_end;
            }
            float s[VPT][8];
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const uint4 z = ok[v] ? ld_stream(p.src[s0] + vi[v]) : make_uint4(0u, 0u, 0u, 0u);
                unpack8<BF16>(z, s[v]);
            }
            for (int j0 = 1; j0 < p.n; j0 += BATCH) {
                uint4 q[VPT][BATCH];
#pragma unroll
                for (int v = 0; v < VPT; ++v)
#pragma unroll
                    for (int b = 0; b < BATCH; ++b)
                        if (j0 + b < p.n && ok[v]) q[v][b] = ld_stream(p.src[s0 + j0 + b] + vi[v]);
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
#pragma unroll
                    for (int b = 0; b < BATCH; ++b) {
                        if (j0 + b < p.n && ok[v]) {
                            float x[8];
                            unpack8<BF16>(q[v][b], x);
#pragma unroll
                            for (int k = 0; k < 8; ++k) s[v][k] = __fadd_rn(s[v][k], x[k]);
                            if constexpr (ACC_LP) {
#pragma unroll
                                for (int k = 0; k < 8; k += 2) round_lp_pair<BF16>(s[v][k], s[v][k + 1]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                float o[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    bad |= !isfinite(s[v][k]);  // zero for lanes past the end
                    o[k] = __fmul_rn(s[v][k], p.inv);
                    two_sum_acc(sq_hi, sq_lo, __fmul_rn(o[k], o[k]));
                }
                // lane l's vector -> stage[2l, 2l+1]; then lane l stores float4 l
                // and 32 + l of the warp's contiguous 1 KB run
                stage[warp][2 * lane] = make_float4(o[0], o[1], o[2], o[3]);
                stage[warp][2 * lane + 1] = make_float4(o[4], o[5], o[6], o[7]);
                __syncwarp();
                const float4 lo = stage[warp][lane];
                const float4 hi = stage[warp][32 + lane];
                __syncwarp();
                const long long wv = vb + (long long)v * THREADS;  // the warp's first vector
                if (wv + (lane >> 1) < v_end) st_stream_f4(gout + 2 * wv + lane, lo);
                if (wv + 16 + (lane >> 1) < v_end) st_stream_f4(gout + 2 * wv + 32 + lane, hi);
            }
        }
        // fixed-shape fp64 tree: lanes (xor butterfly), then warps in order
        double sq = __dadd_rn((double)sq_hi, (double)sq_lo);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            sq = __dadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, off));
        if (lane == 0) warp_sq[warp] = sq;
        __syncthreads();
        if (threadIdx.x == 0) {
            double tsum = 0.0;
#pragma unroll
            for (int w = 0; w < THREADS / 32; ++w) tsum = __dadd_rn(tsum, warp_sq[w]);
            p.seg_partials[seg][p.seg_pbase[seg] + t] = tsum;
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(p.seg_overflow[seg], 1u);
}

// ------------------------------------------------------------------ K2 decide

struct DecideParams {
    const double *partials;
    double *level2;
    const unsigned *overflow;  // per slot
    unsigned *arrivals;        // 0 at launch; the last block resets it
    double *stats_out;         // export: 2 * n_slots
    const double *stats_in;    // global: 2 * n_slots
    long long tiles_per_slot;
    int chunks_per_slot;
    int n_active;              // reduced slots (local, export)
    int n_slots;
    int mode;                  // NormMode
    double remote_sumsq;
    int remote_overflow;
    float clip, loss_scale, beta1, beta2;
    int growth_interval;
    StepRecord *rec;
    long long bc_t0;             // bc*_tab[i] is for step counter bc_t0 - i
    float bc1_tab[kBcTable], bc2_tab[kBcTable];
    short slots[kNormMaxSlots];  // the step's reduced partition slots, ascending
};

constexpr int kDecideThreads = kNormThreads;

// The norm in fixed-order fp64 levels (norm_tree.cuh) and, unless exporting,
// the step decision, in one launch.  Local and export modes: block `item`
// sums one chunk of one reduced partition's tile partials (level 1); the last
// block to arrive (counted after a fence) forms each partition's sum (level 2)
// in a vector indexed by partition.  Global mode: one block takes that vector
// from the caller (every rank's vectors summed element-wise).  Then export
// writes the vector and the partitions' overflow flags; the decision sums the
// vector (level 3), adds the remote term (local mode), and decides.  The order
// of every addition depends only on the partition sizes, never on which block
// finishes first.
// fp64 adds are slow on this part (a 64-cycle latency, under 2 per cycle per
// SM), so every fixed-order sum is a tree, never a long chain.
__global__ void __launch_bounds__(kDecideThreads)
norm_decide(const __grid_constant__ DecideParams p) {
    pdl_enter();
    __shared__ double wsum[kDecideThreads / 32];
    __shared__ double vec[kNormMaxSlots];
    __shared__ unsigned char flag[kNormMaxSlots];
    __shared__ float bias_corr[2];
    __shared__ int any_overflow;
    __shared__ bool last;
    StepRecord *rec = p.rec;
    if (p.mode != kDecideGlobal) {
        const int item = blockIdx.x;
        const int slot = p.slots[item / p.chunks_per_slot];
        const long long t0 = (long long)(item % p.chunks_per_slot) * kPartialChunk;
        const long long t1 = t0 + kPartialChunk < p.tiles_per_slot ? t0 + kPartialChunk : p.tiles_per_slot;
        const double chunk = chunk_sum(p.partials + (long long)slot * p.tiles_per_slot, t0, t1, wsum);
        if (threadIdx.x == 0) {
            p.level2[item] = chunk;
            __threadfence();
            last = atomicAdd(p.arrivals, 1u) == gridDim.x - 1;
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
    }
    // the last (or only) block: per-partition sums and flags in partition order
    for (int i = threadIdx.x; i < p.n_slots; i += kDecideThreads) {
        vec[i] = 0.0;
        flag[i] = 0;
    }
    if (threadIdx.x == 0) any_overflow = 0;
    __syncthreads();
    if (p.mode == kDecideGlobal) {
        for (int i = threadIdx.x; i < p.n_slots; i += kDecideThreads) {
            vec[i] = p.stats_in[i];
            if (p.stats_in[p.n_slots + i] != 0.0) {
                flag[i] = 1;
                any_overflow = 1;  // every writer stores the same value
            }
        }
    } else {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int a = warp; a < p.n_active; a += kDecideThreads / 32) {
            const double *c = p.level2 + (long long)a * p.chunks_per_slot;
            const double sum = slot_sum_warp([c](int k) { return __ldcg(c + k); }, p.chunks_per_slot);
            if (lane == 0) {
                const int slot = p.slots[a];
                vec[slot] = sum;
                if (__ldcg(p.overflow + slot) != 0u) {
                    flag[slot] = 1;
                    any_overflow = 1;
                }
            }
        }
    }
    if (p.mode != kExportStats && (threadIdx.x == 32 || threadIdx.x == 64)) {
        // bias corrections for t + 1 (the step counter if the step is not
        // skipped): from the host's table when it holds that counter, else
        // computed here in fp64
        const int b = threadIdx.x == 64;
        const long long tn = rec->step + 1;
        const long long i = p.bc_t0 - tn;
        if (i >= 0 && i < kBcTable) {
            bias_corr[b] = b ? p.bc2_tab[i] : p.bc1_tab[i];
        } else {
            const double beta = b ? (double)p.beta2 : (double)p.beta1;
            bias_corr[b] = __double2float_rn(__dsub_rn(1.0, pow(beta, (double)tn)));
        }
    }
    __syncthreads();
    if (p.mode == kExportStats) {
        for (int i = threadIdx.x; i < p.n_slots; i += kDecideThreads) {
            p.stats_out[i] = vec[i];
            p.stats_out[p.n_slots + i] = flag[i] ? 1.0 : 0.0;
        }
        if (threadIdx.x == 0) *p.arrivals = 0u;
        return;
    }
    double sumsq;
    if (p.mode == kDecideLocal && p.n_active == 1)
        sumsq = vec[p.slots[0]];  // the other entries are zeros: adding them is exact
    else
        sumsq = vector_sum_block(vec, p.n_slots, wsum);
    if (threadIdx.x != 0) return;
    if (p.mode == kDecideLocal) {
        *p.arrivals = 0u;
        sumsq = __dadd_rn(sumsq, p.remote_sumsq);
    }
    const double norm = sqrt(sumsq);
    const int skip = any_overflow != 0 || (p.mode == kDecideLocal && p.remote_overflow != 0);
    float coef = 1.0f;
    if (p.clip > 0.0f) {
        const double c = __ddiv_rn((double)p.clip, __dadd_rn(norm, 1e-6));
        if (c < 1.0) coef = __double2float_rn(c);
    }
    long long t = rec->step;
    int good = rec->good_steps;
    float s = p.loss_scale;
    if (skip) {
        s = p.growth_interval > 0 ? fmaxf(__fmul_rn(p.loss_scale, 0.5f), 1.0f) : p.loss_scale;
        good = 0;
    } else {
        good += 1;
        if (p.growth_interval > 0 && good >= p.growth_interval) {
            s = __fmul_rn(p.loss_scale, 2.0f);
            good = 0;
        }
        t += 1;
    }
    rec->norm = norm;
    rec->sumsq = sumsq;
    rec->coef = coef;
    rec->skip = skip;
    rec->loss_scale = s;
    rec->good_steps = good;
    rec->step = t;
    if (!skip) {  // a skipped step keeps the previous corrections (Adam does not run)
        rec->bc1 = bias_corr[0];
        rec->bc2 = bias_corr[1];
    }
}

// ------------------------------------------------- TMA / mbarrier primitives

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait: at most `polls` try_wait polls (0: give up at once)
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long polls) {
    for (long long i = 0; i < polls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// make this thread's generic-proxy shared-memory writes visible to later
// bulk (async-proxy) reads of the same bytes
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// named barrier over `count` threads that also ORs a predicate across them
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("barrier.cta.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// -------------------------------------------------------------------- K3 adam

struct AdamScalars {
    float coef, bc1, bc2, lr, beta1, beta2, omb1, omb2, eps, wd, decay;
    int adamw;
};

__device__ __forceinline__ void adam1(const AdamScalars &c, float g, float &w, float &m,
                                      float &v) {
    float gi = __fmul_rn(g, c.coef);
    if (!c.adamw) gi = __fadd_rn(gi, __fmul_rn(c.wd, w));
    m = __fadd_rn(__fmul_rn(c.beta1, m), __fmul_rn(c.omb1, gi));
    v = __fadd_rn(__fmul_rn(c.beta2, v), __fmul_rn(c.omb2, __fmul_rn(gi, gi)));
    const float mhat = __fdiv_rn(m, c.bc1);
    const float vhat = __fdiv_rn(v, c.bc2);
    const float denom = __fadd_rn(__fsqrt_rn(vhat), c.eps);
    const float upd = __fdiv_rn(__fmul_rn(c.lr, mhat), denom);
    if (c.adamw) w = __fmul_rn(w, c.decay);
    w = __fsub_rn(w, upd);
}

// K3: Adam/AdamW + cast with the memory traffic on the TMA engine.  Warp 0
// (one thread) streams 1024-element tiles of g, master, m, v into 4
// shared-memory stages with cp.async.bulk (completion on an mbarrier per
// stage); 8 consumer warps update 4 elements per thread, release the input
// stage (empty mbarrier), write master/m/v/param into one of 2 output stages,
// and one consumer thread stores them back with bulk copies.  Two such
// pipelines (CTAs, 92 KB of shared memory each) run per SM.
// Every pipeline wait polls at most `spin_limit` times (the plan's setting); a
// consumer wait that gives up makes all consumers leave together (the barrier
// vote, before any store of that tile), a producer wait that gives up stops the
// loads, and either sets the error word.  Whatever happens, the producer then
// waits (with its own fixed bound) for every load it issued that no consumer
// is known to have received, so no bulk copy into this CTA's shared memory is
// in flight when the CTA exits; the consumers' store thread waits for its
// stores.
constexpr int kAdamTile = 1024;
constexpr int kAdamInStages = 4;
constexpr int kAdamOutStages = 2;
constexpr int kAdamConsumerWarps = 8;
constexpr int kAdamConsumers = kAdamConsumerWarps * 32;
constexpr int kAdamTmaThreads = kAdamConsumers + 32;
constexpr size_t kAdamInStageBytes = 4 * kAdamTile * sizeof(float);
constexpr size_t kAdamOutStageBytes = 3 * kAdamTile * sizeof(float) + kAdamTile * 2;
constexpr size_t kAdamTmaSmem = kAdamInStages * kAdamInStageBytes + kAdamOutStages * kAdamOutStageBytes;
constexpr int kAdamCtasPerSm = 2;
static_assert(kAdamTile == kAdamConsumers * 4, "4 elements per consumer thread");

// One segment of the tile space: len elements (a multiple of 8) from these
// pointers; its tiles are tile0 .. tile0 + ceil(len / kAdamTile) - 1.
struct AdamSegDev {
    const float *g;
    float *master, *m, *v;
    uint16_t *param;  // NULL: no cast
    long long len;
    long long tile0;
};

struct AdamTmaParams {
    AdamSegDev seg[kMaxAdamSegments];
    long long n_tiles;  // over every segment
    int n_seg;
    const StepRecord *rec;
    int *error;
    long long spin_limit;
    float lr, beta1, beta2, omb1, omb2, eps, wd, decay;
    int adamw;
};

// A thread's current segment, kept in registers: a CTA's tiles increase, so
// the cursor only moves forward, and the segment table (kernel parameters,
// read with a computed index) is touched only when a tile starts a new
// segment -- never with a single segment, whose fields are read once at
// constant offsets.
struct AdamCursor {
    AdamSegDev sg;
    long long next_tile0;  // first tile of the next segment
    int cur;

    __device__ __forceinline__ explicit AdamCursor(const AdamTmaParams &p)
        : sg(p.seg[0]), next_tile0(p.n_seg > 1 ? p.seg[1].tile0 : LLONG_MAX), cur(0) {}

    __device__ __forceinline__ void seek(const AdamTmaParams &p, long long t) {
        while (t >= next_tile0) {
            ++cur;
            sg = p.seg[cur];
            next_tile0 = cur + 1 < p.n_seg ? p.seg[cur + 1].tile0 : LLONG_MAX;
        }
    }
};

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// DEFAULT_SPIN: the wait bound is the compile-time default (the plan's
// setting unless changed), which measured 2.7 % faster at 13B than the same
// loop bounded by a run-time value; otherwise p.spin_limit.
template <bool BF16, bool DEFAULT_SPIN>
__global__ void __launch_bounds__(kAdamTmaThreads, kAdamCtasPerSm)
adam_fused_cast(const __grid_constant__ AdamTmaParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kAdamInStages];
    __shared__ __align__(8) uint64_t empty[kAdamInStages];
    pdl_enter();
    const StepRecord *rec = p.rec;
    if (rec->skip) return;
    const long long spin = DEFAULT_SPIN ? (long long)kDefaultSpinLimit : p.spin_limit;
    const long long n_tiles = p.n_tiles;
    if ((long long)blockIdx.x >= n_tiles) return;
    const long long count = (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;
    unsigned char *in_base = smem;
    unsigned char *out_base = smem + kAdamInStages * kAdamInStageBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kAdamInStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kAdamConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {  // ---------------------------------------------- producer
        if (lane != 0) return;
        long long k = 0;
        bool ok = true;
        AdamCursor at(p);
        for (; k < count; ++k) {
            const int s = (int)(k % kAdamInStages);
            if (k >= kAdamInStages &&
                !mbar_wait_bounded(&empty[s], (uint32_t)(((k / kAdamInStages) - 1) & 1), spin)) {
                ok = false;
                break;
            }
            const long long t = blockIdx.x + k * gridDim.x;
            at.seek(p, t);
            const AdamSegDev &sg = at.sg;
            const long long e0 = (t - sg.tile0) * (long long)kAdamTile;
            const long long n = sg.len - e0 < kAdamTile ? sg.len - e0 : kAdamTile;
            const uint32_t bytes = (uint32_t)(n * sizeof(float));
            unsigned char *dst = in_base + (size_t)s * kAdamInStageBytes;
            mbar_expect_tx(&full[s], 4 * bytes);
            bulk_load(dst, sg.g + e0, bytes, &full[s]);
            bulk_load(dst + 1 * kAdamTile * sizeof(float), sg.master + e0, bytes, &full[s]);
            bulk_load(dst + 2 * kAdamTile * sizeof(float), sg.m + e0, bytes, &full[s]);
            bulk_load(dst + 3 * kAdamTile * sizeof(float), sg.v + e0, bytes, &full[s]);
        }
        if (!ok) atomicExch(p.error, 1);
        // Drain.  k tiles were issued.  Every tile kk < k - kAdamInStages has
        // landed: issuing tile kk + kAdamInStages into the same stage needed
        // the consumers to release tile kk first.  Tile kk >= k - kAdamInStages
        // is the last load of its stage, so waiting for its phase is
        // unambiguous.  In a normal run the consumers wait for these same
        // loads; after a consumer timeout nobody else would.
        const long long first = k > kAdamInStages ? k - kAdamInStages : 0;
        for (long long kk = first; kk < k; ++kk)
            mbar_wait_bounded(&full[kk % kAdamInStages], (uint32_t)((kk / kAdamInStages) & 1), kDrainPolls);
        return;
    }

    // ------------------------------------------------------------- consumers
    const int ct = threadIdx.x - 32;  // 0 .. kAdamConsumers-1
    AdamScalars c;
    c.coef = rec->coef;
    c.bc1 = rec->bc1;
    c.bc2 = rec->bc2;
    c.lr = p.lr;
    c.beta1 = p.beta1;
    c.beta2 = p.beta2;
    c.omb1 = p.omb1;
    c.omb2 = p.omb2;
    c.eps = p.eps;
    c.wd = p.wd;
    c.decay = p.decay;
    c.adamw = p.adamw;
    bool ok = true;
    AdamCursor at(p);
    for (long long k = 0; k < count; ++k) {
        const int s = (int)(k % kAdamInStages);
        const int so = (int)(k % kAdamOutStages);
        const long long t = blockIdx.x + k * gridDim.x;
        at.seek(p, t);
        const AdamSegDev &sg = at.sg;
        const long long e0 = (t - sg.tile0) * (long long)kAdamTile;
        const int n = (int)(sg.len - e0 < kAdamTile ? sg.len - e0 : kAdamTile);
        const bool got = mbar_wait_bounded(&full[s], (uint32_t)((k / kAdamInStages) & 1), spin);
        const bool mine = got && ct * 4 < n;
        float4 g4 = make_float4(0.f, 0.f, 0.f, 0.f), w4 = g4, m4 = g4, v4 = g4;
        if (mine) {
            const float4 *in = reinterpret_cast<const float4 *>(in_base + (size_t)s * kAdamInStageBytes);
            g4 = in[ct];
            w4 = in[kAdamTile / 4 + ct];
            m4 = in[2 * (kAdamTile / 4) + ct];
            v4 = in[3 * (kAdamTile / 4) + ct];
        }
        __syncwarp();
        if (got && lane == 0) mbar_arrive(&empty[s]);
        if (mine) {
            adam1(c, g4.x, w4.x, m4.x, v4.x);
            adam1(c, g4.y, w4.y, m4.y, v4.y);
            adam1(c, g4.z, w4.z, m4.z, v4.z);
            adam1(c, g4.w, w4.w, m4.w, v4.w);
        }
        // the store issued kAdamOutStages tiles ago must have read stage `so`
        if (ct == 0) bulk_wait_read<kAdamOutStages - 1>();
        if (named_barrier_or(1, kAdamConsumers, !got)) {
            ok = false;
            break;
        }
        unsigned char *ob = out_base + (size_t)so * kAdamOutStageBytes;
        if (mine) {
            float4 *o = reinterpret_cast<float4 *>(ob);
            o[ct] = w4;
            o[kAdamTile / 4 + ct] = m4;
            o[2 * (kAdamTile / 4) + ct] = v4;
            uint2 q;
            q.x = pack2<BF16>(w4.x, w4.y);
            q.y = pack2<BF16>(w4.z, w4.w);
            reinterpret_cast<uint2 *>(ob + 3 * kAdamTile * sizeof(float))[ct] = q;
        }
        fence_proxy_async_smem();
        named_barrier(1, kAdamConsumers);
        if (ct == 0) {
            const uint32_t bytes = (uint32_t)(n * sizeof(float));
            bulk_store(sg.master + e0, ob, bytes);
            bulk_store(sg.m + e0, ob + kAdamTile * sizeof(float), bytes);
            bulk_store(sg.v + e0, ob + 2 * kAdamTile * sizeof(float), bytes);
            if (sg.param) bulk_store(sg.param + e0, ob + 3 * kAdamTile * sizeof(float), (uint32_t)(n * 2));
            bulk_commit();
        }
    }
    if (ct == 0) {
        bulk_wait_all();
        if (!ok) atomicExch(p.error, 1);
    }
}

// ------------------------------------------------------------------ K4 gather

template <int MAXN>
struct GatherParams {
    const char *src[MAXN];  // shard j at this unit's offset
    char *dst;              // rank j's bytes go to dst + j * dst_stride
    long long dst_stride;
    long long shard_bytes;
    long long chunks_per_shard;
    long long n_chunks;
    long long spin_limit;
    int *error;
    int n;
};

template <int MAXN>
__global__ void __launch_bounds__(32)
gather_layer_tma(const __grid_constant__ GatherParams<MAXN> p) {
    extern __shared__ __align__(128) unsigned char stage_buf[];
    __shared__ __align__(8) uint64_t bar[kGatherStages];
    pdl_enter();
    if (threadIdx.x != 0) return;  // one thread drives the copy engine
    if (blockIdx.x >= p.n_chunks) return;
    const long long spin = p.spin_limit;  // in a register (see adam_fused_cast)
    const long long count = (p.n_chunks - blockIdx.x + gridDim.x - 1) / gridDim.x;

    for (int s = 0; s < kGatherStages; ++s) mbar_init(&bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

    auto chunk_src = [&](long long k, const char *&src, char *&dst, uint32_t &bytes) {
        const long long c = blockIdx.x + k * gridDim.x;
        const long long j = c / p.chunks_per_shard;
        const long long off = (c - j * p.chunks_per_shard) * (long long)kGatherChunk;
        const long long rem = p.shard_bytes - off;
        bytes = rem < (long long)kGatherChunk ? (uint32_t)rem : kGatherChunk;
        src = p.src[j] + off;
        dst = p.dst + j * p.dst_stride + off;
    };
    auto issue = [&](long long k) {
        const char *src;
        char *dst;
        uint32_t bytes;
        chunk_src(k, src, dst, bytes);
        const int s = (int)(k % kGatherStages);
        mbar_expect_tx(&bar[s], bytes);
        bulk_load(stage_buf + (size_t)s * kGatherChunk, src, bytes, &bar[s]);
    };

    long long issued = 0;
    for (; issued < count && issued < kGatherStages; ++issued) issue(issued);

    long long k = 0;
    bool ok = true;
    for (; k < count; ++k) {
        const int s = (int)(k % kGatherStages);
        const uint32_t parity = (uint32_t)((k / kGatherStages) & 1);
        if (!mbar_wait_bounded(&bar[s], parity, spin)) {
            ok = false;
            break;
        }
        const char *src;
        char *dst;
        uint32_t bytes;
        chunk_src(k, src, dst, bytes);
        bulk_store(dst, stage_buf + (size_t)s * kGatherChunk, bytes);
        bulk_commit();
        // refill the stage of chunk k-1, whose store may still be reading it:
        // allow only the newest store group (chunk k) to be pending.
        if (k >= 1 && issued < count) {
            bulk_wait_read1();
            issue(issued);
            ++issued;
        }
    }
    if (!ok) {
        atomicExch(p.error, 1);
        // drain: every load issued after the failed wait must land before the
        // CTA's shared memory is released
        for (long long kk = k; kk < issued; ++kk) {
            const int s = (int)(kk % kGatherStages);
            mbar_wait_bounded(&bar[s], (uint32_t)((kk / kGatherStages) & 1), kDrainPolls);
        }
    }
    bulk_wait_all();
}

// -------------------------------------------------------------- host helpers

struct DevInfo {
    int sms = 0;
};

DevInfo g_dev[64];
std::mutex g_dev_mu;

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem) != cudaSuccess)
        blocks = 1;
    return blocks < 1 ? 1 : blocks;
}

template <int MAXN, bool BF16, bool ACC_LP, int VPT, int THREADS>
cudaError_t reduce_impl(const void *const *slices, int n_src, int n, const ReduceSegment *segs, int n_segs,
                        float inv, cudaStream_t stream) {
    using Params = ReduceParams<MAXN>;
    if (n_segs < 1 || n_segs > kMaxSegments || n_src < n || n_src > Params::kSrc) return cudaErrorInvalidValue;
    Params p;
    for (int j = 0; j < n_src; ++j) p.src[j] = static_cast<const uint4 *>(slices[j]);
    for (int j = n_src; j < Params::kSrc; ++j) p.src[j] = nullptr;
    long long ctas = 0;
    for (int i = 0; i < n_segs; ++i) {
        if (segs[i].src0 < 0 || segs[i].src0 + n > n_src) return cudaErrorInvalidValue;
        p.seg_off[i] = segs[i].off;
        p.seg_end[i] = segs[i].off + segs[i].len;
        p.seg_pbase[i] = segs[i].pbase;
        p.seg_g[i] = reinterpret_cast<float4 *>(segs[i].g);
        p.seg_partials[i] = segs[i].partials;
        p.seg_overflow[i] = segs[i].overflow;
        p.seg_src0[i] = segs[i].src0;
        p.seg_cta0[i] = (int)ctas;
        ctas += (segs[i].len + kTile - 1) / kTile;  // one tile per CTA
    }
    for (int i = n_segs; i < kMaxSegments; ++i) {
        p.seg_off[i] = p.seg_end[i] = p.seg_pbase[i] = 0;
        p.seg_g[i] = nullptr;
        p.seg_partials[i] = nullptr;
        p.seg_overflow[i] = nullptr;
        p.seg_src0[i] = 0;
    }
    p.seg_cta0[n_segs] = (int)ctas;
    p.inv = inv;
    p.n = n;
    p.n_seg = n_segs;
    if (ctas < 1) return cudaSuccess;
    if (ctas > 0x7fffffffll) return cudaErrorInvalidValue;
    return launch_pdl(reduce_unscale_stats<MAXN, BF16, ACC_LP, VPT, THREADS>, dim3((unsigned)ctas),
                      dim3(THREADS), 0, stream, p);
}

template <bool BF16, bool DEFAULT_SPIN>
cudaError_t adam_tma_impl(const AdamTmaParams &p, cudaStream_t stream) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        adam_fused_cast<BF16, DEFAULT_SPIN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAdamTmaSmem);
    if (attr != cudaSuccess) return attr;
    const long long tiles = p.n_tiles;
    static const int occ = occupancy(adam_fused_cast<BF16, DEFAULT_SPIN>, kAdamTmaThreads, kAdamTmaSmem);
    long long grid = (long long)sm_count() * occ;
    if (grid > tiles) grid = tiles;
    if (grid < 1) return cudaSuccess;
    return launch_pdl(adam_fused_cast<BF16, DEFAULT_SPIN>, dim3((unsigned)grid), dim3(kAdamTmaThreads),
                      kAdamTmaSmem, stream, p);
}

template <int MAXN>
cudaError_t gather_impl(const void *const *shards, int n, int64_t src_off, int64_t shard_bytes,
                        void *out, int64_t dst_stride, int64_t spin_limit, int *error, cudaStream_t stream) {
    GatherParams<MAXN> p;
    for (int j = 0; j < n; ++j) p.src[j] = static_cast<const char *>(shards[j]) + src_off;
    for (int j = n; j < MAXN; ++j) p.src[j] = nullptr;
    p.dst = static_cast<char *>(out);
    p.dst_stride = dst_stride;
    p.shard_bytes = shard_bytes;
    p.chunks_per_shard = (shard_bytes + kGatherChunk - 1) / kGatherChunk;
    p.n_chunks = p.chunks_per_shard * n;
    p.spin_limit = spin_limit;
    p.error = error;
    p.n = n;
    if (p.n_chunks == 0) return cudaSuccess;
    const size_t smem = (size_t)kGatherStages * kGatherChunk;
    static const cudaError_t attr = cudaFuncSetAttribute(
        gather_layer_tma<MAXN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (attr != cudaSuccess) return attr;
    static const int occ = occupancy(gather_layer_tma<MAXN>, 32, smem);
    long long grid = (long long)sm_count() * occ;
    if (grid > p.n_chunks) grid = p.n_chunks;
    return launch_pdl(gather_layer_tma<MAXN>, dim3((unsigned)grid), dim3(32), smem, stream, p);
}

}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev[dev].sms == 0) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_dev[dev].sms = sms > 0 ? sms : 1;
    }
    return g_dev[dev].sms;
}

template <int MAXN, int VPT, int THREADS>
cudaError_t reduce_dispatch(const void *const *slices, int n_src, int n, int lp, bool acc_lp,
                            const ReduceSegment *segs, int n_segs, float inv, cudaStream_t stream) {
    if (lp)
        return acc_lp ? reduce_impl<MAXN, true, true, VPT, THREADS>(slices, n_src, n, segs, n_segs, inv, stream)
                      : reduce_impl<MAXN, true, false, VPT, THREADS>(slices, n_src, n, segs, n_segs, inv, stream);
    return acc_lp ? reduce_impl<MAXN, false, true, VPT, THREADS>(slices, n_src, n, segs, n_segs, inv, stream)
                  : reduce_impl<MAXN, false, false, VPT, THREADS>(slices, n_src, n, segs, n_segs, inv, stream);
}

cudaError_t launch_reduce(const void *const *slices, int n_src, int n, int lp, int acc_lp,
                          const ReduceSegment *segs, int n_segs, float inv, cudaStream_t stream) {
    if (n_src > reduce_src_table(n)) return cudaErrorInvalidValue;
    if (n <= kSmallN)
        return reduce_dispatch<kSmallN, kSmallVpt, kSmallThreads>(slices, n_src, n, lp, acc_lp != 0, segs,
                                                                  n_segs, inv, stream);
    if (n <= 64)
        return reduce_dispatch<64, kReduceVpt, kReduceThreads>(slices, n_src, n, lp, acc_lp != 0, segs, n_segs,
                                                               inv, stream);
    return reduce_dispatch<1024, kReduceVpt, kReduceThreads>(slices, n_src, n, lp, acc_lp != 0, segs, n_segs,
                                                             inv, stream);
}

cudaError_t launch_norm(const NormLaunch &a, cudaStream_t stream) {
    DecideParams p;
    p.partials = a.partials;
    p.level2 = a.level2;
    p.overflow = a.overflow;
    p.arrivals = a.arrivals;
    p.stats_out = a.stats_out;
    p.stats_in = a.stats_in;
    p.tiles_per_slot = a.tiles_per_slot;
    p.chunks_per_slot = (int)((a.tiles_per_slot + kPartialChunk - 1) / kPartialChunk);
    if (p.chunks_per_slot < 1) p.chunks_per_slot = 1;
    if (a.n_slots < 1 || a.n_slots > kNormMaxSlots) return cudaErrorInvalidValue;
    p.n_slots = a.n_slots;
    p.mode = a.mode;
    int active = 0;
    if (a.mode != kDecideGlobal) {
        for (int r = 0; r < a.n_slots; ++r)
            if ((a.active_mask[r >> 6] >> (r & 63)) & 1u) p.slots[active++] = (short)r;
        if (active == 0) return cudaErrorInvalidValue;
    }
    p.n_active = active;
    p.remote_sumsq = a.remote_sumsq;
    p.remote_overflow = a.remote_overflow;
    p.clip = a.clip;
    p.loss_scale = a.loss_scale;
    p.beta1 = a.beta1;
    p.beta2 = a.beta2;
    p.growth_interval = a.growth_interval;
    p.rec = a.rec;
    p.bc_t0 = a.bc_t0;
    for (int i = 0; i < kBcTable; ++i) {
        p.bc1_tab[i] = a.bc1_tab ? a.bc1_tab[i] : 0.0f;
        p.bc2_tab[i] = a.bc2_tab ? a.bc2_tab[i] : 0.0f;
    }
    const long long blocks = a.mode == kDecideGlobal ? 1 : (long long)active * p.chunks_per_slot;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
    return launch_pdl(norm_decide, dim3((unsigned)blocks), dim3(kDecideThreads), 0, stream, p);
}

cudaError_t launch_adam(const AdamSegment *segs, int n_segs, int lp, const StepRecord *rec, int *error,
                        int64_t spin_limit, float lr, float beta1, float beta2, float omb1, float omb2,
                        float eps, float wd, float decay, int adamw, cudaStream_t stream) {
    if (n_segs < 1 || n_segs > kMaxAdamSegments) return cudaErrorInvalidValue;
    AdamTmaParams q;
    long long tiles = 0;
    int k = 0;
    for (int i = 0; i < n_segs; ++i) {
        if (segs[i].len <= 0) continue;
        q.seg[k].g = segs[i].g;
        q.seg[k].master = segs[i].master;
        q.seg[k].m = segs[i].m;
        q.seg[k].v = segs[i].v;
        q.seg[k].param = static_cast<uint16_t *>(segs[i].param);
        q.seg[k].len = segs[i].len;
        q.seg[k].tile0 = tiles;
        tiles += (segs[i].len + kAdamTile - 1) / kAdamTile;
        ++k;
    }
    if (k == 0) return cudaSuccess;
    for (int i = k; i < kMaxAdamSegments; ++i) {
        q.seg[i] = AdamSegDev{nullptr, nullptr, nullptr, nullptr, nullptr, 0, tiles};
    }
    q.n_tiles = tiles;
    q.n_seg = k;
    q.rec = rec;
    q.error = error;
    q.spin_limit = spin_limit;
    q.lr = lr;
    q.beta1 = beta1;
    q.beta2 = beta2;
    q.omb1 = omb1;
    q.omb2 = omb2;
    q.eps = eps;
    q.wd = wd;
    q.decay = decay;
    q.adamw = adamw;
    if (spin_limit == kDefaultSpinLimit)
        return lp ? adam_tma_impl<true, true>(q, stream) : adam_tma_impl<false, true>(q, stream);
    return lp ? adam_tma_impl<true, false>(q, stream) : adam_tma_impl<false, false>(q, stream);
}

cudaError_t launch_gather(const void *const *shards, int n, int64_t src_offset_bytes,
                          int64_t shard_bytes, void *out, int64_t dst_stride_bytes, int64_t spin_limit,
                          int *error, cudaStream_t stream) {
    if (n <= 64)
        return gather_impl<64>(shards, n, src_offset_bytes, shard_bytes, out, dst_stride_bytes, spin_limit,
                               error, stream);
    return gather_impl<1024>(shards, n, src_offset_bytes, shard_bytes, out, dst_stride_bytes, spin_limit,
                             error, stream);
}

}  // namespace zk
