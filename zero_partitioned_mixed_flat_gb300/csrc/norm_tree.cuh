// norm_tree.cuh -- the fixed summation tree of the global gradient norm
// ("从'年糕切片'理解ZeRO" §4.2: clipping by the global L2 norm), shared by the
// decision kernel (kernels.cu) and the allocation-free reduce (noalloc.cu).
//
// Levels (every shape depends only on the partition sizes, never on the grid,
// the bucket size or which block finishes first):
//   0  one fp64 partial per 4096-element norm tile (the reduce kernel);
//   1  chunk_sum: the partials of one chunk of kPartialChunk tiles of one
//      partition -> one double (a 256-thread block: 16 values per thread added
//      pairwise, an xor butterfly per warp, the 8 warps pairwise);
//   2  slot_sum_warp: the chunk sums of one partition -> the partition's sum of
//      squares (one warp: lane l adds chunks l, l+32, ... in order, then the
//      xor butterfly);
//   3  vector_sum_block: the per-partition sums in partition order (zero for a
//      partition not reduced in the step) -> the global sum (thread t adds
//      entries t, t+256, t+512, t+768 pairwise, then the block tree).
// Adding an exact zero never changes a sum, so a partition that is absent on
// one rank and present on another contributes the same bits everywhere.
#pragma once

#include "zero_internal.h"

namespace zk {

constexpr int kNormThreads = 256;
constexpr int kNormMaxSlots = 1024;  // entries of the level-3 vector

// xor butterfly: IEEE addition is commutative, so every lane ends with the
// same value
__device__ __forceinline__ double warp_sum_fixed(double acc) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc = __dadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    return acc;
}

// whole block (kNormThreads); the result is valid in thread 0.  wsum: 8 doubles
// of shared memory, free on entry.
__device__ __forceinline__ double block_sum_fixed(double acc, double *wsum) {
    acc = warp_sum_fixed(acc);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = acc;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {  // pairwise over the warps
        double w[kNormThreads / 32];
#pragma unroll
        for (int i = 0; i < kNormThreads / 32; ++i) w[i] = wsum[i];
#pragma unroll
        for (int h = kNormThreads / 64; h >= 1; h >>= 1)
#pragma unroll
            for (int i = 0; i < h; ++i) w[i] = __dadd_rn(w[i], w[i + h]);
        t = w[0];
    }
    __syncthreads();  // wsum may be reused at once
    return t;
}

// level 1: q[t0, t1), t1 - t0 <= kPartialChunk; every load is issued before the
// first add (a missing term is 0).  Whole block; valid in thread 0.
__device__ __forceinline__ double chunk_sum(const double *q, long long t0, long long t1, double *wsum) {
    constexpr int kPer = (int)(kPartialChunk / kNormThreads);
    static_assert((kPer & (kPer - 1)) == 0 && ((kNormThreads / 32) & (kNormThreads / 32 - 1)) == 0,
                  "pairwise trees need powers of two");
    double x[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const long long t = t0 + threadIdx.x + (long long)i * kNormThreads;
        x[i] = t < t1 ? q[t] : 0.0;
    }
#pragma unroll
    for (int h = kPer / 2; h >= 1; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) x[i] = __dadd_rn(x[i], x[i + h]);
    return block_sum_fixed(x[0], wsum);
}

// level 2: n chunk sums, load(k) gives chunk k.  One whole warp; every lane
// gets the result.
template <typename Load>
__device__ __forceinline__ double slot_sum_warp(Load load, int n) {
    const int lane = threadIdx.x & 31;
    double acc = 0.0;
    for (int k = lane; k < n; k += 32) acc = __dadd_rn(acc, load(k));
    return warp_sum_fixed(acc);
}

// level 3: v[0, n), n <= kNormMaxSlots, in shared or global memory.  Whole
// block; valid in thread 0.
__device__ __forceinline__ double vector_sum_block(const double *v, int n, double *wsum) {
    static_assert(kNormMaxSlots == 4 * kNormThreads, "four entries per thread");
    const int t = threadIdx.x;
    const double a = t < n ? v[t] : 0.0;
    const double b = t + kNormThreads < n ? v[t + kNormThreads] : 0.0;
    const double c = t + 2 * kNormThreads < n ? v[t + 2 * kNormThreads] : 0.0;
    const double d = t + 3 * kNormThreads < n ? v[t + 3 * kNormThreads] : 0.0;
    return block_sum_fixed(__dadd_rn(__dadd_rn(a, b), __dadd_rn(c, d)), wsum);
}

}  // namespace zk
