// noalloc.cu -- zero_reduce_partition_noalloc: the reduce + unscale + overflow
// + sum-of-squares step for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a framework whose caching allocator owns
// every byte of the GPU (an out-of-band cudaMalloc would fail or fragment its
// pool), or a latency-critical loop that must not pay cudaMalloc's implicit
// device synchronisation.  The plan-based zero_reduce_partition allocates its
// scratch (per-tile partial sums and the overflow word) on first use; this
// variant instead keeps that scratch in one fixed-size array in device memory
// that is part of the library image, so it allocates nothing.
//
// The array lives on every GPU that loads the library, until the process
// exits.  Every call shares it and it keeps the last call's contents, so calls
// whose device work overlaps (two streams, two host threads) race on it.
#include "norm_tree.cuh"
#include "zero.h"
#include "zero_internal.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace {

constexpr int64_t kMaxTiles = ZERO_NOALLOC_MAX_ELEMS / zk::kTile;
constexpr int64_t kMaxChunks = (kMaxTiles + zk::kPartialChunk - 1) / zk::kPartialChunk;
constexpr size_t kScratchBytes = size_t(kMaxTiles) * sizeof(double) + 256;
static_assert(ZERO_NOALLOC_MAX_ELEMS % zk::kTile == 0, "maximum must be whole norm tiles");
static_assert(kScratchBytes == size_t(ZERO_NOALLOC_SCRATCH_BYTES),
              "the header's scratch size must match the array");
static_assert(kMaxChunks * sizeof(double) + sizeof(unsigned) <= 256, "tail holds chunk sums and the flag");

// [0, kMaxTiles*8): per-tile fp64 partial sums; then, in the 256-byte tail, one
// 32-bit overflow word
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device

zero_status noalloc_fail(zero_status code, const char *msg) {
    zk::set_last_error(msg);  // reported by zero_last_error()
    return code;
}

// The partition's sum of squares with the plan path's tree (norm_tree.cuh:
// chunk sums, then one warp over the chunks), so *sumsq_out equals what
// zero_partition_stats exports for the same partition, bit for bit; and the
// overflow word.  One block of kNormThreads.
__global__ void __launch_bounds__(zk::kNormThreads)
noalloc_finalize(const double *partials, long long n_tiles, const unsigned *overflow,
                 double *sumsq_out, int *overflow_out) {
    __shared__ double wsum[zk::kNormThreads / 32];
    __shared__ double chunks[kMaxChunks];
    const int n_chunks = n_tiles > 0 ? (int)((n_tiles + zk::kPartialChunk - 1) / zk::kPartialChunk) : 1;
    for (int c = 0; c < n_chunks; ++c) {
        const long long t0 = (long long)c * zk::kPartialChunk;
        const long long t1 = t0 + zk::kPartialChunk < n_tiles ? t0 + zk::kPartialChunk : n_tiles;
        const double s = zk::chunk_sum(partials, t0, t1, wsum);
        if (threadIdx.x == 0) chunks[c] = s;
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;
    const double s = zk::slot_sum_warp([](int k) { return chunks[k]; }, n_chunks);
    if (threadIdx.x == 0) {
        *sumsq_out = s;
        *overflow_out = *overflow ? 1 : 0;
    }
}

}  // namespace

extern "C" zero_status zero_reduce_partition_noalloc(int32_t n_ranks, zero_lp lp,
                                                     const void *const *grad_slices, int64_t len,
                                                     float loss_scale, float *grad_out,
                                                     double *sumsq_out, int32_t *overflow_out,
                                                     void *stream) {
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS) return noalloc_fail(ZERO_EINVAL, "n_ranks out of range");
    if (lp != ZERO_FP16 && lp != ZERO_BF16) return noalloc_fail(ZERO_EINVAL, "unknown lp type");
    if (len < 0 || len % 8 != 0) return noalloc_fail(ZERO_EINVAL, "len must be a non-negative multiple of 8");
    if (len > ZERO_NOALLOC_MAX_ELEMS)
        return noalloc_fail(ZERO_EINVAL, "len exceeds ZERO_NOALLOC_MAX_ELEMS (the fixed scratch holds "
                                         "the partial sums of at most that many elements)");
    if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale))
        return noalloc_fail(ZERO_EINVAL, "loss_scale must be finite and > 0");
    if (!grad_slices || !sumsq_out || !overflow_out || (len > 0 && !grad_out))
        return noalloc_fail(ZERO_EINVAL, "NULL pointer argument");
    for (int32_t j = 0; j < n_ranks; ++j) {
        if (len > 0 && !grad_slices[j]) return noalloc_fail(ZERO_EINVAL, "NULL gradient slice");
        if (reinterpret_cast<uintptr_t>(grad_slices[j]) & 15u)
            return noalloc_fail(ZERO_EALIGN, "a gradient slice is not 16-byte aligned");
    }
    if ((reinterpret_cast<uintptr_t>(grad_out) & 15u) || (reinterpret_cast<uintptr_t>(sumsq_out) & 7u) ||
        (reinterpret_cast<uintptr_t>(overflow_out) & 3u))
        return noalloc_fail(ZERO_EALIGN, "an output pointer is misaligned");

    // set-up, once per device, with that device current: the host-side name of
    // the array is only a stand-in, the kernels need its device address
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return noalloc_fail(ZERO_ECUDA, "cudaGetDevice failed");
    }
    if (dev < 0 || dev >= kMaxDevices)
        return noalloc_fail(ZERO_EINVAL, "device ordinal is 64 or more: the allocation-free reduce keeps "
                                         "its scratch address for devices 0-63 only");
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_addr[dev]) {
            void *ptr = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr) {
                char msg[160];
                std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
                return noalloc_fail(ZERO_ECUDA, msg);
            }
            g_scratch_addr[dev] = ptr;
        }
        base = g_scratch_addr[dev];
    }
    double *partials = static_cast<double *>(base);
    unsigned *overflow = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(base) +
                                                      size_t(kMaxTiles) * sizeof(double));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the overflow word keeps the previous call's value: clear it
    cudaError_t e = cudaMemsetAsync(overflow, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return noalloc_fail(ZERO_ECUDA, cudaGetErrorString(e));
    const float inv = float(1.0 / (double(loss_scale) * double(n_ranks)));
    if (len > 0) {
        const zk::ReduceSegment whole = {0, len, 0, grad_out, partials, overflow, 0};
        e = zk::launch_reduce(grad_slices, n_ranks, n_ranks, lp, 0, &whole, 1, inv, s);
        if (e != cudaSuccess) return noalloc_fail(ZERO_ECUDA, cudaGetErrorString(e));
    }
    const long long n_tiles = (len + zk::kTile - 1) / zk::kTile;
    noalloc_finalize<<<1, zk::kNormThreads, 0, s>>>(partials, n_tiles, overflow, sumsq_out, overflow_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) return noalloc_fail(ZERO_ECUDA, cudaGetErrorString(e));
    return ZERO_OK;
}
