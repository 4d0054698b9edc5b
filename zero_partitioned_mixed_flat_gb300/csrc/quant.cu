// quant.cu -- the quantized stage-3 gather (sm_103a).
//
// ZeRO++ ("ZeRO-1/2/3 分别优化了什么" note, ZeRO++: the all-gathered
// parameters are quantized to cut the traffic): each rank turns its lp shard
// into 1-byte codes with one float scale per 128-element block -- int8
// (symmetric, block max -> 127, nearest-even) or OCP FP8 E4M3 with a
// power-of-two scale -- and the gather expands code * scale back to lp while
// it concatenates the ranks' shards.  Per layer element the gather
// moves 1 B + 4/128 B in and 2 B out, against 2 B in and 2 B out for the lp
// gather.  Both kernels are plain streaming kernels; each thread keeps several
// independent loads in flight before it computes, and every warp load and
// store is one contiguous run.
#include "launch.h"
#include "zero_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace zk {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;   // blocks per warp (quantize) / items per thread (gather)

// two floats -> two lp values in one packed conversion (each rounded to
// nearest, ties to even, as a separate conversion would)
template <bool BF16>
__device__ __forceinline__ uint32_t to_lp2_packed(float a, float b) {
    if constexpr (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// byte k of w (a signed code) as an exact float without the conversion unit:
// w ^ 0x80808080 holds code + 128 in each byte; one byte permute places it in
// the low mantissa bits of 2^23, and subtracting 2^23 + 128 is exact.
__device__ __forceinline__ float code_to_float(uint32_t biased, int k) {
    const uint32_t bits = __byte_perm(biased, 0x4B000000u, 0x7540u + (uint32_t)k);
    return __fsub_rn(__uint_as_float(bits), 8388736.0f);
}

// The code of x: the nearest-even integer of the correctly rounded quotient
// x / scale, clamped to +-127, as a byte (the division, for the rare elements
// that the fast path below leaves to it).
__device__ __forceinline__ uint32_t code_by_division(float x, float scale) {
    if (!(scale > 0.0f)) return 0u;
    int c = __float2int_rn(__fdiv_rn(x, scale));
    c = c > 127 ? 127 : (c < -127 ? -127 : c);
    return (uint32_t)c & 0xffu;
}

// Adding 1.5 * 2^23 to a float q with |q| < 2^22 leaves the nearest-even
// integer k of q in the low mantissa bits (the adder rounds to nearest even,
// and 1.5 * 2^23 is even), so the low byte of the sum is k as a signed byte
// and subtracting the constant back gives k exactly.
constexpr float kRoundMagic = 12582912.0f;

// hardware reciprocal approximation (within one ulp of 1/x for normal x)
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// K codes of one thread's elements (K a multiple of 4), packed 4 per word
// (byte k = element k).
// Fast path, with p = x * rcp the exact product (rcp within one ulp of
// 1/scale, so p lies within 2^-23 |x/scale| <= 1.6e-5 of the exact quotient):
// one fused multiply-add rounds p to its nearest-even integer k (through the
// 1.5 * 2^23 addition) and another gives d = p - k rounded once.  When every
// |d| < 1/2 - 2^-13, the correctly rounded quotient RN(x / scale) (within
// 7.6e-6 of the exact one) is farther than 9e-5 from a half-integer and rounds
// to the same k (and |k| <= 127 needs no clamp).  Otherwise (rare: ties, a
// NaN element), and for a zero, subnormal-small, huge or non-finite scale,
// every element is divided.
template <int K>
__device__ __forceinline__ void quant_codes(const float v[K], float scale, uint32_t packed[K / 4]) {
    bool divide = !(scale >= 0x1p-100f && scale <= 0x1p+100f);
    if (!divide) {
        const float rcp = rcp_approx(scale);
        uint32_t t[K];
        bool near = false;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float r = __fmaf_rn(v[k], rcp, kRoundMagic);
            const float d = __fmaf_rn(v[k], rcp, -__fsub_rn(r, kRoundMagic));
            near |= !(fabsf(d) < 0.5f - 0x1p-13f);
            t[k] = __float_as_uint(r);
        }
#pragma unroll
        for (int w = 0; w < K / 4; ++w)
            packed[w] = __byte_perm(__byte_perm(t[4 * w], t[4 * w + 1], 0x0040u),
                                    __byte_perm(t[4 * w + 2], t[4 * w + 3], 0x0040u), 0x5410u);
        divide = near;
    }
    if (divide) {
#pragma unroll
        for (int w = 0; w < K / 4; ++w) packed[w] = 0u;
#pragma unroll
        for (int k = 0; k < K; ++k) packed[k >> 2] |= code_by_division(v[k], scale) << (8 * (k & 3));
    }
}

// scale = amax / 127 correctly rounded, without the division routine for the
// usual range: Markstein's correction step (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with y = RN(1/127) and q0 = RN(amax * y), the remainder
// r = amax - 127 q0 is exact in one fused multiply-add, and q1 = RN(q0 + r y)
// is the correctly rounded quotient.  The block maximum is always an lp value,
// and the test suite checks q1 against the IEEE division for every positive
// finite fp16 and bf16 value in [2^-90, 2^100]; outside that range (and for an
// infinite maximum) the division routine is used.
__device__ __forceinline__ float scale_of_amax(float amax) {
    if (!(amax >= 0x1p-90f && amax <= 0x1p+100f)) return __fdiv_rn(amax, 127.0f);
    constexpr float y = 1.0f / 127.0f;
    const float q0 = __fmul_rn(amax, y);
    const float r = __fmaf_rn(-q0, 127.0f, amax);
    return __fmaf_rn(r, y, q0);
}

// ---- fp8 (OCP E4M3) variant: a power-of-two block scale 2^e with
// e = floor(log2 amax) - 7 clamped to [-126, 120] (120 for an infinite amax),
// so amax / 2^e lies in [128, 256): code = E4M3(x * 2^-e), nearest even,
// finite overflow and infinities saturated to +-448.

// two floats -> two E4M3 codes, a in the low byte (one conversion instruction)
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// two E4M3 codes (low byte first) -> two exact floats
__device__ __forceinline__ float2 from_e4m3x2(uint32_t two) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)two));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// the block scale exponent from amax's bits (amax >= 0, not NaN)
__device__ __forceinline__ int fp8_scale_exponent(float amax) {
    const int biased = (int)(__float_as_uint(amax) >> 23);
    int e = biased == 0 ? -126 : biased - 127 - 7;
    e = e < -126 ? -126 : e;
    return e > 120 ? 120 : e;
}

template <int K>
__device__ __forceinline__ void quant_codes_fp8(const float v[K], float amax, float &scale,
                                                uint32_t packed[K / 4]) {
    if (amax == 0.0f) {  // an all-zero block: scale 0 and codes 0 (also for -0)
        scale = 0.0f;
#pragma unroll
        for (int w = 0; w < K / 4; ++w) packed[w] = 0u;
        return;
    }
    const int e = fp8_scale_exponent(amax);
    scale = __uint_as_float((uint32_t)(e + 127) << 23);
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
    for (int w = 0; w < K / 4; ++w) {
        const uint32_t lo = to_e4m3x2(__fmul_rn(v[4 * w], inv), __fmul_rn(v[4 * w + 1], inv));
        const uint32_t hi = to_e4m3x2(__fmul_rn(v[4 * w + 2], inv), __fmul_rn(v[4 * w + 3], inv));
        packed[w] = lo | (hi << 16);
    }
}

template <bool BF16>
__device__ __forceinline__ void from_lp4(uint2 raw, float v[4]) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if constexpr (BF16) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        } else {
            const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            v[2 * k] = t.x;
            v[2 * k + 1] = t.y;
        }
    }
}

// Eight lanes per 128-element block, 16 contiguous elements per lane (two
// 16-byte loads), four blocks per warp, one group of four blocks per warp and
// iteration (1 to 4 groups per iteration were swept on GB300: 1 is fastest):
// lane l holds elements 16(l mod 8) .. 16(l mod 8) + 15 of block
// 4*group + l/8.  The block maximum takes three xor shuffles; scale =
// amax / 127 (correctly rounded, scale_of_amax), code = nearest-even integer of
// x / scale (the correctly rounded float quotient, see quant_codes), clamped to
// +-127.  FP8: the E4M3 codes and power-of-two scale of quant_codes_fp8
// instead.  Each lane writes its 16 codes with one 16-byte store.  (Versus a
// half-warp per block with 8 elements per lane: the per-block work -- the
// shuffles and the scale -- is shared by twice the elements.)

template <bool BF16, bool FP8>
__global__ void __launch_bounds__(kQuantThreads, 3)  // 16 values per lane without spills
quantize_shard_blocks(const uint4 *__restrict__ x, uint4 *__restrict__ q, float *__restrict__ scales,
                      long long n_blocks) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int l8 = lane & 7;
    const long long n_groups = (n_blocks + 3) / 4;
    const long long warps = (long long)gridDim.x * (kQuantThreads / 32);
    const long long w0 = (long long)blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5);
    // int8: a software pipeline, the next group's two loads in flight while
    // this group is quantized (the exactness test makes the compute long: 0.081
    // -> 0.071 ms at 7.5B); fp8, whose compute is short, loads then computes
    // (the pipeline measured 3 % slower there)
    auto load = [&](long long group, uint4 r[2]) {
        const long long b = 4 * group + (lane >> 3);
        if (group < n_groups && b < n_blocks) {
            r[0] = __ldg(x + b * 16 + 2 * l8);
            r[1] = __ldg(x + b * 16 + 2 * l8 + 1);
        } else {
            r[0] = r[1] = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    uint4 cur[2], nxt[2];
    if constexpr (!FP8) load(w0, cur);
    for (long long group = w0; group < n_groups; group += warps) {  // uniform across the warp
        if constexpr (FP8) {
            load(group, cur);
        } else {
            load(group + warps, nxt);
        }
        const long long b = 4 * group + (lane >> 3);
        float v[16];
        from_lp4<BF16>(make_uint2(cur[0].x, cur[0].y), v);
        from_lp4<BF16>(make_uint2(cur[0].z, cur[0].w), v + 4);
        from_lp4<BF16>(make_uint2(cur[1].x, cur[1].y), v + 8);
        from_lp4<BF16>(make_uint2(cur[1].z, cur[1].w), v + 12);
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
        for (int off = 4; off > 0; off >>= 1)  // within each group of 8 lanes
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        float scale;
        uint32_t packed[4];
        if constexpr (FP8) {
            quant_codes_fp8<16>(v, amax, scale, packed);
        } else {
            scale = scale_of_amax(amax);
            quant_codes<16>(v, scale, packed);
        }
        if (b < n_blocks) {
            __stcs(q + b * 8 + l8, make_uint4(packed[0], packed[1], packed[2], packed[3]));
            if (l8 == 0) scales[b] = scale;
        }
        if constexpr (!FP8) {
            cur[0] = nxt[0];
            cur[1] = nxt[1];
        }
    }
}

template <int MAXN>
struct DequantGatherParams {
    const uint2 *codes[MAXN];   // rank j's codes at this unit's offset (8 per uint2)
    const float *scales[MAXN];  // rank j's scales at this unit's first block
    uint4 *out;                 // 8 lp per uint4
    long long vec_per_shard;    // shard_len / 8
};

// out[j * shard + k] = lp(code_j[k] * scale_j[k / 128]).  blockIdx.y is the
// rank j; along x a thread takes kQuantUnroll items of 8 codes (one 8-byte
// load each, all issued before any use) and writes each item's 8 lp values
// with one 16-byte store, so a warp's loads and stores are contiguous runs.
// FP8: the codes are E4M3, widened exactly by the conversion instruction.
template <int MAXN, bool BF16, bool FP8>
__global__ void __launch_bounds__(kQuantThreads)
gather_dequant(const __grid_constant__ DequantGatherParams<MAXN> p) {
    pdl_enter();
    const int j = blockIdx.y;
    const uint2 *codes = p.codes[j];
    const float *scales = p.scales[j];
    uint4 *out = p.out + (long long)j * p.vec_per_shard;
    const long long stride = (long long)gridDim.x * kQuantThreads;
    for (long long k0 = (long long)blockIdx.x * kQuantThreads + threadIdx.x; k0 < p.vec_per_shard;
         k0 += stride * kQuantUnroll) {
        uint2 c[kQuantUnroll];
        float sc[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const long long k = k0 + u * stride;
            if (k < p.vec_per_shard) {
                c[u] = __ldcs(codes + k);
                sc[u] = __ldg(scales + (k >> 4));  // 8 codes lie in one 128-block
            }
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const long long k = k0 + u * stride;
            if (k >= p.vec_per_shard) break;
            uint32_t o[4];
            if constexpr (FP8) {
                const uint32_t w[2] = {c[u].x, c[u].y};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 f = from_e4m3x2(w[t >> 1] >> (16 * (t & 1)));
                    o[t] = to_lp2_packed<BF16>(__fmul_rn(f.x, sc[u]), __fmul_rn(f.y, sc[u]));
                }
            } else {
                const uint32_t w[2] = {c[u].x ^ 0x80808080u, c[u].y ^ 0x80808080u};
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    float y[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) y[q] = __fmul_rn(code_to_float(w[t], q), sc[u]);
                    o[2 * t] = to_lp2_packed<BF16>(y[0], y[1]);
                    o[2 * t + 1] = to_lp2_packed<BF16>(y[2], y[3]);
                }
            }
            __stcs(out + k, make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
}

template <typename K>
int blocks_per_sm(K kernel) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kQuantThreads, 0) != cudaSuccess) b = 1;
    return b < 1 ? 1 : b;
}

template <int MAXN, bool BF16, bool FP8>
cudaError_t dequant_gather_impl(const int8_t *const *codes, const float *const *scales, int n,
                                int64_t offset, int64_t shard_len, void *out, cudaStream_t stream) {
    DequantGatherParams<MAXN> p;
    for (int j = 0; j < n; ++j) {
        p.codes[j] = reinterpret_cast<const uint2 *>(codes[j] + offset);
        p.scales[j] = scales[j] + offset / 128;
    }
    for (int j = n; j < MAXN; ++j) {
        p.codes[j] = nullptr;
        p.scales[j] = nullptr;
    }
    p.out = static_cast<uint4 *>(out);
    p.vec_per_shard = shard_len / 8;
    if (p.vec_per_shard == 0 || n == 0) return cudaSuccess;
    static const int occ = blocks_per_sm(gather_dequant<MAXN, BF16, FP8>);
    // about two waves of CTAs over all ranks
    const long long per_rank_need = (p.vec_per_shard + kQuantThreads * kQuantUnroll - 1) /
                                    (kQuantThreads * kQuantUnroll);
    long long gx = (2LL * sm_count() * occ + n - 1) / n;
    if (gx > per_rank_need) gx = per_rank_need;
    if (gx < 1) gx = 1;
    return launch_pdl(gather_dequant<MAXN, BF16, FP8>, dim3((unsigned)gx, (unsigned)n), dim3(kQuantThreads), 0,
                      stream, p);
}

template <bool BF16, bool FP8>
cudaError_t quantize_impl(const void *shard, int64_t len, int8_t *codes, float *scales, cudaStream_t stream) {
    const long long blocks = len / 128;
    if (blocks == 0) return cudaSuccess;
    static const int occ = blocks_per_sm(quantize_shard_blocks<BF16, FP8>);
    long long grid = (long long)sm_count() * occ;
    const long long per_cta = (kQuantThreads / 32) * 4;  // blocks per CTA per iteration
    const long long need = (blocks + per_cta - 1) / per_cta;
    if (grid > need) grid = need;
    return launch_pdl(quantize_shard_blocks<BF16, FP8>, dim3((unsigned)grid), dim3(kQuantThreads), 0, stream,
                      static_cast<const uint4 *>(shard), reinterpret_cast<uint4 *>(codes), scales, blocks);
}

}  // namespace

cudaError_t launch_quantize(const void *shard, int lp, int fp8, int64_t len, int8_t *codes, float *scales,
                            cudaStream_t stream) {
    if (fp8)
        return lp ? quantize_impl<true, true>(shard, len, codes, scales, stream)
                  : quantize_impl<false, true>(shard, len, codes, scales, stream);
    return lp ? quantize_impl<true, false>(shard, len, codes, scales, stream)
              : quantize_impl<false, false>(shard, len, codes, scales, stream);
}

template <int MAXN>
cudaError_t dequant_dispatch(const int8_t *const *codes, const float *const *scales, int n, int lp, int fp8,
                             int64_t offset, int64_t shard_len, void *out, cudaStream_t stream) {
    if (fp8)
        return lp ? dequant_gather_impl<MAXN, true, true>(codes, scales, n, offset, shard_len, out, stream)
                  : dequant_gather_impl<MAXN, false, true>(codes, scales, n, offset, shard_len, out, stream);
    return lp ? dequant_gather_impl<MAXN, true, false>(codes, scales, n, offset, shard_len, out, stream)
              : dequant_gather_impl<MAXN, false, false>(codes, scales, n, offset, shard_len, out, stream);
}

cudaError_t launch_dequant_gather(const int8_t *const *codes, const float *const *scales, int n, int lp,
                                  int fp8, int64_t offset, int64_t shard_len, void *out, cudaStream_t stream) {
    if (n <= 64) return dequant_dispatch<64>(codes, scales, n, lp, fp8, offset, shard_len, out, stream);
    return dequant_dispatch<1024>(codes, scales, n, lp, fp8, offset, shard_len, out, stream);
}

}  // namespace zk
