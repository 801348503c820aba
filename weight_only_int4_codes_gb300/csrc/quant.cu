// quant.cu -- group-wise int4 quantize + pack, and dequantize (test aid), for
// fp16 and bfloat16 weights.
//
// Quantizer (page "Beating FP16 with 4-bit Weights: A Portable W4A16 GEMM in
// Triton", section "The design": one scale and one zero-point per group of 128
// rows, eight 4-bit values per int32 along K; the codes are unsigned in [0,15]
// and dequantize as (q - z) * s, the HQQ form of the GemLite README).
//
// Symmetric variant (the first page's tests cover symmetric and asymmetric
// quantization; its "+8 zero-point" bug is the symmetric packing): signed
// codes c = clamp(rint(w / s), -8, 7) stored as q = c + 8, z = 8, with
// s = fp16(max|w| / 7) -- the largest magnitude maps to +-7.
//
// One thread owns one (group, column): it scans the group's rows for min/max,
// forms s, z in fp64, then codes and packs the rows.  Neighbouring threads own
// neighbouring columns, so every load and store is coalesced along N.  The
// arithmetic is fp64 so that every rounding decision (the scale's rounding to
// fp16, rint of -min/s and of w/s) is taken on the exactly-rounded fp64 value,
// which is what makes the codes bit-exact with an fp64 reference.
#include "common.cuh"

namespace w4a16 {
namespace {

constexpr int kQuantThreads = 128;

__global__ void __launch_bounds__(kQuantThreads)
quantize_pack_kernel(const __half *__restrict__ W, int K, int N, int group, bool symmetric,
                     uint32_t *__restrict__ packed, __half *__restrict__ scales,
                     __half *__restrict__ zeros)
{
    const int n = blockIdx.x * kQuantThreads + threadIdx.x;
    if (n >= N) return;
    for (int j = blockIdx.y; j < K / group; j += gridDim.y) {   // group index
    const size_t k0 = (size_t)j * group;
    float mn = __int_as_float(0x7f800000);          // +inf
    float mx = -mn;
    for (int k = 0; k < group; ++k) {
        const float v = __half2float(W[(k0 + k) * N + n]);   // exact
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
    }
    // difference (or largest magnitude) and quotient in fp64, one rounding to
    // binary16 (RN-even)
    __half sh = symmetric ? __double2half(fmax(-(double)mn, (double)mx) / 7.0)
                          : __double2half(((double)mx - (double)mn) / 15.0);
    double s = (double)__half2float(sh);
    if (s == 0.0) {                                 // degenerate (constant or all-zero) group
        sh = __float2half_rn(1.0f);
        s = 1.0;
    }
    int z = 8;
    if (!symmetric) {
        double zr = rint(-(double)mn / s);
        zr = fmin(fmax(zr, 0.0), 15.0);
        z = (int)zr;                                // +0 for a clamped -0
    }
    scales[(size_t)j * N + n] = sh;
    zeros[(size_t)j * N + n] = __int2half_rn(z);
    for (int r = 0; r < group / 8; ++r) {
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const double v = (double)__half2float(W[(k0 + 8 * r + i) * N + n]);
            double qd = rint(v / s) + (double)z;
            qd = fmin(fmax(qd, 0.0), 15.0);
            word |= (uint32_t)qd << (4 * i);
        }
        packed[(k0 / 8 + r) * N + n] = word;
    }
    }
}

constexpr int kDequantThreads = 256;

// One thread per packed word: W_out[k,n] = fp16((q - z) * s).  q - z is an
// integer in [-15, 15], exact in fp16, and the fp16 multiply rounds the exact
// product once -- the same value as rounding (q - z) * s computed exactly.
__global__ void __launch_bounds__(kDequantThreads)
dequantize_kernel(const uint32_t *__restrict__ packed, const __half *__restrict__ scales,
                  const __half *__restrict__ zeros, __half *__restrict__ W_out,
                  int K, int N, int group)
{
    const int n = blockIdx.x * kDequantThreads + threadIdx.x;
    if (n >= N) return;
    for (int r = blockIdx.y; r < K / 8; r += gridDim.y) {   // rows k = 8r .. 8r+7
    const int j = (8 * r) / group;
    const uint32_t word = packed[(size_t)r * N + n];
    const __half s = scales[(size_t)j * N + n];
    const __half z = zeros[(size_t)j * N + n];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __half q = __int2half_rn((int)((word >> (4 * i)) & 15u));
        W_out[(size_t)(8 * r + i) * N + n] = __hmul(__hsub(q, z), s);
    }
    }
}

// ---------------------------------------------------------------- bfloat16
// double -> bfloat16, round to nearest even, in one rounding: first to float
// with round-to-odd (round toward zero, then set the last bit if anything was
// cut off), then float -> bfloat16 to nearest even.  An intermediate format
// with at least two more bits than the target, rounded to odd, makes the
// second rounding equal the direct one (S. Boldo and G. Melquiond, "When
// double rounding is odd", 2005); float has 16 more bits than bfloat16 at
// every exponent, subnormals included.
__device__ __forceinline__ __nv_bfloat16 f64_to_bf16_rn(double v) {
    float f = __double2float_rz(v);
    if ((double)f != v) f = __uint_as_float(__float_as_uint(f) | 1u);
    return __float2bfloat16_rn(f);
}

// The asymmetric recipe of quantize_pack_kernel with bfloat16 weights, scales
// and zeros: s = bf16((max - min) / 15) from the fp64 quotient, z and q from
// fp64 quotients by the rounded s.
__global__ void __launch_bounds__(kQuantThreads)
quantize_pack_bf16_kernel(const __nv_bfloat16 *__restrict__ W, int K, int N, int group,
                          uint32_t *__restrict__ packed, __nv_bfloat16 *__restrict__ scales,
                          __nv_bfloat16 *__restrict__ zeros)
{
    const int n = blockIdx.x * kQuantThreads + threadIdx.x;
    if (n >= N) return;
    for (int j = blockIdx.y; j < K / group; j += gridDim.y) {
        const size_t k0 = (size_t)j * group;
        float mn = __int_as_float(0x7f800000);
        float mx = -mn;
        for (int k = 0; k < group; ++k) {
            const float v = __bfloat162float(W[(k0 + k) * N + n]);   // exact
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
        }
        __nv_bfloat16 sb = f64_to_bf16_rn(((double)mx - (double)mn) / 15.0);
        double s = (double)__bfloat162float(sb);
        if (s == 0.0) {                                 // degenerate group
            sb = __float2bfloat16_rn(1.0f);
            s = 1.0;
        }
        double zr = rint(-(double)mn / s);
        zr = fmin(fmax(zr, 0.0), 15.0);
        const int z = (int)zr;
        scales[(size_t)j * N + n] = sb;
        zeros[(size_t)j * N + n] = __float2bfloat16_rn((float)z);   // exact
        for (int r = 0; r < group / 8; ++r) {
            uint32_t word = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const double v = (double)__bfloat162float(W[(k0 + 8 * r + i) * N + n]);
                double qd = rint(v / s) + (double)z;
                qd = fmin(fmax(qd, 0.0), 15.0);
                word |= (uint32_t)qd << (4 * i);
            }
            packed[(k0 / 8 + r) * N + n] = word;
        }
    }
}

// W_out[k,n] = bf16((q - z) * s): (q - z) * s is exact in fp32 (a 4-bit
// integer times an 8-bit significand), so one float -> bfloat16 rounding is
// the rounding of the exact product.
__global__ void __launch_bounds__(kDequantThreads)
dequantize_bf16_kernel(const uint32_t *__restrict__ packed, const __nv_bfloat16 *__restrict__ scales,
                       const __nv_bfloat16 *__restrict__ zeros, __nv_bfloat16 *__restrict__ W_out,
                       int K, int N, int group)
{
    const int n = blockIdx.x * kDequantThreads + threadIdx.x;
    if (n >= N) return;
    for (int r = blockIdx.y; r < K / 8; r += gridDim.y) {
        const int j = (8 * r) / group;
        const uint32_t word = packed[(size_t)r * N + n];
        const float s = __bfloat162float(scales[(size_t)j * N + n]);
        const float z = __bfloat162float(zeros[(size_t)j * N + n]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float q = (float)((word >> (4 * i)) & 15u);
            W_out[(size_t)(8 * r + i) * N + n] = __float2bfloat16_rn((q - z) * s);
        }
    }
}

// Repack (the pre-permuted layout; page "Beating FP16 with 4-bit Weights",
// section "What's next": permute the packed weights offline into the order the
// MMA consumes them).  One CTA per block (32-column strip sn, 256-row block
// kb): block words u8 * 128 + L * 4 + c take packed row 32 kb + 4 u8 + L % 4,
// column 32 sn + 4 (L / 4) + c, with the nibbles reordered so that nibble p
// holds natural nibble 2 (p % 4) + p / 4; then the block's scales and zeros,
// 16 bytes per (group row gi, 4-column group g): four scales, four zeros.
__device__ __forceinline__ uint32_t repack_nibbles(uint32_t w) {
    uint32_t r = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) r |= ((w >> (4 * (2 * (p % 4) + p / 4))) & 15u) << (4 * p);
    return r;
}

__global__ void __launch_bounds__(256)
repack_kernel(const uint32_t *__restrict__ packed, const uint16_t *__restrict__ scales,
              const uint16_t *__restrict__ zeros, int K, int N, int group, int gps,
              uint32_t *__restrict__ out)
{
    const int KB = K >> 8;
    const int sn = blockIdx.x / KB, kb = blockIdx.x - sn * KB;
    uint32_t *blk = out + (size_t)blockIdx.x * (1024 + 32 * gps);
    const int u8 = threadIdx.x >> 5, L = threadIdx.x & 31;
    const int r = 32 * kb + 4 * u8 + (L & 3);
    const int n0 = 32 * sn + 4 * (L >> 2);
    const uint4 v = *reinterpret_cast<const uint4 *>(packed + (size_t)r * N + n0);
    *reinterpret_cast<uint4 *>(blk + u8 * 128 + L * 4) =
        make_uint4(repack_nibbles(v.x), repack_nibbles(v.y), repack_nibbles(v.z),
                   repack_nibbles(v.w));
    if (threadIdx.x < gps * 8) {
        const int gi = threadIdx.x >> 3, g = threadIdx.x & 7;
        const int j = (256 * kb) / group + gi;
        const size_t src = (size_t)j * N + 32 * sn + 4 * g;
        const uint2 sv = *reinterpret_cast<const uint2 *>(scales + src);
        const uint2 zv = *reinterpret_cast<const uint2 *>(zeros + src);
        *reinterpret_cast<uint4 *>(blk + 1024 + 4 * threadIdx.x) = make_uint4(sv.x, sv.y, zv.x, zv.y);
    }
}

}  // namespace

cudaError_t launch_quantize_pack(const uint16_t *W, int K, int N, int group, bool symmetric,
                                 uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                 cudaStream_t stream)
{
    dim3 grid((N + kQuantThreads - 1) / kQuantThreads, K / group < 65535 ? K / group : 65535);
    quantize_pack_kernel<<<grid, kQuantThreads, 0, stream>>>(
        reinterpret_cast<const __half *>(W), K, N, group, symmetric, packed,
        reinterpret_cast<__half *>(scales), reinterpret_cast<__half *>(zeros));
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint32_t *packed, const uint16_t *scales,
                              const uint16_t *zeros, uint16_t *W_out, int K, int N,
                              int group, cudaStream_t stream)
{
    dim3 grid((N + kDequantThreads - 1) / kDequantThreads, K / 8 < 65535 ? K / 8 : 65535);
    dequantize_kernel<<<grid, kDequantThreads, 0, stream>>>(
        packed, reinterpret_cast<const __half *>(scales),
        reinterpret_cast<const __half *>(zeros), reinterpret_cast<__half *>(W_out), K, N,
        group);
    return cudaGetLastError();
}

cudaError_t launch_quantize_pack_bf16(const uint16_t *W, int K, int N, int group,
                                      uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                      cudaStream_t stream)
{
    dim3 grid((N + kQuantThreads - 1) / kQuantThreads, K / group < 65535 ? K / group : 65535);
    quantize_pack_bf16_kernel<<<grid, kQuantThreads, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16 *>(W), K, N, group, packed,
        reinterpret_cast<__nv_bfloat16 *>(scales), reinterpret_cast<__nv_bfloat16 *>(zeros));
    return cudaGetLastError();
}

cudaError_t launch_dequantize_bf16(const uint32_t *packed, const uint16_t *scales,
                                   const uint16_t *zeros, uint16_t *W_out, int K, int N,
                                   int group, cudaStream_t stream)
{
    dim3 grid((N + kDequantThreads - 1) / kDequantThreads, K / 8 < 65535 ? K / 8 : 65535);
    dequantize_bf16_kernel<<<grid, kDequantThreads, 0, stream>>>(
        packed, reinterpret_cast<const __nv_bfloat16 *>(scales),
        reinterpret_cast<const __nv_bfloat16 *>(zeros), reinterpret_cast<__nv_bfloat16 *>(W_out),
        K, N, group);
    return cudaGetLastError();
}

bool repack_supported(int K, int N, int group) {
    if (K <= 0 || N <= 0 || K % 256 != 0 || N % 32 != 0 || group % 32 != 0 || K % group != 0)
        return false;
    return group < 256 ? 256 % group == 0 : group % 256 == 0;
}

size_t repacked_bytes(int K, int N, int group) {
    if (!repack_supported(K, N, group)) return 0;
    const int gps = group < 256 ? 256 / group : 1;
    return (size_t)(N / 32) * (K / 256) * (4096 + 128 * gps);
}

cudaError_t launch_repack(const uint32_t *packed, const uint16_t *scales, const uint16_t *zeros,
                          int K, int N, int group, void *out, cudaStream_t stream) {
    if (!repack_supported(K, N, group)) return cudaErrorNotSupported;
    const int gps = group < 256 ? 256 / group : 1;
    const long long blocks = (long long)(N / 32) * (K / 256);
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    repack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(packed, scales, zeros, K, N, group, gps,
                                                          static_cast<uint32_t *>(out));
    return cudaGetLastError();
}

}  // namespace w4a16
