// quant.cu -- group-wise int4 quantize + pack, and dequantize (test aid).
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

}  // namespace w4a16
