// decode_math.cuh -- the per-step arithmetic shared by the decode kernels:
// nibble unpack with the magic-exponent trick, exact (q - z) in fp16, and the
// register-fed tensor-core MMA with swapped roles.
//
// Fragment mapping (mma.m16n8k16, A row-major 16x16, B col 16x8, fp32 C):
//   thread (g = lane/4, t = lane%4) holds one 128-bit load: the packed words of
//   four neighbouring columns c0..c0+3 for one packed row (8 consecutive k).
//   MMA tile j (j = 0, 1): A row g <- column c0+2j, A row g+8 <- column c0+2j+1.
//   K slots (2t, 2t+1, 2t+8, 2t+9) take nibbles (0, 4, 1, 5) for kk = 0 and
//   (2, 6, 3, 7) for kk = 1 of the thread's word, so every A register is one
//   LOP3 + one HSUB2 away from the word, and the thread's x fragment is
//   x[m][k0 + {0,4 | 1,5}] (kk = 0) and x[m][k0 + {2,6 | 3,7}] (kk = 1): a
//   16-byte load of x[m][k0 .. k0+7] and four byte permutes.  K may be permuted
//   inside a reduction as long as x and W use the same permutation.
//   Accumulator: c0, c1 -> (column c0+2j, batch rows 2t, 2t+1); c2, c3 ->
//   (column c0+2j+1, batch rows 2t, 2t+1).
#pragma once

#include "common.cuh"

namespace w4a16 {

constexpr uint32_t kMaskLo = 0x000F000Fu;   // nibbles 0 and 4 of a word
constexpr uint32_t kMaskHi = 0x00F000F0u;   // nibbles 1 and 5
constexpr uint32_t kMagicLo = 0x64006400u;  // 1024.0 | 1024.0: mantissa ulp 1 at bits 0..3
constexpr uint32_t kMagicHi = 0x54005400u;  // 64.0 | 64.0: mantissa ulp 1 at bits 4..7

// D += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Per-group constants of the thread's four columns: the zero biases
// (1024+z, 64+z) broadcast into both halves, and the fp32 scales.
struct GroupConsts {
    uint32_t zA[4], zB[4];
    float sc[4];
};

// zraw / sraw: the fp16 zeros / scales of columns c0..c0+3 (two per word).
__device__ __forceinline__ GroupConsts make_group_consts(uint2 zraw, uint2 sraw) {
    GroupConsts k;
    const uint32_t zlo01 = hadd2_u32(zraw.x, kMagicLo);   // (1024+z0, 1024+z1), exact
    const uint32_t zlo23 = hadd2_u32(zraw.y, kMagicLo);
    const uint32_t zhi01 = hadd2_u32(zraw.x, kMagicHi);   // (64+z0, 64+z1), exact
    const uint32_t zhi23 = hadd2_u32(zraw.y, kMagicHi);
    k.zA[0] = __byte_perm(zlo01, 0, 0x1010);
    k.zA[1] = __byte_perm(zlo01, 0, 0x3232);
    k.zA[2] = __byte_perm(zlo23, 0, 0x1010);
    k.zA[3] = __byte_perm(zlo23, 0, 0x3232);
    k.zB[0] = __byte_perm(zhi01, 0, 0x1010);
    k.zB[1] = __byte_perm(zhi01, 0, 0x3232);
    k.zB[2] = __byte_perm(zhi23, 0, 0x1010);
    k.zB[3] = __byte_perm(zhi23, 0, 0x3232);
    const __half2 s01 = *reinterpret_cast<const __half2 *>(&sraw.x);
    const __half2 s23 = *reinterpret_cast<const __half2 *>(&sraw.y);
    k.sc[0] = __low2float(s01);
    k.sc[1] = __high2float(s01);
    k.sc[2] = __low2float(s23);
    k.sc[3] = __high2float(s23);
    return k;
}

// x[m][k0..k0+7] (natural order, 4 words) -> the two B fragments of kk = 0, 1.
__device__ __forceinline__ void x_fragments(uint4 v, uint32_t (&b)[4]) {
    b[0] = __byte_perm(v.x, v.z, 0x5410);   // (x0, x4)
    b[1] = __byte_perm(v.x, v.z, 0x7632);   // (x1, x5)
    b[2] = __byte_perm(v.y, v.w, 0x5410);   // (x2, x6)
    b[3] = __byte_perm(v.y, v.w, 0x7632);   // (x3, x7)
}

// One 32-k step of one thread: 4 words (columns c0..c0+3) x 8 k, MMAs into the
// group accumulator gacc[p][j][kk] (p = batch tile of 8 rows, j = column pair,
// kk = k half).  The two k halves accumulate separately, so the four MMAs of a
// step are independent and steps that accumulate into the same registers form
// chains only as long as the number of steps.
template <int NT>
__device__ __forceinline__ void step_mma_split(float (&gacc)[NT][2][2][4], uint4 w,
                                               const GroupConsts &k,
                                               const uint32_t (&bx)[NT][4]) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t c0 = wv[2 * j], c1 = wv[2 * j + 1];
        const uint32_t d0 = c0 >> 8, d1 = c1 >> 8;
        const uint32_t a0 = hsub2_u32(lop3_and_or(c0, kMaskLo, kMagicLo), k.zA[2 * j]);
        const uint32_t a1 = hsub2_u32(lop3_and_or(c1, kMaskLo, kMagicLo), k.zA[2 * j + 1]);
        const uint32_t a2 = hsub2_u32(lop3_and_or(c0, kMaskHi, kMagicHi), k.zB[2 * j]);
        const uint32_t a3 = hsub2_u32(lop3_and_or(c1, kMaskHi, kMagicHi), k.zB[2 * j + 1]);
        const uint32_t e0 = hsub2_u32(lop3_and_or(d0, kMaskLo, kMagicLo), k.zA[2 * j]);
        const uint32_t e1 = hsub2_u32(lop3_and_or(d1, kMaskLo, kMagicLo), k.zA[2 * j + 1]);
        const uint32_t e2 = hsub2_u32(lop3_and_or(d0, kMaskHi, kMagicHi), k.zB[2 * j]);
        const uint32_t e3 = hsub2_u32(lop3_and_or(d1, kMaskHi, kMagicHi), k.zB[2 * j + 1]);
#pragma unroll
        for (int p = 0; p < NT; ++p) {
            mma_16816(gacc[p][j][0], a0, a1, a2, a3, bx[p][0], bx[p][1]);
            mma_16816(gacc[p][j][1], e0, e1, e2, e3, bx[p][2], bx[p][3]);
        }
    }
}

// acc += s * (gacc[..][0] + gacc[..][1]) (the group scale, applied once per
// group in fp32), then gacc = 0.
template <int NT>
__device__ __forceinline__ void flush_group_split(float (&acc)[NT][2][4],
                                                  float (&gacc)[NT][2][2][4],
                                                  const GroupConsts &k) {
#pragma unroll
    for (int p = 0; p < NT; ++p)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc[p][j][r] = fmaf(k.sc[2 * j + (r >> 1)], gacc[p][j][0][r] + gacc[p][j][1][r],
                                    acc[p][j][r]);
                gacc[p][j][0][r] = 0.f;
                gacc[p][j][1][r] = 0.f;
            }
}

// D = A * B (+ C): FIRST starts the accumulator from zero inside the MMA.
template <bool FIRST>
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    if (FIRST)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
    else
        mma_16816(d, a0, a1, a2, a3, b0, b1);
}

// ---------------------------------------------------------------- zero-free step
// The zero-free form of a step (M <= 8).  A nibble masked into the low bits of
// an fp16 half with a zero exponent is the exact subnormal q * 2^-24 (bits 0..3)
// or q * 2^-20 (bits 4..7): the codes enter the MMA with no bias to remove.
// The low-position codes of a step go to one MMA (D_lo), the high-position ones
// to another (D_hi), and one more pair of MMAs with an all-ones A operand sums
// the step's x (D_x), so that per group
//     sum_k x (q - z) s = s 2^24 (D_lo + D_hi / 16) - s z D_x,
// with every product exact and no large term to cancel.
constexpr uint32_t kOnes = 0x3C003C00u;       // fp16 (1.0, 1.0)

struct ZfConsts {
    float s24[4], sz[4];      // s * 2^24 and s * z of the thread's four columns
};

__device__ __forceinline__ ZfConsts make_zf_consts(uint2 zraw, uint2 sraw) {
    ZfConsts k;
    const __half2 s01 = *reinterpret_cast<const __half2 *>(&sraw.x);
    const __half2 s23 = *reinterpret_cast<const __half2 *>(&sraw.y);
    const __half2 z01 = *reinterpret_cast<const __half2 *>(&zraw.x);
    const __half2 z23 = *reinterpret_cast<const __half2 *>(&zraw.y);
    const float sv[4] = {__low2float(s01), __high2float(s01), __low2float(s23), __high2float(s23)};
    const float zv[4] = {__low2float(z01), __high2float(z01), __low2float(z23), __high2float(z23)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        k.s24[c] = sv[c] * 16777216.f;
        k.sz[c] = sv[c] * zv[c];
    }
    return k;
}

// One 32-k step, M <= 8: blo / bhi are the x fragments of the low / high
// nibble positions (two registers each).
template <bool FIRST>
__device__ __forceinline__ void zf_step(float (&dlo)[2][4], float (&dhi)[2][4], float (&dx)[4],
                                        uint4 w, const uint32_t (&blo)[2],
                                        const uint32_t (&bhi)[2]) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t c0 = wv[2 * j], c1 = wv[2 * j + 1];
        const uint32_t d0 = c0 >> 8, d1 = c1 >> 8;
        mma_acc<FIRST>(dlo[j], c0 & kMaskLo, c1 & kMaskLo, d0 & kMaskLo, d1 & kMaskLo, blo[0],
                       blo[1]);
        mma_acc<FIRST>(dhi[j], c0 & kMaskHi, c1 & kMaskHi, d0 & kMaskHi, d1 & kMaskHi, bhi[0],
                       bhi[1]);
    }
    mma_acc<FIRST>(dx, kOnes, kOnes, kOnes, kOnes, blo[0], blo[1]);
    mma_16816(dx, kOnes, kOnes, kOnes, kOnes, bhi[0], bhi[1]);
}

// acc += s 2^24 (D_lo + D_hi / 16) - s z D_x for the thread's 8 outputs
// (D_x element r & 1 holds the x sum of batch row 2t + (r & 1)).
__device__ __forceinline__ void zf_flush(float (&acc)[1][2][4], const float (&dlo)[2][4],
                                         const float (&dhi)[2][4], const float (&dx)[4],
                                         const ZfConsts &k) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int c = 2 * j + (r >> 1);
            const float g = fmaf(0.0625f, dhi[j][r], dlo[j][r]);
            acc[0][j][r] = fmaf(-k.sz[c], dx[r & 1], fmaf(k.s24[c], g, acc[0][j][r]));
        }
}

// ---------------------------------------------------------------- bfloat16
// bfloat16 has 7 fraction bits, so only the low nibble of a half fits under
// the magic exponent: 128.0 (0x4300) has its mantissa ulp at bit 0, and
// 0x4300 | q is 128 + q exactly.  The other nibbles are shifted down first
// (w >> 4, w >> 8, w >> 12 bring nibbles (1,5), (2,6), (3,7) to bits 0..3 and
// 16..19), which keeps the fragment mapping above.  Each weight is then
// ((128 + q) - (128 + z)) * s: the difference is exact, the product is one
// bfloat16 rounding of (q - z) * s -- the dequantized bfloat16 weight bit for
// bit, which the MMA multiplies by x exactly (products of two bfloat16 values
// fit fp32) and accumulates in fp32.
constexpr uint32_t kMagicBf = 0x43004300u;   // 128.0 | 128.0 (bfloat16)

__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Per-group constants of the thread's four columns: (128 + z) and the scale,
// each broadcast into both halves of a bfloat16 pair.
struct GroupConstsBf {
    uint32_t zA[4], s2[4];
};

__device__ __forceinline__ GroupConstsBf make_group_consts_bf(uint2 zraw, uint2 sraw) {
    GroupConstsBf k;
    const uint32_t z01 = badd2_u32(zraw.x, kMagicBf);   // (128+z0, 128+z1), exact
    const uint32_t z23 = badd2_u32(zraw.y, kMagicBf);
    k.zA[0] = __byte_perm(z01, 0, 0x1010);
    k.zA[1] = __byte_perm(z01, 0, 0x3232);
    k.zA[2] = __byte_perm(z23, 0, 0x1010);
    k.zA[3] = __byte_perm(z23, 0, 0x3232);
    k.s2[0] = __byte_perm(sraw.x, 0, 0x1010);
    k.s2[1] = __byte_perm(sraw.x, 0, 0x3232);
    k.s2[2] = __byte_perm(sraw.y, 0, 0x1010);
    k.s2[3] = __byte_perm(sraw.y, 0, 0x3232);
    return k;
}

// Two dequantized bfloat16 weights from bits 0..3 and 16..19 of v.
__device__ __forceinline__ uint32_t dq_bf16(uint32_t v, uint32_t zA, uint32_t s2) {
    return bmul2_u32(bsub2_u32(lop3_and_or(v, kMaskLo, kMagicBf), zA), s2);
}

// One 32-k step of one thread, bfloat16: as step_mma_split, with the scale
// already inside each weight, so the MMAs accumulate straight into the
// running sums acc[p][j][kk].
template <int NT>
__device__ __forceinline__ void step_mma_bf16(float (&acc)[NT][2][2][4], uint4 w,
                                              const GroupConstsBf &k,
                                              const uint32_t (&bx)[NT][4]) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t c0 = wv[2 * j], c1 = wv[2 * j + 1];
        const uint32_t z0 = k.zA[2 * j], z1 = k.zA[2 * j + 1];
        const uint32_t s0 = k.s2[2 * j], s1 = k.s2[2 * j + 1];
        const uint32_t a0 = dq_bf16(c0, z0, s0), a1 = dq_bf16(c1, z1, s1);
        const uint32_t a2 = dq_bf16(c0 >> 4, z0, s0), a3 = dq_bf16(c1 >> 4, z1, s1);
        const uint32_t e0 = dq_bf16(c0 >> 8, z0, s0), e1 = dq_bf16(c1 >> 8, z1, s1);
        const uint32_t e2 = dq_bf16(c0 >> 12, z0, s0), e3 = dq_bf16(c1 >> 12, z1, s1);
#pragma unroll
        for (int p = 0; p < NT; ++p) {
            mma_16816_bf16(acc[p][j][0], a0, a1, a2, a3, bx[p][0], bx[p][1]);
            mma_16816_bf16(acc[p][j][1], e0, e1, e2, e3, bx[p][2], bx[p][3]);
        }
    }
}

// fp32 -> the output element (fp16 or bfloat16, round to nearest even).
template <bool BF>
__device__ __forceinline__ uint16_t to_out(float v) {
    if constexpr (BF)
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    else
        return __half_as_ushort(__float2half_rn(v));
}

}  // namespace w4a16
