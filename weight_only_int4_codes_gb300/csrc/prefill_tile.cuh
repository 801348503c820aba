// prefill_tile.cuh -- pieces shared by the tcgen05 prefill kernels: the stage
// geometry, the dequantization of a block of packed words into fp16 pairs, and
// the epilogue that reads the accumulator out of tensor memory.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace w4a16 {

constexpr int kTileN = 128;            // weight columns per CTA (one TMEM lane each)
constexpr int kChunkK = 64;            // k per 128-byte swizzle row of fp16
constexpr int kStageK = 128;           // k per pipeline stage (two swizzle chunks)
constexpr int kChunks = kStageK / kChunkK;
constexpr int kPackedRows = kStageK / 8;
constexpr int kDeqWarp0 = 2;           // warps 2.. dequantize and run the epilogue

// Dequantize B consecutive packed words (packed rows c0 .. c0+B-1, column n)
// of a stage held at shared address `st`.  The scale and zero come from row
// `zrow` of the stage's scale/zero rows.  Output: 4B pairs in natural k
// order, h[4c + i] = (w[k0+8c+2i], w[k0+8c+2i+1]).
//
// fp16: pair (q_2i, q_2i+1) comes from byte i of the word: the low half
// becomes 1024 + q_2i (mantissa bits 0..3), the high half 64 + q_2i+1
// (mantissa bits 4..7); minus (1024 + z, 64 + z) is q - z exactly, and times
// the scale is one fp16 rounding of the exact product -- the dequantized
// weight bit for bit.
// bfloat16 (BF): only 7 fraction bits, so both codes sit at bits 0..3 of
// their half -- q_2i from byte i of the word, q_2i+1 from byte i of the word
// shifted right by 4 -- under 128.0 (0x4300); minus (128 + z) is exact, times
// the scale one bfloat16 rounding.
template <int B, bool BF = false>
__device__ __forceinline__ void dequant_words(uint32_t st, int p_off, int s_off, int z_off,
                                              int c0, int zrow, int n, uint32_t (&h)[4 * B]) {
    uint32_t s2, zA;
    {
        uint16_t sb, zb;
        const uint32_t so = st + s_off + zrow * (kTileN * 2) + 2 * n;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(sb) : "r"(so));
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(zb) : "r"(so + (z_off - s_off)));
        s2 = (uint32_t)sb | ((uint32_t)sb << 16);
        // fp16: (1024 + z) in the low half and (64 + z) in the high half;
        // bfloat16: (128 + z) in both
        zA = BF ? badd2_u32((uint32_t)zb | ((uint32_t)zb << 16), 0x43004300u)
                : hadd2_u32((uint32_t)zb | ((uint32_t)zb << 16), 0x54006400u);
    }
    uint32_t wv[B];
#pragma unroll
    for (int cc = 0; cc < B; ++cc)
        asm volatile("ld.shared.u32 %0, [%1];"
                     : "=r"(wv[cc])
                     : "r"(st + p_off + ((c0 + cc) * kTileN + n) * 4));
#pragma unroll
    for (int cc = 0; cc < B; ++cc) {
        if constexpr (BF) {
            const uint32_t hi = wv[cc] >> 4;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // byte i of the word (low half) and of the word >> 4 (high half)
                const uint32_t b = __byte_perm(wv[cc], hi, (uint32_t)(i | ((4 + i) << 8)));
                h[cc * 4 + i] = bmul2_u32(bsub2_u32(lop3_and_or(b, 0x000F000Fu, 0x43004300u), zA), s2);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t b = __byte_perm(wv[cc], 0, 0x4040 + 0x0101 * i);
                h[cc * 4 + i] = hmul2_u32(hsub2_u32(lop3_and_or(b, 0x00F0000Fu, 0x54006400u), zA), s2);
            }
        }
    }
}

// The row of the stage's scale/zero rows that serves packed row c: groups are
// multiples of 64 k, so k0 + 64 is the only place inside a 128-k stage where a
// new group can start.
__device__ __forceinline__ int stage_zrow(int k0, int group, int c) {
    return (c >= kPackedRows / 2 && ((k0 + kChunkK) % group) == 0) ? 1 : 0;
}

// Staged epilogue of one warp: its 32 TMEM lanes (weight columns n = lane
// base + lane, one per thread) for the accumulator columns mc = first, first +
// step, ... (rows of x) become an fp16 (BF: bfloat16) tile [tile_m][128] in
// shared memory at
// `tile` (one 256-byte row per row of x), ready for one TMA store.  With
// nred > 0 the fp32 partial tiles [tile_m][128] at red, red + tile_m * 512,
// ... (the other CTAs of a split-K cluster, in rank order) are added to the
// accumulator first, before the one rounding to fp16.  A warp's stores for
// one row cover 64 contiguous bytes.
template <bool BF = false>
__device__ __forceinline__ void stage_accumulator(uint32_t taddr, uint32_t tile, int n, int tile_m,
                                                  int first, int step, uint32_t red = 0,
                                                  int nred = 0) {
    const uint32_t slot = (uint32_t)tile_m * kTileN * 4;
    for (int mc = first; mc < tile_m; mc += step) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + mc, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (mc + i < tile_m) {
                float acc = __uint_as_float(v[i]);
                const uint32_t e = (uint32_t)((mc + i) * kTileN + n) * 4;
                for (int q = 0; q < nred; ++q) {
                    float p;
                    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(p) : "r"(red + q * slot + e));
                    acc += p;
                }
                const uint16_t h = BF ? __bfloat16_as_ushort(__float2bfloat16_rn(acc))
                                      : __half_as_ushort(__float2half_rn(acc));
                asm volatile("st.shared.u16 [%0], %1;" ::"r"(tile + ((mc + i) * kTileN + n) * 2),
                             "h"(h)
                             : "memory");
            }
    }
}

// The fp32 partial of one warp's accumulator share (as above) as a tile
// [tile_m][128] of floats at `tile`, for a split-K cluster's leader.
__device__ __forceinline__ void stage_partial_f32(uint32_t taddr, uint32_t tile, int n, int tile_m,
                                                  int first, int step) {
    for (int mc = first; mc < tile_m; mc += step) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + mc, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (mc + i < tile_m)
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(tile + ((mc + i) * kTileN + n) * 4),
                             "r"(v[i])
                             : "memory");
    }
}

}  // namespace w4a16
