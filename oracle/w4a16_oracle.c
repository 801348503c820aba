/*
 * w4a16_oracle.c -- plain, slow, fp64 CPU oracle for the W4A16 weight-only GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header or constant table with the
 * CUDA library; it is written from the method's description alone.
 *
 * What it computes (sources are the three pages on the subject):
 *   - "Beating FP16 with 4-bit Weights: A Portable W4A16 GEMM in Triton",
 *     section "The design": weights are quantized to 4 bits with one scale and
 *     one zero-point per group of 128 rows along the contraction dimension,
 *     eight 4-bit values packed into one int32 along K, row 8*i+j of the
 *     unpacked tile being K = 8*i+j; dequantization is (w - zero) * scale and
 *     the product accumulates in fp32.
 *   - GemLite README, usage section: the HQQ form (W_q - zeros) * scales ~= W.
 *   - The task's stated recipe for the quantizer: asymmetric min/max per
 *     (group, column), scale = (max - min)/15, zero = round(-min/scale),
 *     q in [0, 15], nibble for k at bits 4*(k % 8).
 *
 * Readings taken where the pages are silent (each is listed with its reason in
 * the design notes of the repository):
 *   - "round" is round-half-to-even (C rint in the default rounding mode).
 *   - The scale is computed in fp64 and rounded ONCE to binary16; zero and
 *     codes are computed from the ROUNDED scale, in fp64:
 *        z = clamp(rint(-min / s), 0, 15),  q = clamp(rint(w / s) + z, 0, 15).
 *   - A group whose rounded scale is 0 (max == min) uses s = 1.0.
 *   - The dequantized weight is binary16(round((q - z) * s)); (q - z) * s is
 *     exact in fp64, so this is a single rounding.
 *   - The GEMM reference is sum_k x[m,k] * Wdq[k,n] in fp64, ascending k.
 *
 * binary16 <-> fp64 conversion is written here from the IEEE 754 binary16
 * definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits,
 * subnormals with quantum 2^-24), not taken from any library.
 *
 * Every entry point returns 0 on success and a negative value on a bad
 * argument.  Arrays are row-major; fp16 values travel as their 16-bit
 * patterns.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- binary16 */

/* Exact value of a binary16 bit pattern. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* zero or subnormal */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1.frac) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even. */
uint16_t oracle_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7e00);
    /* 65504 is the largest finite value; 65520 is the midpoint to 2^16 and
       ties to the even neighbour 2^16, i.e. overflows. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: multiples of 2^-24; a result of 1024 is the
           smallest normal and encodes correctly as 0x0400 */
        double q = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e;
    double f = frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;                        /* a = (2f) * 2^E, 2f in [1, 2) */
    double m = rint(ldexp(f, 11));        /* 11 significant bits: [1024, 2048] */
    /* m == 2048 carries into the exponent, which the sum below absorbs */
    uint32_t bits = (uint32_t)((E + 15) << 10) + (uint32_t)(m - 1024.0);
    return (uint16_t)(sign | bits);
}

/* ---------------------------------------------------------- quantize/pack */

static int check_shape(int K, int N, int group)
{
    if (K <= 0 || N <= 0 || group <= 0) return -1;
    if (group % 8 != 0) return -2;
    if (K % group != 0) return -3;
    return 0;
}

/*
 * Quantize W [K,N] (binary16 patterns) group-wise and pack the codes.
 *   packed [K/8, N] : nibble for row k at bits 4*(k%8) of word (k/8, n)
 *   scales [K/g, N] : binary16 scale s
 *   zeros  [K/g, N] : binary16 zero z (an integer in [0, 15])
 * Optionally also returns the codes q [K,N] (one byte each) when q != NULL.
 */
int oracle_quantize_pack(const uint16_t *W, int K, int N, int group,
                         uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                         uint8_t *q_out)
{
    int rc = check_shape(K, N, group);
    if (rc) return rc;
    int G = K / group;
    memset(packed, 0, sizeof(uint32_t) * (size_t)(K / 8) * (size_t)N);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int j = 0; j < G; ++j) {
            double mn = INFINITY, mx = -INFINITY;
            for (int k = j * group; k < (j + 1) * group; ++k) {
                double w = oracle_half_to_double(W[(size_t)k * N + n]);
                if (w < mn) mn = w;
                if (w > mx) mx = w;
            }
            uint16_t s_bits = oracle_double_to_half((mx - mn) / 15.0);
            double s = oracle_half_to_double(s_bits);
            if (s == 0.0) {          /* degenerate group: max == min */
                s_bits = 0x3c00;     /* 1.0 */
                s = 1.0;
            }
            double zr = rint(-mn / s);
            if (zr < 0.0) zr = 0.0;
            if (zr > 15.0) zr = 15.0;
            int z = (int)zr;
            scales[(size_t)j * N + n] = s_bits;
            zeros[(size_t)j * N + n] = oracle_double_to_half((double)z);
            for (int k = j * group; k < (j + 1) * group; ++k) {
                double w = oracle_half_to_double(W[(size_t)k * N + n]);
                double qd = rint(w / s) + (double)z;
                if (qd < 0.0) qd = 0.0;
                if (qd > 15.0) qd = 15.0;
                uint32_t q = (uint32_t)qd;
                packed[(size_t)(k / 8) * N + n] |= q << (4 * (k % 8));
                if (q_out) q_out[(size_t)k * N + n] = (uint8_t)q;
            }
        }
    }
    return 0;
}

/*
 * Symmetric variant (the pages test "symmetric and asymmetric quantization"
 * and name the "+8 zero-point" of the symmetric packing): signed codes
 * c in [-8, 7] stored as q = c + 8, so the zero is 8 and the dequantization
 * (q - z) * s is the same.  Per (group j, column n):
 *   a = max_k |W[k,n]|;  s = binary16(a / 7) (fp64 quotient, one rounding),
 *   s = 1.0 if that rounds to 0;  z = 8;  q = clamp(rint(W / s) + 8, 0, 15).
 */
int oracle_quantize_pack_symmetric(const uint16_t *W, int K, int N, int group,
                                   uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                                   uint8_t *q_out)
{
    int rc = check_shape(K, N, group);
    if (rc) return rc;
    int G = K / group;
    memset(packed, 0, sizeof(uint32_t) * (size_t)(K / 8) * (size_t)N);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int j = 0; j < G; ++j) {
            double a = 0.0;
            for (int k = j * group; k < (j + 1) * group; ++k) {
                double w = fabs(oracle_half_to_double(W[(size_t)k * N + n]));
                if (w > a) a = w;
            }
            uint16_t s_bits = oracle_double_to_half(a / 7.0);
            double s = oracle_half_to_double(s_bits);
            if (s == 0.0) {          /* all-zero group */
                s_bits = 0x3c00;
                s = 1.0;
            }
            scales[(size_t)j * N + n] = s_bits;
            zeros[(size_t)j * N + n] = oracle_double_to_half(8.0);
            for (int k = j * group; k < (j + 1) * group; ++k) {
                double w = oracle_half_to_double(W[(size_t)k * N + n]);
                double cd = rint(w / s) + 8.0;        /* signed code + 8 */
                cd = cd < 0.0 ? 0.0 : (cd > 15.0 ? 15.0 : cd);
                uint32_t code = (uint32_t)cd;
                packed[(size_t)(k / 8) * N + n] |= code << (4 * (k % 8));
                if (q_out) q_out[(size_t)k * N + n] = (uint8_t)code;
            }
        }
    }
    return 0;
}

/* Codes back out of the packed words: q[k,n] = (packed[k/8,n] >> 4*(k%8)) & 15. */
int oracle_unpack(const uint32_t *packed, int K, int N, uint8_t *q)
{
    if (K <= 0 || N <= 0 || K % 8 != 0) return -1;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n)
            q[(size_t)k * N + n] =
                (uint8_t)((packed[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 15u);
    return 0;
}

/* Wdq[k,n] = binary16((q - z) * s), one rounding of an exact product. */
int oracle_dequant(const uint32_t *packed, const uint16_t *scales,
                   const uint16_t *zeros, int K, int N, int group, uint16_t *Wdq)
{
    int rc = check_shape(K, N, group);
    if (rc) return rc;
#pragma omp parallel for schedule(static)
    for (int k = 0; k < K; ++k) {
        int j = k / group;
        for (int n = 0; n < N; ++n) {
            double q = (double)((packed[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 15u);
            double s = oracle_half_to_double(scales[(size_t)j * N + n]);
            double z = oracle_half_to_double(zeros[(size_t)j * N + n]);
            Wdq[(size_t)k * N + n] = oracle_double_to_half((q - z) * s);
        }
    }
    return 0;
}

/*
 * ref[m,n] = sum_k x[m,k] * Wdq[k,n], fp64, ascending k.
 * The weight is dequantized first (v1 of the "Three Kernel Versions" section of
 * "Triton Kernel Matches bitsandbytes": dequantize, then a plain matmul), then
 * each output is one fp64 dot product.
 */
int oracle_gemm(const uint16_t *x, const uint32_t *packed, const uint16_t *scales,
                const uint16_t *zeros, int M, int N, int K, int group, double *ref)
{
    int rc = check_shape(K, N, group);
    if (rc) return rc;
    if (M < 0) return -4;
    if (M == 0) return 0;
    uint16_t *Wdq = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)K * (size_t)N);
    double *WT = (double *)malloc(sizeof(double) * (size_t)K * (size_t)N);
    double *xd = (double *)malloc(sizeof(double) * (size_t)M * (size_t)K);
    if (!Wdq || !WT || !xd) {
        free(Wdq); free(WT); free(xd);
        return -5;
    }
    oracle_dequant(packed, scales, zeros, K, N, group, Wdq);
    /* column n of Wdq as a contiguous fp64 row, for a cache-friendly dot */
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            WT[(size_t)n * K + k] = oracle_half_to_double(Wdq[(size_t)k * N + n]);
    for (size_t i = 0; i < (size_t)M * K; ++i) xd[i] = oracle_half_to_double(x[i]);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const double *w = WT + (size_t)n * K;
        for (int m = 0; m < M; ++m) {
            const double *xm = xd + (size_t)m * K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += xm[k] * w[k];
            ref[(size_t)m * N + n] = acc;
        }
    }
    free(Wdq); free(WT); free(xd);
    return 0;
}

/* ---------------------------------------------------------------- bfloat16
 *
 * The bf16 variant ("Beating FP16 with 4-bit Weights", section "What's next",
 * names variants beyond fp16 activations; the GemLite README's usage section
 * takes the model dtype, fp16 or bf16, for the activations, scales and zeros).
 * The pages give no bf16 recipe; the reading taken here keeps every step of
 * the fp16 recipe and replaces binary16 by bfloat16 wherever a value is stored:
 * weights, scales, zeros, activations and outputs are bfloat16, the codes and
 * their packing are unchanged, and the dequantized weight is one bfloat16
 * rounding of the exact (q - z) * s.
 *
 * bfloat16: 1 sign bit, 8 exponent bits with bias 127, 7 fraction bits,
 * subnormals with quantum 2^-133 -- written here from that definition.
 */
double oracle_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133);                /* zero or subnormal */
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + frac), expo - 134);  /* (1.frac) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16, ties to even. */
uint16_t oracle_double_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(sign | 0x7fc0);
    /* (2 - 2^-7) * 2^127 is the largest finite value; the midpoint to 2^128,
       (2 - 2^-8) * 2^127, ties to the even neighbour 2^128: overflow */
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127)) return (uint16_t)(sign | 0x7f80);
    if (a < ldexp(1.0, -126)) {
        /* subnormal range: multiples of 2^-133; 128 encodes the smallest normal */
        double q = rint(ldexp(a, 133));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e;
    double f = frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;
    double m = rint(ldexp(f, 8));         /* 8 significant bits: [128, 256] */
    uint32_t bits = (uint32_t)((E + 127) << 7) + (uint32_t)(m - 128.0);
    return (uint16_t)(sign | bits);
}

/* The asymmetric quantizer of oracle_quantize_pack with bfloat16 weights,
 * scales and zeros: s = bf16((max - min) / 15) (fp64 quotient, one rounding;
 * 1.0 if that rounds to 0), z = clamp(rint(-min / s), 0, 15),
 * q = clamp(rint(w / s) + z, 0, 15), codes packed as before. */
int oracle_quantize_pack_bf16(const uint16_t *W, int K, int N, int group,
                              uint32_t *packed, uint16_t *scales, uint16_t *zeros,
                              uint8_t *q_out)
{
    int rc = check_shape(K, N, group);
    if (rc) return rc;
    int G = K / group;
    memset(packed, 0, sizeof(uint32_t) * (size_t)(K / 8) * (size_t)N);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int j = 0; j < G; ++j) {
            double mn = INFINITY, mx = -INFINITY;
            for (int k = j * group; k < (j + 1) * group; ++k) {
                double w = oracle_bf16_to_double(W[(size_t)k * N + n]);
                if (w < mn) mn = w;
                if (w > mx) mx = w;
            }
            uint16_t s_bits = oracle_double_to_bf16((mx - mn) / 15.0);
            double s = oracle_bf16_to_double(s_bits);
            if (s == 0.0) {          /* degenerate group: max == min */
                s_bits = 0x3f80;     /* 1.0 */
                s = 1.0;
            }
            double zq = rint(-mn / s);
            zq = zq < 0.0 ? 0.0 : (zq > 15.0 ? 15.0 : zq);
            int z = (int)zq;
            scales[(size_t)j * N + n] = s_bits;
            zeros[(size_t)j * N + n] = oracle_double_to_bf16((double)z);
            for (int k = j * group; k < (j + 1) * group; ++k) {
                double w = oracle_bf16_to_double(W[(size_t)k * N + n]);
                double qv = rint(w / s) + (double)z;
                qv = qv < 0.0 ? 0.0 : (qv > 15.0 ? 15.0 : qv);
                uint32_t q = (uint32_t)qv;
                packed[(size_t)(k / 8) * N + n] |= q << (4 * (k & 7));
                if (q_out) q_out[(size_t)k * N + n] = (uint8_t)q;
            }
        }
    }
    return 0;
}

/* Wdq[k,n] = bfloat16((q - z) * s), one rounding of an exact product. */
int oracle_dequant_bf16(const uint32_t *packed, const uint16_t *scales,
                        const uint16_t *zeros, int K, int N, int group, uint16_t *Wdq)
{
    int rc = check_shape(K, N, group);
    if (rc) return rc;
#pragma omp parallel for schedule(static)
    for (int k = 0; k < K; ++k) {
        int j = k / group;
        for (int n = 0; n < N; ++n) {
            double q = (double)((packed[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 15u);
            double s = oracle_bf16_to_double(scales[(size_t)j * N + n]);
            double z = oracle_bf16_to_double(zeros[(size_t)j * N + n]);
            Wdq[(size_t)k * N + n] = oracle_double_to_bf16((q - z) * s);
        }
    }
    return 0;
}

/* ref[m,n] = sum_k x[m,k] * Wdq[k,n] in fp64, ascending k, with bfloat16 x and
 * the bfloat16 dequantized weight. */
int oracle_gemm_bf16(const uint16_t *x, const uint32_t *packed, const uint16_t *scales,
                     const uint16_t *zeros, int M, int N, int K, int group, double *ref)
{
    int rc = check_shape(K, N, group);
    if (rc) return rc;
    if (M < 0) return -4;
    if (M == 0) return 0;
    uint16_t *Wdq = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)K * (size_t)N);
    double *WT = (double *)malloc(sizeof(double) * (size_t)K * (size_t)N);
    double *xd = (double *)malloc(sizeof(double) * (size_t)M * (size_t)K);
    if (!Wdq || !WT || !xd) {
        free(Wdq); free(WT); free(xd);
        return -5;
    }
    oracle_dequant_bf16(packed, scales, zeros, K, N, group, Wdq);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            WT[(size_t)n * K + k] = oracle_bf16_to_double(Wdq[(size_t)k * N + n]);
    for (size_t i = 0; i < (size_t)M * K; ++i) xd[i] = oracle_bf16_to_double(x[i]);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const double *w = WT + (size_t)n * K;
        for (int m = 0; m < M; ++m) {
            const double *xm = xd + (size_t)m * K;
            double sum = 0.0;
            for (int k = 0; k < K; ++k) sum += xm[k] * w[k];
            ref[(size_t)m * N + n] = sum;
        }
    }
    free(Wdq); free(WT); free(xd);
    return 0;
}

/* --------------------------------------------------- pre-permuted layout
 *
 * "Beating FP16 with 4-bit Weights", section "What's next": permute the packed
 * weights offline so that they reach the tensor cores in the order the MMA
 * consumes them, and pipeline the loads with asynchronous copies; "Triton
 * Kernel Matches bitsandbytes", section "Why Marlin Is Still Faster" credits
 * the same offline reordering.  The pages give no byte layout; this library's
 * layout (the repacked form) is defined here, as a plain index map:
 *
 *   requirements: K % 256 == 0, N % 32 == 0, and either group divides 256 or
 *   256 divides group (group a multiple of 32).
 *   gps = 256 / group if group < 256, else 1   (group rows stored per block)
 *   block (sn, kb), sn = 32-column strip in [0, N/32), kb = 256-row block of K
 *   in [0, K/256), starts at 32-bit word  (sn * (K/256) + kb) * BW,
 *   BW = 1024 + 32 * gps words (4096 + 128 * gps bytes).
 *   Word i = u8 * 128 + L * 4 + c of a block (u8 in 0..7, L in 0..31, c in 0..3)
 *   holds the codes of packed row  r = 32 * kb + 4 * u8 + (L % 4)  and column
 *   n = 32 * sn + 4 * (L / 4) + c, with its nibbles reordered: nibble p of the
 *   repacked word is nibble 2 * (p % 4) + p / 4 of the natural word (so the
 *   nibble pairs (0,4), (1,5), (2,6), (3,7) hold the codes of k = 8r + (0,1),
 *   (2,3), (4,5), (6,7)).
 *   After the 1024 words, the block's scales and zeros as binary16 values:
 *   half index  h = (gi * 8 + g) * 8 + c  (scale) and  h + 4  (zero), for
 *   gi in 0..gps-1, g in 0..7, c in 0..3, of group row  256 * kb / group + gi
 *   and column  32 * sn + 4 * g + c.
 */
static int check_permuted_shape(int K, int N, int group)
{
    if (K <= 0 || N <= 0 || K % 256 != 0 || N % 32 != 0) return -1;
    if (group <= 0 || group % 32 != 0 || K % group != 0) return -2;
    if (group < 256 ? (256 % group != 0) : (group % 256 != 0)) return -2;
    return 0;
}

static int permuted_gps(int group) { return group < 256 ? 256 / group : 1; }

/* nibble p of the result = nibble 2*(p%4) + p/4 of w */
static uint32_t permute_nibbles(uint32_t w)
{
    uint32_t r = 0;
    for (int p = 0; p < 8; ++p) {
        uint32_t src = (uint32_t)(2 * (p % 4) + p / 4);
        r |= ((w >> (4 * src)) & 15u) << (4 * p);
    }
    return r;
}

static uint32_t unpermute_nibbles(uint32_t w)
{
    uint32_t r = 0;
    for (int p = 0; p < 8; ++p) {
        uint32_t dst = (uint32_t)(2 * (p % 4) + p / 4);
        r |= ((w >> (4 * p)) & 15u) << (4 * dst);
    }
    return r;
}

/* Number of 32-bit words of the repacked form (0 for an unsupported shape). */
long long oracle_permuted_words(int K, int N, int group)
{
    if (check_permuted_shape(K, N, group)) return 0;
    return (long long)(N / 32) * (K / 256) * (1024 + 32 * permuted_gps(group));
}

/* natural (packed [K/8,N], scales/zeros [K/g,N]) -> repacked words */
int oracle_permute(const uint32_t *packed, const uint16_t *scales, const uint16_t *zeros,
                   int K, int N, int group, uint32_t *out)
{
    int rc = check_permuted_shape(K, N, group);
    if (rc) return rc;
    const int gps = permuted_gps(group), KB = K / 256;
    const long long BW = 1024 + 32 * gps;
    for (int sn = 0; sn < N / 32; ++sn)
        for (int kb = 0; kb < KB; ++kb) {
            uint32_t *blk = out + ((long long)sn * KB + kb) * BW;
            for (int u8 = 0; u8 < 8; ++u8)
                for (int L = 0; L < 32; ++L)
                    for (int c = 0; c < 4; ++c) {
                        int r = 32 * kb + 4 * u8 + L % 4;
                        int n = 32 * sn + 4 * (L / 4) + c;
                        blk[u8 * 128 + L * 4 + c] = permute_nibbles(packed[(size_t)r * N + n]);
                    }
            uint16_t *sz = (uint16_t *)(blk + 1024);
            for (int gi = 0; gi < gps; ++gi)
                for (int g = 0; g < 8; ++g)
                    for (int c = 0; c < 4; ++c) {
                        int j = 256 * kb / group + gi;
                        int n = 32 * sn + 4 * g + c;
                        int h = (gi * 8 + g) * 8 + c;
                        sz[h] = scales[(size_t)j * N + n];
                        sz[h + 4] = zeros[(size_t)j * N + n];
                    }
        }
    return 0;
}

/* repacked words -> natural (packed, scales, zeros): the inverse map */
int oracle_unpermute(const uint32_t *in, int K, int N, int group, uint32_t *packed,
                     uint16_t *scales, uint16_t *zeros)
{
    int rc = check_permuted_shape(K, N, group);
    if (rc) return rc;
    const int gps = permuted_gps(group), KB = K / 256;
    const long long BW = 1024 + 32 * gps;
    for (int sn = 0; sn < N / 32; ++sn)
        for (int kb = 0; kb < KB; ++kb) {
            const uint32_t *blk = in + ((long long)sn * KB + kb) * BW;
            for (int u8 = 0; u8 < 8; ++u8)
                for (int L = 0; L < 32; ++L)
                    for (int c = 0; c < 4; ++c) {
                        int r = 32 * kb + 4 * u8 + L % 4;
                        int n = 32 * sn + 4 * (L / 4) + c;
                        packed[(size_t)r * N + n] = unpermute_nibbles(blk[u8 * 128 + L * 4 + c]);
                    }
            const uint16_t *sz = (const uint16_t *)(blk + 1024);
            for (int gi = 0; gi < gps; ++gi)
                for (int g = 0; g < 8; ++g)
                    for (int c = 0; c < 4; ++c) {
                        int j = 256 * kb / group + gi;
                        int n = 32 * sn + 4 * g + c;
                        int h = (gi * 8 + g) * 8 + c;
                        scales[(size_t)j * N + n] = sz[h];
                        zeros[(size_t)j * N + n] = sz[h + 4];
                    }
        }
    return 0;
}

/* Threads the OpenMP loops above run on (1 when built without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
