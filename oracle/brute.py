"""Pure-Python brute force of the W4A16 method -- TEST INFRASTRUCTURE ONLY.

An independent second restatement of the same steps as ``w4a16_oracle.c``, for
tiny shapes only, used to cross-check the C oracle.  It shares nothing with the
C code: binary16 rounding comes from Python's ``struct`` 'e' format (IEEE 754
half, round-half-even), rounding to integers from ``round()`` (half-even), and
the GEMM sum is exact (``fractions.Fraction``).

Steps, as the C oracle (page "Beating FP16 with 4-bit Weights", section "The
design"; GemLite README, usage: (W_q - zeros) * scales ~= W):
  s = fp16((max - min) / 15)   (1.0 if that rounds to 0)
  z = clamp(round(-min / s), 0, 15)
  q = clamp(round(w / s) + z, 0, 15)
  word(k/8, n) holds q(k, n) at bits 4*(k % 8)
  Wdq = fp16((q - z) * s)
  ref = sum_k x[m,k] * Wdq[k,n]   (exact rational sum)
"""
from __future__ import annotations

import struct
from fractions import Fraction


def f16(v: float) -> float:
    """Round a Python float to the nearest binary16 value (ties to even)."""
    return struct.unpack("<e", struct.pack("<e", v))[0]


def f16_bits(v: float) -> int:
    return struct.unpack("<H", struct.pack("<e", v))[0]


def bits_f16(b: int) -> float:
    return struct.unpack("<e", struct.pack("<H", b))[0]


def quantize_pack(W, group):
    """W: list of K rows, each a list of N Python floats (already fp16 values)."""
    K, N = len(W), len(W[0])
    assert K % group == 0 and group % 8 == 0
    packed = [[0] * N for _ in range(K // 8)]
    scales = [[0.0] * N for _ in range(K // group)]
    zeros = [[0.0] * N for _ in range(K // group)]
    codes = [[0] * N for _ in range(K)]
    for n in range(N):
        for j in range(K // group):
            col = [W[k][n] for k in range(j * group, (j + 1) * group)]
            mn, mx = min(col), max(col)
            s = f16((mx - mn) / 15.0)
            if s == 0.0:
                s = 1.0
            z = min(max(round(-mn / s), 0), 15)
            scales[j][n] = s
            zeros[j][n] = float(z)
            for k in range(j * group, (j + 1) * group):
                q = min(max(round(W[k][n] / s) + z, 0), 15)
                codes[k][n] = q
                packed[k // 8][n] |= q << (4 * (k % 8))
    return packed, scales, zeros, codes


def dequant(codes, scales, zeros, group):
    K, N = len(codes), len(codes[0])
    return [[f16((codes[k][n] - zeros[k // group][n]) * scales[k // group][n])
             for n in range(N)] for k in range(K)]


def gemm(x, Wdq):
    """Exact sum of products as a Fraction, returned as a float."""
    M, K, N = len(x), len(x[0]), len(Wdq[0])
    out = [[0.0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(x[m][k]) * Fraction(Wdq[k][n])
            out[m][n] = float(acc)
    return out
