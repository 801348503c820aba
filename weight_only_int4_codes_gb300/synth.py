"""Seeded synthetic inputs for the W4A16 workloads.

This module only draws random numbers: it holds none of the method's
arithmetic (no quantization, packing or GEMM), so both the CUDA path's tests
and the fp64 oracle may take their inputs from it.

Distributions (the workloads the pages measure on: decode-regime dense FFN,
square projections and MoE-expert projections at group 128):
  x ~ N(0, 1)      drawn as float32, rounded to fp16 (or to bfloat16 for the
                   bf16 variant: the same draws, stored as bfloat16)
  W ~ N(0, 0.02)   drawn as float32 (standard deviation 0.02), rounded to fp16
                   (or bfloat16)
  outliers: each W entry independently with probability 0.001 is multiplied
            by 20 (in float32, before the fp16 rounding)

numpy's PCG64 generator is used because its streams are the same on every
platform (the x86 build host and the Arm GPU hosts draw identical inputs).
Seeds: x uses 1000*config + 10*log2(M) (+ 100000*expert), W uses
1000*config + 7 (+ expert).
"""
from __future__ import annotations

import math

import numpy as np

# name -> dict(K, N, Ms, outliers, experts, group)
WORKLOADS = {
    "tiny": dict(config=0, shapes=[(512, 256)], Ms=[1], outliers=False, experts=1),
    "decode_square": dict(config=1, shapes=[(4096, 4096)], Ms=[1, 2, 4, 8, 16],
                          outliers=False, experts=1),
    "decode_ffn": dict(config=2, shapes=[(4096, 14336), (14336, 4096)], Ms=[1, 2, 4, 8, 16],
                       outliers=True, experts=1),
    "moe_experts": dict(config=3, shapes=[(2048, 768), (768, 2048)], Ms=[1, 2, 4, 8, 16],
                        outliers=False, experts=64),
    "prefill_sweep": dict(config=4, shapes=[(4096, 14336), (8192, 28672)],
                          Ms=[16, 32, 64, 128, 256, 1024, 4096], outliers=False, experts=1),
}
GROUP = 128


def weight_seed(config: int, expert: int = 0, shape_index: int = 0) -> int:
    return 1000 * config + 7 + expert + 500 * shape_index


def x_seed(config: int, M: int, expert: int = 0, shape_index: int = 0) -> int:
    return 1000 * config + 10 * int(round(math.log2(max(M, 1)))) + 100000 * expert \
        + 500 * shape_index


def weight(K: int, N: int, seed: int, outliers: bool = False, std: float = 0.02) -> np.ndarray:
    """fp16 [K, N] weight, N(0, std) with optional 0.1% x20 outliers."""
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((K, N), dtype=np.float32)
    w *= np.float32(std)
    if outliers:
        mask = rng.random((K, N), dtype=np.float32) < np.float32(0.001)
        w[mask] *= np.float32(20.0)
    return w.astype(np.float16)


def _draw_weight(K: int, N: int, seed: int, outliers: bool, std: float) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((K, N), dtype=np.float32)
    w *= np.float32(std)
    if outliers:
        mask = rng.random((K, N), dtype=np.float32) < np.float32(0.001)
        w[mask] *= np.float32(20.0)
    return w


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 values -> bfloat16 bit patterns (uint16), round to nearest even
    on the float32 bit pattern (finite inputs; these are the storage format of
    the random draws, numpy having no bfloat16 type)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def weight_bf16(K: int, N: int, seed: int, outliers: bool = False,
                std: float = 0.02) -> np.ndarray:
    """bfloat16 [K, N] weight (bit patterns), the draws of weight() stored as bf16."""
    return bf16_bits(_draw_weight(K, N, seed, outliers, std))


def activations_bf16(M: int, K: int, seed: int) -> np.ndarray:
    """bfloat16 [M, K] activations (bit patterns), the draws of activations()."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def activations(M: int, K: int, seed: int) -> np.ndarray:
    """fp16 [M, K] activations, N(0, 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal((M, K), dtype=np.float32).astype(np.float16)


def codes_and_params(K: int, N: int, group: int, seed: int):
    """Random raw format fields (not a quantization): codes q in [0,15] as packed
    words, positive fp16 scales and integer fp16 zeros in [0,15].  Used to drive
    the GEMM with arbitrary valid encodings."""
    rng = np.random.Generator(np.random.PCG64(seed))
    packed = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    scales = (rng.random((K // group, N), dtype=np.float32) * np.float32(0.004)
              + np.float32(0.0005)).astype(np.float16)
    zeros = rng.integers(0, 16, size=(K // group, N)).astype(np.float16)
    return packed, scales, zeros
