"""fp64 CPU oracle for the W4A16 weight-only GEMM -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never does, and the two share no code.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, fp64, optional OpenMP);
this module compiles it with gcc on first use and wraps it with ctypes and
numpy.  ``brute.py`` next to it is an independent pure-Python restatement used
to cross-check the C code on tiny shapes.

Pins (tests that tie the oracle to something other than itself) are in
``tests/test_oracle_*.py``.  Parity with numbers printed on the pages is
unpinned: the pages print no worked numeric example for this path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_w4a16.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc a C oracle source file into a shared library (fp64, no fast-math,
    no FMA contraction, OpenMP over columns)."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the committed oracle into ``oracle/liboracle_w4a16.so``."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class Oracle:
    """The C oracle loaded from one shared library (the default build, or a
    test-only variant compiled from a modified copy of the source)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.oracle_double_to_half.restype = ctypes.c_uint16
        lib.oracle_quantize_pack.argtypes = [P, I, I, I, P, P, P, P]
        lib.oracle_quantize_pack_symmetric.argtypes = [P, I, I, I, P, P, P, P]
        lib.oracle_unpack.argtypes = [P, I, I, P]
        lib.oracle_dequant.argtypes = [P, P, P, I, I, I, P]
        lib.oracle_gemm.argtypes = [P, P, P, P, I, I, I, I, P]
        lib.oracle_num_threads.argtypes = []
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_quantize_pack_bf16.argtypes = [P, I, I, I, P, P, P, P]
        lib.oracle_dequant_bf16.argtypes = [P, P, P, I, I, I, P]
        lib.oracle_gemm_bf16.argtypes = [P, P, P, P, I, I, I, I, P]
        lib.oracle_permuted_words.argtypes = [I, I, I]
        lib.oracle_permuted_words.restype = ctypes.c_longlong
        lib.oracle_permute.argtypes = [P, P, P, I, I, I, P]
        lib.oracle_unpermute.argtypes = [P, I, I, I, P, P, P]
        for f in (lib.oracle_quantize_pack, lib.oracle_quantize_pack_symmetric, lib.oracle_unpack,
                  lib.oracle_dequant, lib.oracle_gemm, lib.oracle_num_threads,
                  lib.oracle_permute, lib.oracle_unpermute, lib.oracle_quantize_pack_bf16,
                  lib.oracle_dequant_bf16, lib.oracle_gemm_bf16):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    # ------------------------------------------------------------ binary16
    def half_to_double(self, bits: int) -> float:
        return self.lib.oracle_half_to_double(int(bits))

    def double_to_half(self, v: float) -> int:
        return int(self.lib.oracle_double_to_half(float(v)))

    # ------------------------------------------------------ quantize/pack
    def quantize_pack(self, W, group: int = 128, return_codes: bool = False,
                      symmetric: bool = False):
        """W [K,N] fp16 -> (packed uint32 [K/8,N], scales fp16 [K/g,N], zeros fp16 [K/g,N]).
        symmetric=True: s = fp16(max|w| / 7), z = 8 (signed codes stored with +8)."""
        Wb = _as_half_bits(W)
        K, N = Wb.shape
        G = K // group if group > 0 else 0
        packed = np.zeros((max(K // 8, 0), N), dtype=np.uint32)
        scales = np.zeros((G, N), dtype=np.uint16)
        zeros = np.zeros((G, N), dtype=np.uint16)
        q = np.zeros((K, N), dtype=np.uint8) if return_codes else None
        fn = self.lib.oracle_quantize_pack_symmetric if symmetric else self.lib.oracle_quantize_pack
        rc = fn(_ptr(Wb), K, N, group, _ptr(packed), _ptr(scales), _ptr(zeros),
                _ptr(q) if q is not None else None)
        _check(rc, "quantize_pack")
        out = (packed, scales.view(np.float16), zeros.view(np.float16))
        return out + (q,) if return_codes else out

    def unpack(self, packed: np.ndarray) -> np.ndarray:
        """packed uint32 [K/8,N] -> codes uint8 [K,N]."""
        packed = np.ascontiguousarray(packed, dtype=np.uint32)
        K8, N = packed.shape
        q = np.zeros((K8 * 8, N), dtype=np.uint8)
        _check(self.lib.oracle_unpack(_ptr(packed), K8 * 8, N, _ptr(q)), "unpack")
        return q

    def dequant(self, packed, scales, zeros, group: int = 128) -> np.ndarray:
        """-> Wdq fp16 [K,N], Wdq = fp16((q - z) * s)."""
        packed = np.ascontiguousarray(packed, dtype=np.uint32)
        sb, zb = _as_half_bits(scales), _as_half_bits(zeros)
        K, N = packed.shape[0] * 8, packed.shape[1]
        Wdq = np.zeros((K, N), dtype=np.uint16)
        _check(self.lib.oracle_dequant(_ptr(packed), _ptr(sb), _ptr(zb), K, N, group,
                                       _ptr(Wdq)), "dequant")
        return Wdq.view(np.float16)

    def gemm(self, x, packed, scales, zeros, group: int = 128) -> np.ndarray:
        """x fp16 [M,K] -> ref fp64 [M,N] = x @ dequant(packed, scales, zeros)."""
        xb = _as_half_bits(x)
        packed = np.ascontiguousarray(packed, dtype=np.uint32)
        sb, zb = _as_half_bits(scales), _as_half_bits(zeros)
        M, K = xb.shape
        N = packed.shape[1]
        if packed.shape[0] * 8 != K:
            raise ValueError("x has K=%d but packed holds %d rows" % (K, packed.shape[0] * 8))
        ref = np.zeros((M, N), dtype=np.float64)
        _check(self.lib.oracle_gemm(_ptr(xb), _ptr(packed), _ptr(sb), _ptr(zb), M, N, K,
                                    group, _ptr(ref)), "gemm")
        return ref

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    # ------------------------------------------------------------- bfloat16
    # bfloat16 values travel as uint16 bit patterns (numpy has no bfloat16)
    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(int(bits))

    def double_to_bf16(self, v: float) -> int:
        return int(self.lib.oracle_double_to_bf16(float(v)))

    def quantize_pack_bf16(self, W_bits, group: int = 128, return_codes: bool = False):
        """W [K,N] bfloat16 bit patterns -> (packed uint32 [K/8,N], scales and zeros
        as bfloat16 bit patterns [K/g,N])."""
        Wb = _as_u16(W_bits)
        K, N = Wb.shape
        G = K // group if group > 0 else 0
        packed = np.zeros((max(K // 8, 0), N), dtype=np.uint32)
        scales = np.zeros((G, N), dtype=np.uint16)
        zeros = np.zeros((G, N), dtype=np.uint16)
        q = np.zeros((K, N), dtype=np.uint8) if return_codes else None
        _check(self.lib.oracle_quantize_pack_bf16(_ptr(Wb), K, N, group, _ptr(packed),
                                                  _ptr(scales), _ptr(zeros),
                                                  _ptr(q) if q is not None else None),
               "quantize_pack_bf16")
        out = (packed, scales, zeros)
        return out + (q,) if return_codes else out

    def dequant_bf16(self, packed, scales, zeros, group: int = 128) -> np.ndarray:
        """-> Wdq [K,N] bfloat16 bit patterns, bf16((q - z) * s)."""
        packed = np.ascontiguousarray(packed, dtype=np.uint32)
        K, N = packed.shape[0] * 8, packed.shape[1]
        Wdq = np.zeros((K, N), dtype=np.uint16)
        _check(self.lib.oracle_dequant_bf16(_ptr(packed), _ptr(_as_u16(scales)),
                                            _ptr(_as_u16(zeros)), K, N, group, _ptr(Wdq)),
               "dequant_bf16")
        return Wdq

    def gemm_bf16(self, x_bits, packed, scales, zeros, group: int = 128) -> np.ndarray:
        """x [M,K] bfloat16 bit patterns -> ref fp64 [M,N] = x @ bf16 dequant."""
        xb = _as_u16(x_bits)
        packed = np.ascontiguousarray(packed, dtype=np.uint32)
        M, K = xb.shape
        N = packed.shape[1]
        ref = np.zeros((M, N), dtype=np.float64)
        _check(self.lib.oracle_gemm_bf16(_ptr(xb), _ptr(packed), _ptr(_as_u16(scales)),
                                         _ptr(_as_u16(zeros)), M, N, K, group, _ptr(ref)),
               "gemm_bf16")
        return ref

    # ------------------------------------------------- pre-permuted layout
    def permute(self, packed, scales, zeros, group: int = 128) -> np.ndarray:
        """natural (packed [K/8,N], scales, zeros) -> repacked uint32 words (the
        pre-permuted layout defined in w4a16_oracle.c)."""
        packed = np.ascontiguousarray(packed, dtype=np.uint32)
        sb, zb = _as_half_bits(scales), _as_half_bits(zeros)
        K, N = packed.shape[0] * 8, packed.shape[1]
        n = int(self.lib.oracle_permuted_words(K, N, group))
        if n <= 0:
            raise ValueError("permute: unsupported shape K=%d N=%d group=%d" % (K, N, group))
        out = np.zeros(n, dtype=np.uint32)
        _check(self.lib.oracle_permute(_ptr(packed), _ptr(sb), _ptr(zb), K, N, group, _ptr(out)),
               "permute")
        return out

    def unpermute(self, words, K: int, N: int, group: int = 128):
        """repacked words -> (packed uint32 [K/8,N], scales fp16, zeros fp16)."""
        words = np.ascontiguousarray(words, dtype=np.uint32)
        if words.size != int(self.lib.oracle_permuted_words(K, N, group)):
            raise ValueError("unpermute: %d words do not fit K=%d N=%d group=%d"
                             % (words.size, K, N, group))
        packed = np.zeros((K // 8, N), dtype=np.uint32)
        scales = np.zeros((K // group, N), dtype=np.uint16)
        zeros = np.zeros((K // group, N), dtype=np.uint16)
        _check(self.lib.oracle_unpermute(_ptr(words), K, N, group, _ptr(packed), _ptr(scales),
                                         _ptr(zeros)), "unpermute")
        return packed, scales.view(np.float16), zeros.view(np.float16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_half_bits(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("expected float16 values or uint16 bit patterns, got %s" % a.dtype)
    return np.ascontiguousarray(a)


def _as_u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expected uint16 bit patterns, got %s" % a.dtype)
    return np.ascontiguousarray(a)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError("%s: bad argument (oracle code %d)" % (what, rc))


def default() -> Oracle:
    """The oracle built from the committed source (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def half_to_double(bits: int) -> float:
    return default().half_to_double(bits)


def double_to_half(v: float) -> int:
    return default().double_to_half(v)


def quantize_pack(W, group: int = 128, return_codes: bool = False, symmetric: bool = False):
    return default().quantize_pack(W, group, return_codes, symmetric)


def unpack(packed):
    return default().unpack(packed)


def dequant(packed, scales, zeros, group: int = 128):
    return default().dequant(packed, scales, zeros, group)


def gemm(x, packed, scales, zeros, group: int = 128):
    return default().gemm(x, packed, scales, zeros, group)


def num_threads() -> int:
    return default().num_threads()


def quantize_pack_bf16(W_bits, group: int = 128, return_codes: bool = False):
    return default().quantize_pack_bf16(W_bits, group, return_codes)


def dequant_bf16(packed, scales, zeros, group: int = 128):
    return default().dequant_bf16(packed, scales, zeros, group)


def gemm_bf16(x_bits, packed, scales, zeros, group: int = 128):
    return default().gemm_bf16(x_bits, packed, scales, zeros, group)


def permute(packed, scales, zeros, group: int = 128):
    return default().permute(packed, scales, zeros, group)


def unpermute(words, K: int, N: int, group: int = 128):
    return default().unpermute(words, K, N, group)


def rel_err(out, ref) -> float:
    """max over elements of |out - ref| / max(1, |ref|) -- the acceptance measure."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if out.size == 0:
        return 0.0
    return float(np.max(np.abs(out - ref) / np.maximum(1.0, np.abs(ref))))
