"""ctypes binding of libw4a16.so (declared in include/w4a16.h).

Argument marshalling only: tensors are checked for device, dtype and
contiguity, their data pointers and the current CUDA stream are handed to the
C ABI, and a non-OK status becomes a ``W4A16Error``.  Every step of the
computation runs in the library's CUDA kernels; if the library is missing this
module raises instead of falling back to anything else.

PyTorch is used here only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libw4a16.so"

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "MISALIGNED", 4: "CUDA",
                5: "TIMEOUT"}
PATHS = {"auto": 0, "decode": 1, "prefill": 2}
VARIANTS = {"auto": 0, "tma": 1, "registers": 2, "stream": 3, "warp": 4,   # decode path
            "tmem": 1, "smem": 2}                  # prefill path: A's home
DTYPES = {"f16": 0, "fp16": 0, "float16": 0, "bf16": 1, "bfloat16": 1}
DTYPE_F16, DTYPE_BF16 = 0, 1
QUANT_ASYMMETRIC, QUANT_SYMMETRIC = 0, 1
FLAG_PDL = 0x1
FLAG_TEST_TIMEOUT = 0x100


class W4A16Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("w4a16 %s (%d): %s" % (STATUS_NAMES.get(status, "?"), status, message))
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("split_k", ctypes.c_int), ("warps_k", ctypes.c_int),
                ("warps_n", ctypes.c_int), ("steps", ctypes.c_int), ("tile_m", ctypes.c_int),
                ("flags", ctypes.c_int), ("variant", ctypes.c_int), ("ctas", ctypes.c_int),
                ("dtype", ctypes.c_int)]

    @classmethod
    def make(cls, cfg):
        if cfg is None:
            return None
        if isinstance(cfg, Config):
            return cfg
        try:
            key = tuple(sorted(cfg.items()))
            hit = _cfg_cache.get(key)
        except (AttributeError, TypeError):
            key, hit = None, None
        if hit is not None:
            return hit
        c = cls._build(cfg)
        if key is not None and len(_cfg_cache) < 256:
            _cfg_cache[key] = c
        return c

    @classmethod
    def _build(cls, cfg):
        c = cls()
        for k, v in dict(cfg).items():
            if k == "path" and isinstance(v, str):
                v = PATHS[v]
            if k == "variant" and isinstance(v, str):
                v = VARIANTS[v]
            if k == "dtype" and isinstance(v, str):
                v = DTYPES[v]
            if k == "pdl":
                c.flags |= FLAG_PDL if v else 0
                continue
            setattr(c, k, int(v))
        return c

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class GemmArgs(ctypes.Structure):
    """w4a16_gemm_args: the argument block of w4a16_gemm_call."""
    _fields_ = [("x", ctypes.c_void_p), ("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p), ("out", ctypes.c_void_p), ("M", ctypes.c_int),
                ("N", ctypes.c_int), ("K", ctypes.c_int), ("group", ctypes.c_int),
                ("cfg", ctypes.POINTER(Config))]


_lock = threading.Lock()
_lib = None
_cfg_cache = {}       # config dict items -> Config (read-only once built)


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


def load_library():
    """Load libw4a16.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise W4A16Error(4, "%s is not built; run `python -c 'import __graft_entry__ as g; "
                                "g.build()'`" % path)
        lib = ctypes.CDLL(path)
        P, I = ctypes.c_void_p, ctypes.c_int
        sig = {
            "w4a16_quantize_pack": [P, I, I, I, P, P, P, P],
            "w4a16_quantize_pack_ex": [P, I, I, I, I, P, P, P, P],
            "w4a16_dequantize": [P, P, P, P, I, I, I, P],
            "w4a16_quantize_pack_bf16": [P, I, I, I, P, P, P, P],
            "w4a16_dequantize_bf16": [P, P, P, P, I, I, I, P],
            "w4a16_gemm": [P, P, P, P, P, I, I, I, I, P],
            "w4a16_gemm_ex": [P, P, P, P, P, I, I, I, I, ctypes.POINTER(Config), P],
            "w4a16_plan": [I, I, I, I, ctypes.POINTER(Config), ctypes.POINTER(Config)],
            "w4a16_gemm_grouped": [I, P, P, P, P, P, I, I, I, I, ctypes.POINTER(Config), P],
            "w4a16_repack": [P, P, P, I, I, I, P, P],
            "w4a16_gemm_repacked": [P, P, P, I, I, I, I, ctypes.POINTER(Config), P],
            "w4a16_gemm_grouped_repacked": [I, P, P, P, I, I, I, I, ctypes.POINTER(Config), P],
            "w4a16_get_kernel_status": [P],
            "w4a16_stream_read": [P, ctypes.c_size_t, P, I, P],
            "w4a16_gemm_noalloc": [P, P, P, P, P, I, I, I, I, P],
            "w4a16_gemm_call": [ctypes.POINTER(GemmArgs), P],
            "w4a16_last_error": [],
            "w4a16_version": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.w4a16_last_error.restype = ctypes.c_char_p
        lib.w4a16_repacked_bytes.argtypes = [I, I, I]
        lib.w4a16_repacked_bytes.restype = ctypes.c_size_t
        _lib = lib
        return lib


def _lib_fast():
    lib = _lib
    return lib if lib is not None else load_library()


def _check(status: int):
    if status != 0:
        msg = load_library().w4a16_last_error().decode(errors="replace")
        raise W4A16Error(status, msg)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream) -> int:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _dev(t: torch.Tensor, name: str, dtype) -> int:
    # fast path first: the per-call host cost matters at decode sizes
    if type(t) is torch.Tensor and t.dtype is dtype and t.is_cuda and t.is_contiguous():
        return t.data_ptr()
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def quantize_pack(W: torch.Tensor, group: int = 128, stream=None, symmetric: bool = False):
    """fp16 W [K,N] -> (packed int32 [K/8,N], scales fp16 [K/g,N], zeros fp16 [K/g,N]).
    symmetric=True: s = fp16(max|w| / 7), z = 8 (signed codes stored with +8)."""
    K, N = W.shape
    packed = torch.empty((K // 8, N), dtype=torch.int32, device=W.device)
    scales = torch.empty((K // group, N), dtype=torch.float16, device=W.device)
    zeros = torch.empty((K // group, N), dtype=torch.float16, device=W.device)
    _check(load_library().w4a16_quantize_pack_ex(
        _dev(W, "W", torch.float16), K, N, group, QUANT_SYMMETRIC if symmetric else QUANT_ASYMMETRIC,
        _dev(packed, "packed", torch.int32),
        _dev(scales, "scales", torch.float16), _dev(zeros, "zeros", torch.float16),
        _stream_handle(stream)))
    return packed, scales, zeros


def dequantize(packed, scales, zeros, group: int = 128, stream=None) -> torch.Tensor:
    """-> fp16 W [K,N] = fp16((q - z) * s)."""
    K, N = packed.shape[0] * 8, packed.shape[1]
    W = torch.empty((K, N), dtype=torch.float16, device=packed.device)
    _check(load_library().w4a16_dequantize(
        _dev(packed, "packed", torch.int32), _dev(scales, "scales", torch.float16),
        _dev(zeros, "zeros", torch.float16), _dev(W, "W_out", torch.float16), K, N, group,
        _stream_handle(stream)))
    return W


def quantize_pack_bf16(W: torch.Tensor, group: int = 128, stream=None):
    """bfloat16 W [K,N] -> (packed int32 [K/8,N], scales bf16 [K/g,N], zeros bf16 [K/g,N])."""
    K, N = W.shape
    packed = torch.empty((K // 8, N), dtype=torch.int32, device=W.device)
    scales = torch.empty((K // group, N), dtype=torch.bfloat16, device=W.device)
    zeros = torch.empty((K // group, N), dtype=torch.bfloat16, device=W.device)
    _check(load_library().w4a16_quantize_pack_bf16(
        _dev(W, "W", torch.bfloat16), K, N, group, _dev(packed, "packed", torch.int32),
        _dev(scales, "scales", torch.bfloat16), _dev(zeros, "zeros", torch.bfloat16),
        _stream_handle(stream)))
    return packed, scales, zeros


def dequantize_bf16(packed, scales, zeros, group: int = 128, stream=None) -> torch.Tensor:
    """-> bfloat16 W [K,N] = bf16((q - z) * s)."""
    K, N = packed.shape[0] * 8, packed.shape[1]
    W = torch.empty((K, N), dtype=torch.bfloat16, device=packed.device)
    _check(load_library().w4a16_dequantize_bf16(
        _dev(packed, "packed", torch.int32), _dev(scales, "scales", torch.bfloat16),
        _dev(zeros, "zeros", torch.bfloat16), _dev(W, "W_out", torch.bfloat16), K, N, group,
        _stream_handle(stream)))
    return W


def _bf16_config(config):
    """``config`` with dtype = bfloat16 (a new Config; the caller's is not changed)."""
    base = Config.make(config)
    c = _copy_config(base) if base is not None else Config()
    c.dtype = DTYPE_BF16
    return c


def gemm_ex(x, packed, scales, zeros, group: int = 128, out=None, config=None, stream=None):
    """out [M,N] = x [M,K] @ dequant(packed, scales, zeros); ``config`` is a
    dict of w4a16_config fields (path may be 'auto' | 'decode' | 'prefill',
    pdl=True sets W4A16_FLAG_PDL).  x, scales, zeros and out are all fp16, or
    all bfloat16 (then the call runs with dtype = W4A16_DTYPE_BF16)."""
    M, K = x.shape
    N = packed.shape[1]
    et = torch.bfloat16 if x.dtype is torch.bfloat16 else torch.float16
    if out is None:
        out = torch.empty((M, N), dtype=et, device=x.device)
    cfg = _bf16_config(config) if et is torch.bfloat16 else Config.make(config)
    _check(_lib_fast().w4a16_gemm_ex(
        _dev(x, "x", et), _dev(packed, "packed", torch.int32),
        _dev(scales, "scales", et), _dev(zeros, "zeros", et),
        _dev(out, "out", et), M, N, K, group,
        ctypes.byref(cfg) if cfg is not None else None, _stream_handle(stream)))
    return out


class PreparedGemm:
    """One GEMM call with its arguments checked and marshalled once.

    ``prepare_gemm`` validates the tensors (device, dtype, contiguity), takes
    their data pointers and builds the argument block of ``w4a16_gemm_call``;
    each call passes that block and the current (or the given) CUDA stream,
    so a loop that repeats the same product with new contents in x pays only
    a two-argument C call.  The tensors are referenced by the object and must
    keep their storage (no resize) while it is used; ``out`` is the result.
    """
    __slots__ = ("_fn", "_ref", "_block", "_cfg", "_keep", "_dev", "out")

    def __init__(self, fn, block, cfg, keep, dev, out):
        self._fn, self._block, self._cfg, self._keep, self._dev = fn, block, cfg, keep, dev
        self._ref = ctypes.byref(block)
        self.out = out

    def __call__(self, stream=None):
        if stream is None and _raw_stream is not None:
            h = _raw_stream(self._dev)
        else:
            h = _stream_handle(stream)
        st = self._fn(self._ref, h)
        if st != 0:
            _check(st)
        return self.out


def prepare_gemm(x, packed, scales, zeros, group: int = 128, out=None, config=None):
    """A reusable call of ``gemm_ex(x, packed, scales, zeros, group, out, config)``;
    see ``PreparedGemm``."""
    M, K = x.shape
    N = packed.shape[1]
    et = torch.bfloat16 if x.dtype is torch.bfloat16 else torch.float16
    if out is None:
        out = torch.empty((M, N), dtype=et, device=x.device)
    cfg = _bf16_config(config) if et is torch.bfloat16 else Config.make(config)
    if cfg is not None:
        cfg = _copy_config(cfg)            # private: the caller may change theirs later
    block = GemmArgs(_dev(x, "x", et), _dev(packed, "packed", torch.int32),
                     _dev(scales, "scales", et), _dev(zeros, "zeros", et), _dev(out, "out", et),
                     M, N, K, group, ctypes.pointer(cfg) if cfg is not None else None)
    return PreparedGemm(_lib_fast().w4a16_gemm_call, block, cfg, (x, packed, scales, zeros),
                        x.device.index if x.device.index is not None else 0, out)


def _copy_config(c):
    d = Config()
    ctypes.memmove(ctypes.byref(d), ctypes.byref(c), ctypes.sizeof(Config))
    return d


def gemm(x, packed, scales, zeros, group: int = 128, out=None, stream=None):
    """out [M,N] fp16 = x [M,K] @ dequant(packed, scales, zeros), automatic path."""
    M, K = x.shape
    N = packed.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check(_lib_fast().w4a16_gemm(
        _dev(x, "x", torch.float16), _dev(packed, "packed", torch.int32),
        _dev(scales, "scales", torch.float16), _dev(zeros, "zeros", torch.float16),
        _dev(out, "out", torch.float16), M, N, K, group, _stream_handle(stream)))
    return out


def repacked_bytes(K: int, N: int, group: int = 128) -> int:
    """Bytes of the repacked (pre-permuted) form of a [K, N] weight; 0 if unsupported."""
    return int(load_library().w4a16_repacked_bytes(K, N, group))


def repack(packed, scales, zeros, group: int = 128, stream=None) -> torch.Tensor:
    """natural (packed, scales, zeros) -> the repacked layout, a uint8 device
    tensor of ``repacked_bytes(K, N, group)`` bytes."""
    K, N = packed.shape[0] * 8, packed.shape[1]
    n = repacked_bytes(K, N, group)
    if n == 0:
        raise W4A16Error(2, "repacked layout does not support K=%d N=%d group=%d" % (K, N, group))
    out = torch.empty(n, dtype=torch.uint8, device=packed.device)
    _check(load_library().w4a16_repack(
        _dev(packed, "packed", torch.int32), _dev(scales, "scales", torch.float16),
        _dev(zeros, "zeros", torch.float16), K, N, group, _dev(out, "repacked", torch.uint8),
        _stream_handle(stream)))
    return out


def gemm_repacked(x, repacked, N: int, group: int = 128, out=None, config=None, stream=None):
    """out [M,N] fp16 = x [M,K] @ W with W in the repacked layout."""
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    cfg = Config.make(config)
    _check(_lib_fast().w4a16_gemm_repacked(
        _dev(x, "x", torch.float16), _dev(repacked, "repacked", torch.uint8),
        _dev(out, "out", torch.float16), M, N, K, group,
        ctypes.byref(cfg) if cfg is not None else None, _stream_handle(stream)))
    return out


def gemm_noalloc(x, packed, scales, zeros, group: int = 128, out=None, stream=None):
    """out [M,N] fp16 = x [M,K] @ dequant(packed, scales, zeros) through the entry
    point that allocates no GPU memory (its scratch is a fixed array inside the
    library; calls that overlap on the GPU must not share it).  M <= 16."""
    M, K = x.shape
    N = packed.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check(_lib_fast().w4a16_gemm_noalloc(
        _dev(x, "x", torch.float16), _dev(packed, "packed", torch.int32),
        _dev(scales, "scales", torch.float16), _dev(zeros, "zeros", torch.float16),
        _dev(out, "out", torch.float16), M, N, K, group, _stream_handle(stream)))
    return out


def stream_read(src: torch.Tensor, sink: torch.Tensor, pdl: bool = False, stream=None):
    """Measurement aid: stream all of ``src`` into shared memory the way the
    decode kernels stream weights (no arithmetic); one word per SM to ``sink``."""
    if not (src.is_cuda and src.is_contiguous()):
        raise ValueError("src must be a contiguous CUDA tensor")
    _check(_lib_fast().w4a16_stream_read(src.data_ptr(), src.numel() * src.element_size(),
                                         _dev(sink, "sink", torch.int32),
                                         FLAG_PDL if pdl else 0, _stream_handle(stream)))


MAX_EXPERTS = 64


def _experts(t, name, dtype):
    """A stacked tensor [E, ...] or a sequence of E tensors -> list of device pointers."""
    if isinstance(t, torch.Tensor):
        return [_dev(t[e], name, dtype) for e in range(t.shape[0])]
    return [_dev(v, name, dtype) for v in t]


def gemm_grouped(xs, packed, scales, zeros, group: int = 128, out=None, config=None,
                 stream=None):
    """E expert GEMMs of one shape in one launch: out[e] = xs[e] @ dequant(packed[e], ...).
    Each argument is a stacked tensor with a leading expert dimension or a
    sequence of per-expert tensors; ``out`` likewise (allocated stacked if None
    and the experts' slices stay 16-byte aligned, else as a list)."""
    E = xs.shape[0] if isinstance(xs, torch.Tensor) else len(xs)
    x0 = xs[0]
    M, K = x0.shape
    N = packed[0].shape[1]
    if out is None:
        # stacked when every expert's slice stays 16-byte aligned, else one
        # tensor per expert
        if (M * N) % 8 == 0:
            out = torch.empty((E, M, N), dtype=torch.float16, device=x0.device)
        else:
            out = [torch.empty((M, N), dtype=torch.float16, device=x0.device) for _ in range(E)]
    ptrs = [_experts(xs, "x", torch.float16), _experts(packed, "packed", torch.int32),
            _experts(scales, "scales", torch.float16), _experts(zeros, "zeros", torch.float16),
            _experts(out, "out", torch.float16)]
    if any(len(p) != E for p in ptrs):
        raise ValueError("every argument needs %d experts" % E)
    tables = [(ctypes.c_void_p * E)(*p) for p in ptrs]
    cfg = Config.make(config)
    _check(load_library().w4a16_gemm_grouped(
        E, *[ctypes.cast(t, ctypes.c_void_p) for t in tables], M, N, K, group,
        ctypes.byref(cfg) if cfg is not None else None, _stream_handle(stream)))
    return out


def gemm_grouped_repacked(xs, repacked, N: int, group: int = 128, out=None, config=None,
                          stream=None):
    """E expert GEMMs of one shape in one launch with repacked weights (M <= 16)."""
    E = xs.shape[0] if isinstance(xs, torch.Tensor) else len(xs)
    x0 = xs[0]
    M, K = x0.shape
    if out is None:
        out = torch.empty((E, M, N), dtype=torch.float16, device=x0.device)
    ptrs = [_experts(xs, "x", torch.float16), _experts(repacked, "repacked", torch.uint8),
            _experts(out, "out", torch.float16)]
    if any(len(p) != E for p in ptrs):
        raise ValueError("every argument needs %d experts" % E)
    tables = [(ctypes.c_void_p * E)(*p) for p in ptrs]
    cfg = Config.make(config)
    _check(load_library().w4a16_gemm_grouped_repacked(
        E, *[ctypes.cast(t, ctypes.c_void_p) for t in tables], M, N, K, group,
        ctypes.byref(cfg) if cfg is not None else None, _stream_handle(stream)))
    return out


def plan(M: int, N: int, K: int, group: int = 128, **request) -> dict:
    """Launch configuration the library would use (host only, nothing enqueued)."""
    req = Config.make(request) if request else None
    out = Config()
    _check(load_library().w4a16_plan(M, N, K, group, ctypes.byref(req) if req else None,
                                     ctypes.byref(out)))
    return out.as_dict()


def kernel_status(stream=None) -> int:
    """Synchronize ``stream`` and read-and-clear the device status word."""
    lib = load_library()
    return int(lib.w4a16_get_kernel_status(_stream_handle(stream)))


def raw():
    """The loaded ctypes library, for callers that pass raw pointers."""
    return load_library()
