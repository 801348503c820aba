"""GB300-native W4A16 weight-only GEMM.

out[M,N] = x[M,K] @ W[K,N] with x fp16, fp32 accumulation and an fp16 output,
where W is held as unsigned 4-bit codes packed eight per int32 along K and
each group of 128 K-rows of each column carries one fp16 scale and one fp16
zero (W = (q - z) * s, dequantized inside the kernel).

All compute runs in the CUDA library ``libw4a16.so`` (hand-written sm_103a
kernels behind a C ABI, declared in ``include/w4a16.h``).  ``native`` is a thin
ctypes binding with the same names; it raises if the library is missing.  The
binding is imported on first attribute access, so ``synth`` (input generation)
can be used without the native library.
"""
_NATIVE_NAMES = {
    "W4A16Error", "gemm", "gemm_ex", "gemm_grouped", "dequantize", "quantize_pack",
    "kernel_status", "library_path", "load_library", "plan", "native", "repack",
    "repacked_bytes", "gemm_repacked", "gemm_grouped_repacked", "gemm_noalloc",
    "quantize_pack_bf16", "dequantize_bf16", "prepare_gemm", "PreparedGemm",
}


def __getattr__(name):
    if name in _NATIVE_NAMES:
        import importlib
        native = importlib.import_module(__name__ + ".native")
        return native if name == "native" else getattr(native, name)
    raise AttributeError(name)
