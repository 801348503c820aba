"""Host-only checks of the C-ABI library: it loads, exports every entry point
include/w4a16.h declares, and its host logic (validation, planning) behaves.
No test here launches a kernel."""
import ctypes
import os
import re

import pytest

import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
import weight_only_int4_codes_gb300 as w4
from weight_only_int4_codes_gb300 import build as wbuild
from weight_only_int4_codes_gb300 import native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    wbuild.build()
    return native.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"W4A16_API\s+[\w\s\*]+?\b(w4a16_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for required in ("w4a16_quantize_pack", "w4a16_gemm", "w4a16_gemm_ex", "w4a16_dequantize",
                     "w4a16_plan", "w4a16_get_kernel_status", "w4a16_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_no_internal_symbols_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", native.library_path()],
                         capture_output=True, text=True).stdout
    text_syms = [ln.split()[-1] for ln in out.splitlines() if " T " in ln]
    assert text_syms and all(s.startswith("w4a16_") for s in text_syms), text_syms


def test_version(lib):
    assert lib.w4a16_version() >= 100


@pytest.mark.parametrize("M,N,K,group,status", [
    (1, 4096, 4000, 128, 1),    # K not a multiple of group
    (1, 4096, 4096, 100, 1),    # group not a multiple of 8
    (1, 4096, 4096, 8, 2),      # valid format, group below the library's minimum
    (1, 4094, 4096, 128, 3),    # N % 4 != 0
    (-1, 4096, 4096, 128, 1),   # negative size
    (1, 4096, 0, 128, 1),       # K == 0
])
def test_validation_statuses(lib, M, N, K, group, status):
    out = native.Config()
    assert lib.w4a16_plan(M, N, K, group, None, ctypes.byref(out)) == status
    assert lib.w4a16_last_error().decode()


def test_gemm_rejects_before_touching_the_gpu(lib):
    # shape errors and null pointers are caught on the host; M == 0 is a no-op
    assert lib.w4a16_gemm(None, None, None, None, None, 1, 256, 500, 128, None) == 1
    assert lib.w4a16_gemm(None, None, None, None, None, 0, 256, 512, 128, None) == 0
    assert lib.w4a16_gemm(None, None, None, None, None, 1, 256, 512, 128, None) == 1
    assert b"null" in lib.w4a16_last_error()
    # misaligned pointers (never dereferenced: validation fails first)
    assert lib.w4a16_gemm(8, 16, 16, 16, 16, 1, 256, 512, 128, None) == 3


def test_quantize_mode_is_checked_first(lib):
    # an unknown mode is refused before anything else is looked at
    assert lib.w4a16_quantize_pack_ex(None, 512, 256, 128, 2, None, None, None, None) == 1
    assert b"mode" in lib.w4a16_last_error()
    # known modes go on to the usual checks (null pointers here)
    for mode in (0, 1):
        assert lib.w4a16_quantize_pack_ex(None, 512, 256, 128, mode, None, None, None, None) == 1
        assert b"null" in lib.w4a16_last_error()


def test_grouped_rejects_before_touching_the_gpu(lib):
    P = ctypes.c_void_p
    good = (P * 2)(16, 32)
    bad = (P * 2)(16, 8)          # second expert's pointer not 16-byte aligned
    null = (P * 2)(16, None)
    call = lambda E, t, u=good: lib.w4a16_gemm_grouped(E, t, u, u, u, u, 1, 256, 512, 128,
                                                       None, None)
    assert call(0, good) == 1                 # no experts
    assert call(65, good) == 1                # above W4A16_MAX_EXPERTS
    assert lib.w4a16_gemm_grouped(2, None, good, good, good, good, 1, 256, 512, 128,
                                  None, None) == 1
    assert call(2, null) == 1 and b"expert 1" in lib.w4a16_last_error()
    assert call(2, bad) == 3 and b"expert 1" in lib.w4a16_last_error()
    assert lib.w4a16_gemm_grouped(2, good, good, good, good, good, 1, 256, 500, 128,
                                  None, None) == 1    # K not a multiple of the group
    assert lib.w4a16_gemm_grouped(2, good, good, good, good, good, 0, 256, 512, 128,
                                  None, None) == 0    # M == 0: nothing to do
    tma = native.Config.make(dict(variant="tma"))
    assert lib.w4a16_gemm_grouped(2, good, good, good, good, good, 1, 256, 512, 128,
                                  ctypes.byref(tma), None) == 2


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 4096, 4096), (4, 14336, 4096),
                                   (8, 4096, 14336), (1, 768, 2048), (16, 2048, 768),
                                   (3, 260, 512), (40, 1024, 1024)])
def test_decode_plan_covers_k(M, N, K):
    p = w4.plan(M, N, K, 128, path="decode", variant="registers")
    assert p["path"] == 1 and p["variant"] == 2
    assert 1 <= p["split_k"] <= 8
    assert p["warps_k"] * p["steps"] * 4 * p["split_k"] >= K // 8
    assert p["steps"] % 4 == 0
    if N % 8:
        with pytest.raises(native.W4A16Error) as e:   # scale rows would not be 16-byte pitched
            w4.plan(M, N, K, 128, path="decode", variant="tma")
        assert e.value.status == 2
        return
    t = w4.plan(M, N, K, 128, path="decode", variant="tma")
    assert t["variant"] == 1 and t["warps_n"] in (2, 4) and 1 <= t["split_k"] <= 8
    assert t["steps"] * 256 * t["split_k"] >= K


def test_plan_respects_requests():
    p = w4.plan(1, 4096, 4096, 128, path="decode", variant="registers", split_k=4, warps_k=4,
                warps_n=1)
    assert (p["split_k"], p["warps_k"], p["warps_n"]) == (4, 4, 1)
    assert p["steps"] * 4 * 4 * 4 >= 4096 // 8
    with pytest.raises(native.W4A16Error) as e:
        w4.plan(1, 4096, 4096, 128, path="decode", variant="registers", split_k=9)
    assert e.value.status == 2


def test_prefill_split_k_requests():
    p = w4.plan(64, 4096, 4096, 128, path="prefill", tile_m=64, split_k=4)
    assert (p["path"], p["split_k"], p["tile_m"]) == (2, 4, 64)
    for bad in (dict(split_k=9), dict(split_k=2, variant=3), dict(split_k=2, variant="smem"),
                dict(split_k=4, tile_m=128, warps_k=4)):
        with pytest.raises(native.W4A16Error) as e:
            w4.plan(64, 4096, 4096, 128, path="prefill", **dict(dict(tile_m=64), **bad))
        assert e.value.status == 2


def test_auto_path_small_m_is_decode():
    for M in (1, 2, 4, 8, 16):
        p = w4.plan(M, 4096, 4096)
        assert p["path"] == 1 and p["variant"] in (1, 2, 4)
    # measured dispatch table rows
    assert w4.plan(1, 4096, 4096)["variant"] == 1         # TMA variant at M <= 2
    assert w4.plan(4, 4096, 4096)["variant"] == 4         # warp-stream variant at M = 3..4
    assert w4.plan(8, 4096, 4096)["variant"] == 2         # registers variant at M = 8
    assert w4.plan(16, 4096, 4096)["variant"] == 2         # registers variant at M = 16
    t = w4.plan(4, 14336, 4096)
    assert (t["variant"], t["warps_n"], t["warps_k"], t["split_k"], t["steps"]) == (1, 2, 4, 2, 8)
    assert w4.plan(1, 4092, 4096)["variant"] == 2         # N % 8 != 0: registers variant
    assert w4.plan(1, 4096, 4096, 512)["variant"] == 2    # group 512: registers variant
    # off-table shapes take the TMA planner when the format allows it
    assert w4.plan(1, 8192, 8192)["variant"] == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(native, "_lib", None)
    monkeypatch.setattr(native, "_PKG", str(tmp_path))
    with pytest.raises(native.W4A16Error):
        native.load_library()


def test_bf16_planning():
    """dtype = bf16: decode on the registers or TMA variant (a measured table
    row for another variant falls back to the TMA planner), prefill on A in
    tensor memory; the other variants and unknown dtypes are refused."""
    for M in (1, 8, 16):
        p = w4.plan(M, 4096, 4096, dtype="bf16")
        assert (p["path"], p["dtype"]) == (1, 1) and p["variant"] in (1, 2)
    # the bf16 dispatch table (measured on bf16 data)
    t = w4.plan(1, 4096, 4096, dtype="bf16")
    assert (t["variant"], t["split_k"], t["warps_k"], t["warps_n"], t["steps"]) == (1, 8, 4, 2, 2)
    assert w4.plan(16, 2048, 768, dtype="bf16")["variant"] == 2
    assert w4.plan(4, 4096, 14336, dtype="bf16")["variant"] == 1
    # off the table: the TMA planner
    assert w4.plan(1, 8192, 8192, dtype="bf16")["variant"] == 1
    p = w4.plan(1024, 14336, 4096, dtype="bf16")
    assert (p["path"], p["dtype"]) == (2, 1) and p["variant"] == 1
    for bad in (dict(path="decode", variant="warp"), dict(path="decode", variant="stream"),
                dict(path="prefill", variant="smem", tile_m=64)):
        with pytest.raises(native.W4A16Error) as e:
            w4.plan(64 if bad["path"] == "prefill" else 4, 4096, 4096, dtype="bf16", **bad)
        assert e.value.status == 2
    with pytest.raises(native.W4A16Error) as e:
        w4.plan(4, 4096, 4096, dtype=7)
    assert e.value.status == 1
    assert w4.plan(4, 4096, 4096)["dtype"] == 0


def test_gemm_call_validates(lib):
    """The argument-block entry: a null block is refused; a block with a bad
    shape returns the same status as w4a16_gemm_ex."""
    assert lib.w4a16_gemm_call(None, None) == 1
    blk = native.GemmArgs(16, 16, 16, 16, 16, 1, 4096, 4000, 128, None)   # K % group != 0
    assert lib.w4a16_gemm_call(ctypes.byref(blk), None) == 1
    blk = native.GemmArgs(16, 16, 16, 16, 16, 1, 4094, 4096, 128, None)   # N % 4 != 0
    assert lib.w4a16_gemm_call(ctypes.byref(blk), None) == 3


def test_bf16_entries_validate_before_touching_the_gpu(lib):
    assert lib.w4a16_quantize_pack_bf16(None, 512, 256, 128, None, None, None, None) == 1
    assert lib.w4a16_quantize_pack_bf16(16, 500, 256, 128, 16, 16, 16, None) == 1   # K % group
    assert lib.w4a16_dequantize_bf16(16, 16, 17, 16, 512, 256, 128, None) == 3     # misaligned
    assert lib.w4a16_quantize_pack_bf16(16, 512, 0, 128, 16, 16, 16, None) == 0    # N == 0


def test_repacked_entries_validate_before_touching_the_gpu(lib):
    """The repacked GEMM entries refuse bad shapes, variants, dtypes and
    pointers on the host (no pointer below is ever dereferenced)."""
    cfg = lambda **kw: ctypes.byref(native.Config.make(kw))
    call = lambda M, K=1024, c=None, ptrs=(16, 32, 48): lib.w4a16_gemm_repacked(
        *ptrs, M, 512, K, 128, c, None)
    assert call(1, K=384) == 2                                  # K % 256 != 0
    assert call(9, c=cfg(path="decode", variant="warp")) == 2   # warp kernel: M <= 8
    assert b"M <= 8" in lib.w4a16_last_error()
    assert call(1, c=cfg(path="decode", variant="registers")) == 2
    assert call(1, c=cfg(dtype="bf16")) == 2 and b"fp16" in lib.w4a16_last_error()
    assert call(1, ptrs=(None, None, None)) == 1 and b"null" in lib.w4a16_last_error()
    assert call(1, ptrs=(16, 40, 48)) == 3                      # misaligned repacked
    assert call(0) == 0                                         # nothing to do
    P = ctypes.c_void_p
    good = (P * 2)(16, 32)
    gcall = lambda E, M, t=good, c=None: lib.w4a16_gemm_grouped_repacked(
        E, t, t, t, M, 512, 1024, 128, c, None)
    assert gcall(0, 1) == 1 and gcall(65, 1) == 1               # 1..64 experts
    assert gcall(2, 17) == 2                                    # M <= 16
    assert gcall(2, 1, t=(P * 2)(16, None)) == 1
    assert gcall(2, 1, t=(P * 2)(16, 8)) == 3
