"""Pins for the fp64 oracle: checks that tie it to something other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a hand-worked example, a closed form, an independent
library routine or the pure-Python brute force.  ``test_oracle_pins.py`` runs
them on the committed oracle; ``test_oracle_mutants.py`` runs them on copies of
the oracle with a plausible mistake planted, and requires that some pin fails.
"""
from __future__ import annotations

import json
import os
import struct

import numpy as np

from oracle import brute
from weight_only_int4_codes_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _hex16(h: str) -> int:
    return int(h, 16)


def _f16_exact(vals) -> np.ndarray:
    a = np.asarray(vals, dtype=np.float64)
    h = a.astype(np.float16)
    assert np.array_equal(h.astype(np.float64), a), "fixture value not exact in fp16"
    return h


# --------------------------------------------------------------------- codec
def pin_half_decode_exhaustive(orc):
    """Every one of the 65,536 binary16 patterns decodes like numpy's float16."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def pin_half_encode(orc):
    """Round-to-nearest-even encoding: all finite patterns round-trip, midpoints
    between neighbours go to the even one, and random doubles match both numpy
    and Python's struct 'e' packing."""
    for b in range(65536):
        e = (b >> 10) & 31
        if e == 31:
            continue
        v = struct.unpack("<e", struct.pack("<H", b))[0]
        if b == 0x8000:
            v = -0.0
        assert orc.double_to_half(v) == b, hex(b)
    # exact midpoints between consecutive positive finite halves
    for b in range(0, 0x7bff):
        lo = struct.unpack("<e", struct.pack("<H", b))[0]
        hi = struct.unpack("<e", struct.pack("<H", b + 1))[0]
        mid = (lo + hi) / 2.0
        want = b if b % 2 == 0 else b + 1
        assert orc.double_to_half(mid) == want, hex(b)
        assert orc.double_to_half(-mid) == (want | 0x8000), hex(b)
    rng = np.random.Generator(np.random.PCG64(12345))
    vals = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
                           rng.uniform(-70000, 70000, 2000)])
    with np.errstate(over="ignore"):
        want_np = vals.astype(np.float16).view(np.uint16)
    for v, w in zip(vals, want_np):
        got = orc.double_to_half(float(v))
        assert got == int(w), v
        if abs(v) < 65520:
            assert got == struct.unpack("<H", struct.pack("<e", float(v)))[0], v
    assert orc.double_to_half(65519.99) == 0x7BFF
    assert orc.double_to_half(65520.0) == 0x7C00
    assert orc.double_to_half(-1e9) == 0xFC00
    assert orc.double_to_half(2.0 ** -25) == 0x0000        # tie to even (0)
    assert orc.double_to_half(3 * 2.0 ** -25) == 0x0002    # tie to even (2)


# -------------------------------------------------------------------- packing
def pin_pack_closed_forms(orc):
    """codes 0..7 along k -> 0x76543210; 8..15 -> 0xFEDCBA98; all 15 -> 0xFFFFFFFF."""
    W = _f16_exact(np.arange(16, dtype=np.float64)[:, None] * np.ones((1, 3)))
    packed, scales, zeros = orc.quantize_pack(W, group=16)
    assert packed[:, 0].tolist() == [0x76543210, 0xFEDCBA98]
    assert scales.view(np.uint16)[0, 0] == 0x3C00 and zeros.view(np.uint16)[0, 0] == 0
    W15 = _f16_exact(np.full((8, 2), 15.0))
    p15, s15, z15 = orc.quantize_pack(W15, group=8)
    assert p15.tolist() == [[0xFFFFFFFF, 0xFFFFFFFF]]
    assert s15.view(np.uint16).tolist() == [[0x3C00, 0x3C00]]


def pin_pack_roundtrip(orc):
    """unpack(pack(q)) == q on random weights (codes from the oracle's own
    quantizer), and every code appears in every nibble position."""
    W = _f16_exact(((np.arange(16)[:, None] + np.arange(16)[None, :]) % 16).astype(np.float64))
    packed, _, _, q = orc.quantize_pack(W, group=16, return_codes=True)
    assert np.array_equal(q, ((np.arange(16)[:, None] + np.arange(16)[None, :]) % 16))
    # independent numpy unpack of the words
    np_unpack = np.stack([(packed >> np.uint32(4 * j)) & np.uint32(15) for j in range(8)], axis=1)
    np_unpack = np_unpack.reshape(16, 16)
    assert np.array_equal(np_unpack, q)
    assert np.array_equal(orc.unpack(packed), q)
    Wr = synth.weight(256, 24, seed=99)
    pr, _, _, qr = orc.quantize_pack(Wr, group=128, return_codes=True)
    assert np.array_equal(orc.unpack(pr), qr)


# --------------------------------------------------------------- hand-worked
def pin_golden_8x8(orc):
    g = json.load(open(os.path.join(GOLDEN, "hand_8x8_g8.json")))
    K, N = g["K"], g["N"]
    W = np.zeros((K, N))
    for n, col in g["columns"].items():
        n = int(n)
        if "w" in col:
            W[:, n] = col["w"]
        elif "w_times_2^10" in col:
            W[:, n] = np.array(col["w_times_2^10"], dtype=np.float64) * 2.0 ** -10
        else:
            W[:, n] = np.array(col["w_times_2^24"], dtype=np.float64) * 2.0 ** -24
    Wh = _f16_exact(W)
    packed, scales, zeros = orc.quantize_pack(Wh, group=g["group"])
    assert [int(v) for v in packed[0]] == [int(h, 16) for h in g["packed_hex"]]
    assert scales.view(np.uint16)[0].tolist() == [_hex16(h) for h in g["scales_hex"]]
    assert zeros.view(np.uint16)[0].tolist() == [_hex16(h) for h in g["zeros_hex"]]
    wdq = orc.dequant(packed, scales, zeros, group=g["group"]).view(np.uint16)
    for n, col in g["wdq_hex_by_column"].items():
        assert wdq[:, int(n)].tolist() == [_hex16(h) for h in col], n
    for n in g["wdq_equals_w_columns"]:
        assert np.array_equal(wdq[:, n], Wh.view(np.uint16)[:, n]), n


def pin_golden_zero_from_rounded_scale(orc):
    g = json.load(open(os.path.join(GOLDEN, "hand_8x1_zero_from_rounded_scale.json")))
    Wh = _f16_exact(np.array(g["w"], dtype=np.float64)[:, None])
    packed, scales, zeros = orc.quantize_pack(Wh, group=g["group"])
    assert int(packed[0, 0]) == int(g["packed_hex"], 16)
    assert int(scales.view(np.uint16)[0, 0]) == _hex16(g["scale_hex"])
    assert int(zeros.view(np.uint16)[0, 0]) == _hex16(g["zero_hex"])
    wdq = orc.dequant(packed, scales, zeros, group=g["group"]).view(np.uint16)
    assert wdq[:, 0].tolist() == [_hex16(h) for h in g["wdq_hex"]]


def pin_golden_symmetric_8x4(orc):
    g = json.load(open(os.path.join(GOLDEN, "hand_8x4_g8_symmetric.json")))
    W = np.zeros((g["K"], g["N"]))
    for n, col in g["columns"].items():
        W[:, int(n)] = col["w"]
    packed, scales, zeros = orc.quantize_pack(_f16_exact(W), group=g["group"], symmetric=True)
    assert [int(v) for v in packed[0]] == [int(h, 16) for h in g["packed_hex"]]
    assert scales.view(np.uint16)[0].tolist() == [_hex16(h) for h in g["scales_hex"]]
    assert zeros.view(np.uint16)[0].tolist() == [_hex16(h) for h in g["zeros_hex"]]


def pin_symmetric_invariants(orc):
    """Symmetric quantizer on a random weight with outliers: z = 8 everywhere,
    the scale is the fp16 rounding of max|w| / 7 (checked with numpy's
    binary16), every code is within half a scale of w and never clipped, and
    the codes c = q - 8 are odd-symmetric: quantizing -W gives -c (the
    maximum magnitude maps to +-7, so -8 is never needed)."""
    W = synth.weight(512, 16, seed=41, outliers=True)
    packed, scales, zeros, q = orc.quantize_pack(W, group=128, return_codes=True, symmetric=True)
    assert np.all(zeros.view(np.uint16) == 0x4800)
    a = np.abs(W.astype(np.float64)).reshape(4, 128, 16).max(axis=1)
    assert np.array_equal(scales, (a / 7.0).astype(np.float16))
    s = np.repeat(scales.astype(np.float64), 128, axis=0)
    c = q.astype(np.int64) - 8
    assert np.all(np.abs(W.astype(np.float64) - c * s) <= s / 2 * (1 + 1e-12))
    assert c.min() >= -7 and c.max() <= 7
    _, _, _, qn = orc.quantize_pack(-W, group=128, return_codes=True, symmetric=True)
    assert np.array_equal(qn.astype(np.int64) - 8, -c)


def _hand_128x4():
    K = 128
    W = np.zeros((K, 4))
    k = np.arange(K)
    W[:, 0] = (k % 16 - 8) * 0.125
    W[:, 1] = -3.0
    cyc2 = [0.125, 0.375, -0.125, -0.375, 0.625, -0.625]
    W[0, 2], W[1, 2] = -0.75, 3.0
    W[2:, 2] = [cyc2[(kk - 2) % 6] for kk in range(2, K)]
    cyc3 = [0.5, 2.0, 1.0, 1.5]
    W[:, 3] = [cyc3[kk % 4] for kk in range(K)]
    return _f16_exact(W)


def pin_golden_128x4(orc):
    g = json.load(open(os.path.join(GOLDEN, "hand_128x4_g128.json")))
    Wh = _hand_128x4()
    packed, scales, zeros = orc.quantize_pack(Wh, group=128)
    assert scales.view(np.uint16)[0].tolist() == [_hex16(h) for h in g["scales_hex"]]
    assert zeros.view(np.uint16)[0].tolist() == [_hex16(h) for h in g["zeros_hex"]]
    ev, od = [int(h, 16) for h in g["packed_hex_col0_even_odd"]]
    assert packed[:, 0].tolist() == [ev if r % 2 == 0 else od for r in range(16)]
    assert packed[:, 1].tolist() == [int(g["packed_hex_col1"], 16)] * 16
    rows2 = g["packed_hex_col2_rows_r_mod3"]
    want2 = [int(g["packed_hex_col2_row0"], 16)] + [int(rows2[str(r % 3)], 16)
                                                    for r in range(1, 16)]
    assert packed[:, 2].tolist() == want2
    assert packed[:, 3].tolist() == [int(g["packed_hex_col3"], 16)] * 16
    wdq = orc.dequant(packed, scales, zeros, group=128)
    wb = wdq.view(np.uint16)
    assert np.array_equal(wb[:, 0], Wh.view(np.uint16)[:, 0])
    assert set(wb[:, 1].tolist()) == {_hex16(g["wdq_hex_col1"])}
    q2 = orc.unpack(packed)[:, 2]
    for kk in range(128):
        assert wb[kk, 2] == _hex16(g["wdq_hex_col2_by_code"][str(int(q2[kk]))])
        assert wb[kk, 3] == _hex16(g["wdq_hex_col3_by_w"][repr(float(Wh[kk, 3]))])


# ------------------------------------------------------------- closed forms
def pin_dequant_closed_form(orc):
    """Wdq == fp16((q - z) * s) computed with numpy, and |w - (q-z)s| <= s/2 on
    every entry whose code is not clipped."""
    for seed, outl in ((5, False), (6, True)):
        W = synth.weight(512, 64, seed=seed, outliers=outl)
        packed, scales, zeros, q = orc.quantize_pack(W, group=128, return_codes=True)
        s = np.repeat(scales.astype(np.float64), 128, axis=0)
        z = np.repeat(zeros.astype(np.float64), 128, axis=0)
        want = ((q.astype(np.float64) - z) * s).astype(np.float16)
        got = orc.dequant(packed, scales, zeros, group=128)
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
        w = W.astype(np.float64)
        unclipped = (np.rint(w / s) + z > 0) & (np.rint(w / s) + z < 15)
        err = np.abs(w - (q - z) * s)
        assert np.all(err[unclipped] <= s[unclipped] / 2)
        # min and max of every group are reproduced to within s/2 as well
        assert np.all(z >= 0) and np.all(z <= 15) and np.all(z == np.rint(z))


def pin_gemm_one_hot(orc):
    """x = e_k picks row k of the dequantized weight exactly."""
    W = synth.weight(256, 40, seed=11)
    packed, scales, zeros = orc.quantize_pack(W, group=128)
    wdq = orc.dequant(packed, scales, zeros, group=128).astype(np.float64)
    for kk in (0, 1, 7, 8, 127, 128, 200, 255):
        x = np.zeros((1, 256), dtype=np.float16)
        x[0, kk] = 1.0
        out = orc.gemm(x, packed, scales, zeros, group=128)
        assert np.array_equal(out[0], wdq[kk]), kk


def pin_gemm_linear(orc):
    """x = 0 gives 0; doubling x doubles the output exactly; a matmul of numpy on
    the dequantized weight agrees to fp64 rounding."""
    W = synth.weight(384, 24, seed=12)
    packed, scales, zeros = orc.quantize_pack(W, group=128)
    x = synth.activations(3, 384, seed=13)
    out = orc.gemm(x, packed, scales, zeros, group=128)
    out2 = orc.gemm((x.astype(np.float32) * 2).astype(np.float16), packed, scales, zeros, 128)
    assert np.array_equal(out2, 2 * out)
    assert not np.any(orc.gemm(np.zeros_like(x), packed, scales, zeros, 128))
    wdq = orc.dequant(packed, scales, zeros, group=128).astype(np.float64)
    ref = x.astype(np.float64) @ wdq
    assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def pin_brute_force(orc):
    """The pure-Python brute force (struct fp16, exact Fraction sums) agrees:
    bit-exact encoding, GEMM to fp64 rounding."""
    rng = np.random.Generator(np.random.PCG64(2024))
    for (M, K, N, grp) in ((1, 8, 3, 8), (3, 64, 5, 32), (2, 256, 8, 128), (3, 128, 4, 64)):
        W = (rng.standard_normal((K, N)) * 0.02).astype(np.float16)
        x = rng.standard_normal((M, K)).astype(np.float16)
        Wl = W.astype(np.float64).tolist()
        bp, bs, bz, bq = brute.quantize_pack(Wl, grp)
        packed, scales, zeros = orc.quantize_pack(W, group=grp)
        assert packed.tolist() == bp
        assert scales.astype(np.float64).tolist() == bs
        assert zeros.astype(np.float64).tolist() == bz
        bw = brute.dequant(bq, bs, bz, grp)
        wdq = orc.dequant(packed, scales, zeros, group=grp)
        assert wdq.astype(np.float64).tolist() == bw
        bref = np.array(brute.gemm(x.astype(np.float64).tolist(), bw))
        ref = orc.gemm(x, packed, scales, zeros, group=grp)
        assert np.max(np.abs(ref - bref)) <= 1e-13 * max(1.0, float(np.max(np.abs(bref))))


# ------------------------------------------------------- pre-permuted layout
def _fixture_inputs(case):
    K, N, group = case["K"], case["N"], case["group"]
    packed = np.zeros((K // 8, N), dtype=np.uint32)
    G = K // group
    jj, nn = np.meshgrid(np.arange(G), np.arange(N), indexing="ij")
    if case["N"] == 64:            # third case: every nibble of a word equal
        rr, cc = np.meshgrid(np.arange(K // 8), np.arange(N), indexing="ij")
        packed[:] = (0x11111111 * ((rr + cc) % 16)).astype(np.uint32)
        scales = (0x3C00 + 64 * jj + nn).astype(np.uint16)
        zeros = (0x4000 + 64 * jj + nn).astype(np.uint16)
    else:
        scales = (0x3C00 + 32 * jj + nn).astype(np.uint16)
        zeros = (0x4000 + 32 * jj + nn).astype(np.uint16)
    for w in case["words"]:
        packed[w["r"], w["n"]] = int(w["natural"], 16)
    return packed, scales, zeros


def pin_golden_permuted_layout(orc):
    """Hand-worked positions and values of the repacked layout (words, nibble
    order, scale/zero halves) for groups 128, 512 and 32; every word not listed
    is zero (the first two cases) and the inverse map restores the input."""
    with open(os.path.join(GOLDEN, "permuted_layout_hand.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        K, N, group = case["K"], case["N"], case["group"]
        packed, scales, zeros = _fixture_inputs(case)
        words = orc.permute(packed, scales.view(np.float16), zeros.view(np.float16), group)
        halves = words.view(np.uint16)
        for w in case["words"]:
            assert int(words[w["index"]]) == int(w["repacked"], 16), (case["group"], w)
        for h in case["halves"]:
            assert int(halves[h["half_index"]]) == int(h["bits"], 16), (case["group"], h)
        if N == 32:
            gps = 256 // group if group < 256 else 1
            bw = 1024 + 32 * gps
            listed = {w["index"] for w in case["words"]}
            for b in range(words.size // bw):
                blk = words[b * bw:b * bw + 1024]
                nz = set((np.nonzero(blk)[0] + b * bw).tolist())
                assert nz <= listed, sorted(nz - listed)[:4]
        back = orc.unpermute(words, K, N, group)
        assert np.array_equal(back[0], packed)
        assert np.array_equal(back[1].view(np.uint16), scales)
        assert np.array_equal(back[2].view(np.uint16), zeros)


def _permute_numpy(packed, scales, zeros, group):
    """The same layout written as an axis permutation of numpy arrays (an
    independent restatement of the index map)."""
    K8, N = packed.shape
    K = K8 * 8
    KB, S = K // 256, N // 32
    gps = 256 // group if group < 256 else 1
    # packed rows r = 32 kb + 4 u8 + t, columns n = 32 sn + 4 g + c
    p6 = packed.reshape(KB, 8, 4, S, 8, 4)                  # kb, u8, t, sn, g, c
    words = p6.transpose(3, 0, 1, 4, 2, 5).reshape(S, KB, 1024)   # sn, kb, (u8, g, t, c)
    nib = [(words >> np.uint32(4 * q)) & np.uint32(15) for q in range(8)]
    rep = np.zeros_like(words)
    for p in range(8):
        rep |= nib[2 * (p % 4) + p // 4] << np.uint32(4 * p)
    # scales / zeros of group rows 256 kb / group + gi
    rows = (np.arange(KB)[:, None] * 256 // group + np.arange(gps)[None, :])   # kb, gi
    sc = scales.view(np.uint16)[rows].reshape(KB, gps, S, 8, 4)             # kb, gi, sn, g, c
    ze = zeros.view(np.uint16)[rows].reshape(KB, gps, S, 8, 4)
    sz = np.concatenate([sc, ze], axis=-1)                                    # kb, gi, sn, g, 8
    sz = sz.transpose(2, 0, 1, 3, 4).reshape(S, KB, gps * 64)                 # sn, kb, halves
    sz_words = np.ascontiguousarray(sz).view(np.uint32)                       # sn, kb, 32 gps
    return np.concatenate([rep, sz_words], axis=2).reshape(-1)


def pin_permuted_layout_numpy(orc):
    """The C map equals the numpy axis-permutation restatement on random words,
    for every supported group size, and the inverse restores the input."""
    rng = np.random.default_rng(2024)
    for K, N, group in [(256, 32, 128), (512, 64, 32), (1024, 96, 64), (768, 32, 256),
                        (1024, 64, 512), (2048, 32, 1024)]:
        packed = rng.integers(0, 2 ** 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
        scales = rng.integers(0, 2 ** 16, size=(K // group, N), dtype=np.uint64).astype(np.uint16)
        zeros = rng.integers(0, 16, size=(K // group, N)).astype(np.uint16)
        words = orc.permute(packed, scales.view(np.float16), zeros.view(np.float16), group)
        assert np.array_equal(words, _permute_numpy(packed, scales, zeros, group)), (K, N, group)
        back = orc.unpermute(words, K, N, group)
        assert np.array_equal(back[0], packed)
        assert np.array_equal(back[1].view(np.uint16), scales)
        assert np.array_equal(back[2].view(np.uint16), zeros)


# ------------------------------------------------------------------ bfloat16
def _bf16_from_f32_bits(u32: np.ndarray) -> np.ndarray:
    """Independent bfloat16 rounding of float32 values: round to nearest even on
    the integer bit pattern (the upper 16 bits, plus one when the dropped half
    is above the midpoint or at it with an odd kept part)."""
    u = u32.astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def pin_bf16_decode_exhaustive(orc):
    """Every bfloat16 pattern decodes to the float32 whose upper 16 bits it is."""
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([orc.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def pin_bf16_encode(orc):
    """bfloat16 encoding, round to nearest even: finite patterns round-trip,
    midpoints go to the even neighbour, and random float32 values (subnormal
    to huge) match the integer rounding of their bit patterns."""
    for b in list(range(0, 0x7f80, 7)) + [0x0001, 0x007f, 0x0080, 0x7f7f]:
        v = float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])
        assert orc.double_to_bf16(v) == b, hex(b)
        assert orc.double_to_bf16(-v) == (b | 0x8000) or v == 0.0, hex(b)
    for b in range(0, 0x7f7f, 13):
        lo = float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])
        hi = float(np.array([(b + 1) << 16], dtype=np.uint32).view(np.float32)[0])
        mid = (lo + hi) / 2                     # exact in fp64
        even = b if b % 2 == 0 else b + 1
        assert orc.double_to_bf16(mid) == even, hex(b)
    rng = np.random.Generator(np.random.PCG64(77))
    u = rng.integers(0, 0x7f800000, size=20000, dtype=np.uint64).astype(np.uint32)
    ref = _bf16_from_f32_bits(u)
    vals = u.view(np.float32).astype(np.float64)
    got = np.array([orc.double_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    assert orc.double_to_bf16(3.5e38) == 0x7f80          # past the largest finite: inf


def pin_golden_bf16_8x4(orc):
    """The hand-worked bfloat16 example: codes, scales, zeros and every
    dequantized weight (including a rounding tie) bit for bit."""
    with open(os.path.join(GOLDEN, "hand_8x4_g8_bf16.json")) as f:
        fx = json.load(f)
    W = np.array([[int(v, 16) for v in r] for r in fx["w_bits"]], dtype=np.uint16)
    packed, scales, zeros = orc.quantize_pack_bf16(W, fx["group"])
    assert [int(v) for v in packed[0]] == [int(v, 16) for v in fx["packed"]]
    assert [int(v) for v in scales[0]] == [int(v, 16) for v in fx["scales"]]
    assert [int(v) for v in zeros[0]] == [int(v, 16) for v in fx["zeros"]]
    wdq = orc.dequant_bf16(packed, scales, zeros, fx["group"])
    assert np.array_equal(wdq, np.array([[int(v, 16) for v in r] for r in fx["wdq"]],
                                        dtype=np.uint16))


def pin_bf16_code_ties(orc):
    """Codes at exact ties of w / s, worked by hand: the group [-1, 14, 0.5,
    1.5, 2.5, -0.5, 0, 7.5] has s = 15 / 15 = 1 and z = rint(1 / 1) = 1, and
    q = rint(w / s) + z rounds each half-integer w / s to the even integer
    before the zero is added: codes [0, 15, 1, 3, 3, 1, 1, 9]."""
    w = np.array([-1.0, 14.0, 0.5, 1.5, 2.5, -0.5, 0.0, 7.5], dtype=np.float32)
    bits = (w.view(np.uint32) >> 16).astype(np.uint16).reshape(8, 1)
    packed, scales, zeros = orc.quantize_pack_bf16(bits, 8)
    assert int(scales[0, 0]) == 0x3F80 and int(zeros[0, 0]) == 0x3F80   # s = 1, z = 1
    codes = [(int(packed[0, 0]) >> (4 * k)) & 15 for k in range(8)]
    assert codes == [0, 15, 1, 3, 3, 1, 1, 9], codes


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_bf16_gemm(orc):
    """The bfloat16 GEMM: one-hot rows of x return the dequantized rows exactly,
    and a random x agrees with numpy's matmul of the bf16 values; the quantizer
    keeps |w - (q - z) s| <= s/2 for unclipped entries."""
    K, N, M, g = 256, 24, 5, 64
    W = synth.weight_bf16(K, N, seed=88)
    packed, scales, zeros, q = orc.quantize_pack_bf16(W, g, return_codes=True)
    s = np.repeat(_bf16_values(scales), g, axis=0)
    z = np.repeat(_bf16_values(zeros), g, axis=0)
    w = _bf16_values(W)
    err = np.abs(w - (q.astype(np.float64) - z) * s)
    inside = (q > 0) & (q < 15)
    assert np.all(err[inside] <= s[inside] / 2 + 1e-12)
    wdq = _bf16_values(orc.dequant_bf16(packed, scales, zeros, g))
    ks = [0, 7, 100, 255, 64]
    x = np.zeros((len(ks), K), dtype=np.uint16)
    x[np.arange(len(ks)), ks] = 0x3F80                    # bfloat16 1.0
    ref = orc.gemm_bf16(x, packed, scales, zeros, g)
    assert np.array_equal(ref, wdq[ks])
    xr = synth.activations_bf16(M, K, seed=89)
    ref = orc.gemm_bf16(xr, packed, scales, zeros, g)
    assert np.allclose(ref, _bf16_values(xr) @ wdq, rtol=1e-12, atol=1e-12)


ALL_PINS = [
    pin_half_decode_exhaustive,
    pin_half_encode,
    pin_pack_closed_forms,
    pin_pack_roundtrip,
    pin_golden_8x8,
    pin_golden_128x4,
    pin_golden_zero_from_rounded_scale,
    pin_golden_symmetric_8x4,
    pin_symmetric_invariants,
    pin_dequant_closed_form,
    pin_gemm_one_hot,
    pin_gemm_linear,
    pin_brute_force,
    pin_golden_permuted_layout,
    pin_permuted_layout_numpy,
    pin_bf16_decode_exhaustive,
    pin_bf16_encode,
    pin_golden_bf16_8x4,
    pin_bf16_code_ties,
    pin_bf16_gemm,
]
