"""Plant plausible mistakes in copies of the oracle (on the CPU) and require
that at least one pin catches each one.  This shows the pins are strong enough
to detect a dropped term, a wrong sign or index, a wrong rounding rule or a
reversed operand anywhere in the oracle."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "w4a16_oracle.c")

# (name, text in the committed source, planted replacement)
MUTANTS = [
    ("nibble_order_reversed",
     "packed[(size_t)(k / 8) * N + n] |= q << (4 * (k % 8));",
     "packed[(size_t)(k / 8) * N + n] |= q << (4 * (7 - k % 8));"),
    ("hqq_style_rounding",
     "double qd = rint(w / s) + (double)z;",
     "double qd = rint(w / s + (double)z);"),
    ("half_away_rounding",
     "double qd = rint(w / s) + (double)z;",
     "double qd = round(w / s) + (double)z;"),
    ("scale_divisor_16",
     "oracle_double_to_half((mx - mn) / 15.0);",
     "oracle_double_to_half((mx - mn) / 16.0);"),
    ("zero_from_unrounded_scale",
     "double zr = rint(-mn / s);",
     "double zr = rint(-mn / ((mx - mn) / 15.0 + (mx == mn)));"),
    ("zero_not_clamped_high",
     "if (zr > 15.0) zr = 15.0;",
     "if (zr > 31.0) zr = 31.0;"),
    ("dequant_sign",
     "Wdq[(size_t)k * N + n] = oracle_double_to_half((q - z) * s);",
     "Wdq[(size_t)k * N + n] = oracle_double_to_half((q + z) * s);"),
    ("unpack_mask_3_bits",
     "(uint8_t)((packed[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 15u);",
     "(uint8_t)((packed[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 7u);"),
    ("gemm_drops_last_term",
     "for (int k = 0; k < K; ++k) acc += xm[k] * w[k];",
     "for (int k = 0; k < K - 1; ++k) acc += xm[k] * w[k];"),
    ("gemm_reversed_k",
     "for (int k = 0; k < K; ++k) acc += xm[k] * w[k];",
     "for (int k = 0; k < K; ++k) acc += xm[k] * w[K - 1 - k];"),
    ("codec_subnormal_threshold",
     "if (a < ldexp(1.0, -14)) {",
     "if (a < ldexp(1.0, -15)) {"),
    ("codec_truncates",
     "double m = rint(ldexp(f, 11));",
     "double m = floor(ldexp(f, 11));"),
    ("codec_decode_bias",
     "v = ldexp((double)(1024 + frac), expo - 25);",
     "v = ldexp((double)(1024 + frac), expo - 24);"),
    ("symmetric_missing_plus_8",
     "double cd = rint(w / s) + 8.0;",
     "double cd = rint(w / s);"),
    ("symmetric_divisor_8",
     "oracle_double_to_half(a / 7.0);",
     "oracle_double_to_half(a / 8.0);"),
    ("symmetric_max_not_absolute",
     "double w = fabs(oracle_half_to_double(W[(size_t)k * N + n]));",
     "double w = oracle_half_to_double(W[(size_t)k * N + n]);"),
    ("permute_lane_swaps_g_and_t",
     "int r = 32 * kb + 4 * u8 + L % 4;\n                        int n = 32 * sn + 4 * (L / 4) + c;\n                        blk[u8 * 128 + L * 4 + c] = permute_nibbles",
     "int r = 32 * kb + 4 * u8 + L / 8;\n                        int n = 32 * sn + 4 * (L % 8) + c;\n                        blk[u8 * 128 + L * 4 + c] = permute_nibbles"),
    ("permute_nibble_map_transposed",
     "uint32_t src = (uint32_t)(2 * (p % 4) + p / 4);",
     "uint32_t src = (uint32_t)(4 * (p % 2) + p / 2);"),
    ("permute_blocks_strip_inner",
     "uint32_t *blk = out + ((long long)sn * KB + kb) * BW;",
     "uint32_t *blk = out + ((long long)kb * (N / 32) + sn) * BW;"),
    ("permute_scale_zero_swapped",
     "sz[h] = scales[(size_t)j * N + n];\n                        sz[h + 4] = zeros[(size_t)j * N + n];",
     "sz[h] = zeros[(size_t)j * N + n];\n                        sz[h + 4] = scales[(size_t)j * N + n];"),
    ("permute_group_row_ignores_block",
     "int j = 256 * kb / group + gi;\n                        int n = 32 * sn + 4 * g + c;\n                        int h = (gi * 8 + g) * 8 + c;\n                        sz[h]",
     "int j = gi;\n                        int n = 32 * sn + 4 * g + c;\n                        int h = (gi * 8 + g) * 8 + c;\n                        sz[h]"),
    ("bf16_decode_bias",
     "v = ldexp((double)(128 + frac), expo - 134);",
     "v = ldexp((double)(128 + frac), expo - 133);"),
    ("bf16_encode_truncates",
     "double m = rint(ldexp(f, 8));",
     "double m = floor(ldexp(f, 8));"),
    ("bf16_subnormal_truncates",
     "double q = rint(ldexp(a, 133));",
     "double q = floor(ldexp(a, 133));"),
    ("bf16_scale_divisor_16",
     "uint16_t s_bits = oracle_double_to_bf16((mx - mn) / 15.0);",
     "uint16_t s_bits = oracle_double_to_bf16((mx - mn) / 16.0);"),
    ("bf16_degenerate_scale_fp16_pattern",
     "s_bits = 0x3f80;     /* 1.0 */",
     "s_bits = 0x3c00;     /* 1.0 */"),
    ("bf16_dequant_sign",
     "Wdq[(size_t)k * N + n] = oracle_double_to_bf16((q - z) * s);",
     "Wdq[(size_t)k * N + n] = oracle_double_to_bf16((z - q) * s);"),
    ("bf16_hqq_style_rounding",
     "double qv = rint(w / s) + (double)z;",
     "double qv = rint(w / s + (double)z);"),
    ("bf16_half_away_rounding",
     "double qv = rint(w / s) + (double)z;",
     "double qv = round(w / s) + (double)z;"),
    ("bf16_nibble_order_reversed",
     "packed[(size_t)(k / 8) * N + n] |= q << (4 * (k & 7));",
     "packed[(size_t)(k / 8) * N + n] |= q << (4 * (7 - (k & 7)));"),
    ("bf16_zero_not_clamped",
     "zq = zq < 0.0 ? 0.0 : (zq > 15.0 ? 15.0 : zq);",
     "zq = zq < 0.0 ? 0.0 : zq;"),
    ("bf16_gemm_drops_last_term",
     "for (int k = 0; k < K; ++k) sum += xm[k] * w[k];",
     "for (int k = 0; k < K - 1; ++k) sum += xm[k] * w[k];"),
    ("degenerate_scale_kept_zero",
     "s_bits = 0x3c00;     /* 1.0 */\n                s = 1.0;",
     "s_bits = 0x3c00;     /* 1.0 */\n                s = 1e-300;"),
]


@pytest.fixture(scope="module")
def source():
    return open(SRC).read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) == 1, "mutation anchor not unique: " + name
    mutated = source.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    lib = oracle.compile_source(str(src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception:  # any failure of a pin counts as detection
            caught.append(pin.__name__)
    assert caught, "no pin detects the planted mistake " + name
