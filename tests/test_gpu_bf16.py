"""Parity of the bfloat16 variant (x, scales, zeros and out in bfloat16) with
the oracle's bfloat16 functions, through the C ABI.

Bars: packing, scales, zeros and dequantized weights bit-exact; GEMM outputs
max |out - ref| / max(1, |ref|) <= 5e-3 elementwise (the same bar as fp16:
the kernels multiply x by the exactly dequantized bfloat16 weight, so the
difference from the fp64 reference is fp32 accumulation plus one bfloat16
rounding of the output, at most 2^-9 of |out|); one-hot activations give the
dequantized row bit-exactly.  Shapes: the five workloads (tiny, square decode,
FFN with outliers, MoE experts, prefill sweep), with ragged tails and other
group sizes.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_codes_gb300 as w4
from weight_only_int4_codes_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 5e-3
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def bf_dev(bits):
    """uint16 bfloat16 bit patterns -> a bfloat16 CUDA tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(DEV)


def bits_of(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def values_of(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def i32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(DEV)


def quantize_both(Wb, group):
    ref = oracle.quantize_pack_bf16(Wb, group)
    got = w4.quantize_pack_bf16(bf_dev(Wb), group)
    torch.cuda.synchronize()
    assert np.array_equal(got[0].cpu().numpy().view(np.uint32), ref[0]), "packed words differ"
    assert np.array_equal(bits_of(got[1]), ref[1]), "scales differ"
    assert np.array_equal(bits_of(got[2]), ref[2]), "zeros differ"
    return got, ref


@functools.lru_cache(maxsize=4)
def quantized(K, N, group, seed, outliers=False):
    Wb = synth.weight_bf16(K, N, seed=seed, outliers=outliers)
    dev_w, ref_w = quantize_both(Wb, group)
    return dev_w, ref_w


def check_gemm(xb, dev_w, ref_w, group, config=None, tol=TOL):
    out = w4.gemm_ex(bf_dev(xb), *dev_w, group=group, config=config)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    assert w4.kernel_status() == 0
    ref = oracle.gemm_bf16(xb, *ref_w, group=group)
    err = oracle.rel_err(values_of(bits_of(out)), ref)
    assert err <= tol, "rel err %.3g > %g (M=%d, config=%s)" % (err, tol, xb.shape[0], config)
    return out


# ----------------------------------------------------------------- packing
@pytest.mark.parametrize("K,N,group,outliers", [
    (512, 256, 128, False),      # tiny correctness case
    (4096, 4096, 128, False),    # decode square projection
    (4096, 14336, 128, True),    # FFN gate/up with outliers (also the first prefill shape)
    (14336, 4096, 128, True),    # FFN down with outliers
    (2048, 768, 128, False),     # MoE expert
    (768, 2048, 128, False),
    (256, 260, 128, False),      # ragged N
    (256, 64, 32, False),        # other group sizes
    (512, 96, 64, True),
    (1024, 128, 256, False),
])
def test_quantize_pack_and_dequantize_bf16_bit_exact(K, N, group, outliers):
    dev_w, ref_w = quantized(K, N, group, synth.weight_seed(1) + K + N, outliers)
    wdq = w4.dequantize_bf16(*dev_w, group=group)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(wdq), oracle.dequant_bf16(*ref_w, group=group))


def test_quantize_bf16_prefill_size_sampled_columns():
    """K=8192, N=28672 (the largest prefill weight): packed words, scales and
    zeros of 64 sampled columns against the oracle on those columns."""
    K, N = 8192, 28672
    Wb = synth.weight_bf16(K, N, seed=synth.weight_seed(4, shape_index=1))
    packed, scales, zeros = w4.quantize_pack_bf16(bf_dev(Wb), 128)
    torch.cuda.synchronize()
    cols = np.sort(np.random.Generator(np.random.PCG64(5)).choice(N, 64, replace=False))
    ref = oracle.quantize_pack_bf16(np.ascontiguousarray(Wb[:, cols]), 128)
    assert np.array_equal(packed.cpu().numpy().view(np.uint32)[:, cols], ref[0])
    assert np.array_equal(bits_of(scales)[:, cols], ref[1])
    assert np.array_equal(bits_of(zeros)[:, cols], ref[2])


def test_quantize_bf16_special_columns():
    """Constant, zero, all-positive, all-negative, huge and tiny (subnormal
    scale) groups: the degenerate scale 1.0, clamped zeros and the double ->
    bfloat16 rounding of the scale in every binade."""
    K, N = 256, 16
    v = synth._draw_weight(K, N, seed=3, outliers=False, std=0.02)
    v[:, 0] = 0.0
    v[:, 1] = -3.0
    v[:, 2] = np.abs(v[:, 2]) + 1.0
    v[:, 3] = -np.abs(v[:, 3]) - 1.0
    v[:, 4] *= np.float32(1e30)
    v[:, 5] *= np.float32(1e-36)          # scale in the bfloat16 subnormal range
    v[:, 6] *= np.float32(1e-39)
    v[:128, 7] = 5.0                      # one constant group, one random
    Wb = synth.bf16_bits(v)
    dev_w, ref_w = quantize_both(Wb, 128)
    wdq = w4.dequantize_bf16(*dev_w, group=128)
    torch.cuda.synchronize()
    assert np.array_equal(bits_of(wdq), oracle.dequant_bf16(*ref_w, group=128))


# -------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("K,N,outliers", [
    (512, 256, False), (4096, 4096, False), (2048, 768, False), (768, 2048, False),
    (4096, 14336, True), (14336, 4096, True),
])
def test_gemm_bf16_decode_configs(K, N, outliers, M):
    dev_w, ref_w = quantized(K, N, 128, synth.weight_seed(1) + K + N, outliers)
    xb = synth.activations_bf16(M, K, seed=synth.x_seed(1, M) + K)
    check_gemm(xb, dev_w, ref_w, 128)


@pytest.mark.parametrize("cfg", [
    dict(path="decode", variant="registers", split_k=1, warps_k=8, warps_n=1),
    dict(path="decode", variant="registers", split_k=3, warps_k=4, warps_n=1),
    dict(path="decode", variant="registers", split_k=2, warps_k=4, warps_n=2),
    dict(path="decode", variant="registers", split_k=1, warps_k=2, warps_n=4),
    dict(path="decode", variant="registers", split_k=4, warps_k=2, warps_n=2),
])
@pytest.mark.parametrize("M", [1, 3, 9, 16])
def test_gemm_bf16_decode_launch_shapes(cfg, M):
    K, N = 2048, 776                      # ragged last column tile
    dev_w, ref_w = quantized(K, N, 128, 71, True)
    xb = synth.activations_bf16(M, K, seed=72 + M)
    check_gemm(xb, dev_w, ref_w, 128, config=cfg)


@pytest.mark.parametrize("cfg", [
    dict(path="decode", variant="tma", warps_k=4, warps_n=2),
    dict(path="decode", variant="tma", warps_k=8, warps_n=4, split_k=3),
    dict(path="decode", variant="tma", warps_k=16, warps_n=2, split_k=8),
    dict(path="decode", variant="tma", warps_k=4, warps_n=4, split_k=2, pdl=True),
])
@pytest.mark.parametrize("M", [1, 5, 9, 16])
def test_gemm_bf16_decode_tma(cfg, M):
    """The TMA decode kernel's bfloat16 instantiations: every consumer count,
    tile width and several cluster sizes; a ragged last column tile."""
    K, N = 2048, 776
    dev_w, ref_w = quantized(K, N, 128, 71, True)
    xb = synth.activations_bf16(M, K, seed=76 + M)
    check_gemm(xb, dev_w, ref_w, 128, config=cfg)


@pytest.mark.parametrize("group", [32, 64, 256])
@pytest.mark.parametrize("M", [1, 12])
def test_gemm_bf16_tma_groups(group, M):
    K, N = 2048, 512
    dev_w, ref_w = quantized(K, N, group, 81 + group, False)
    xb = synth.activations_bf16(M, K, seed=83 + M)
    check_gemm(xb, dev_w, ref_w, group, config=dict(path="decode", variant="tma"))


@pytest.mark.parametrize("group", [32, 64, 256, 512])
@pytest.mark.parametrize("M", [1, 12])
def test_gemm_bf16_other_groups(group, M):
    K, N = 2048, 512
    dev_w, ref_w = quantized(K, N, group, 81 + group, False)
    xb = synth.activations_bf16(M, K, seed=82 + M)
    check_gemm(xb, dev_w, ref_w, group)


@pytest.mark.parametrize("M", [17, 48, 128, 256, 300, 600])
@pytest.mark.parametrize("K,N", [(1024, 512), (512, 1000), (2048, 392)])
def test_gemm_bf16_prefill(K, N, M):
    dev_w, ref_w = quantized(K, N, 128, 91 + K + N, True)
    xb = synth.activations_bf16(M, K, seed=92 + M)
    check_gemm(xb, dev_w, ref_w, 128)


@pytest.mark.parametrize("config", [
    dict(path="prefill", tile_m=16), dict(path="prefill", tile_m=64),
    dict(path="prefill", tile_m=128, warps_k=8), dict(path="prefill", tile_m=256, warps_k=4),
    dict(path="prefill", tile_m=256, warps_k=16), dict(path="prefill", tile_m=64, split_k=3),
    dict(path="prefill", tile_m=128, split_k=2, warps_k=8),
])
def test_gemm_bf16_prefill_kernels(config):
    """Both tcgen05 kernels (one ring, split ring), every dequantizing-warp
    count, split-K clusters; K with a group boundary inside a 128-k stage."""
    K, N = 1088, 264
    dev_w, ref_w = quantized(K, N, 64, 95, True)
    xb = synth.activations_bf16(300, K, seed=96)
    check_gemm(xb, dev_w, ref_w, 64, config=config)


def test_gemm_bf16_prefill_full_size_sampled():
    """The prefill workloads in bfloat16: K=8192, N=28672 at M=4096 and K=4096,
    N=14336 at M=1024 through the automatic dispatch, every row and 48 sampled
    columns against the oracle."""
    for (K, N, M, si) in ((8192, 28672, 4096, 1), (4096, 14336, 1024, 0)):
        Wb = synth.weight_bf16(K, N, seed=synth.weight_seed(4, shape_index=si))
        dev_w = w4.quantize_pack_bf16(bf_dev(Wb), 128)
        cols = np.sort(np.random.Generator(np.random.PCG64(11)).choice(N, 48, replace=False))
        ref_w = oracle.quantize_pack_bf16(np.ascontiguousarray(Wb[:, cols]), 128)
        del Wb
        xb = synth.activations_bf16(M, K, seed=synth.x_seed(4, M, shape_index=si))
        out = w4.gemm_ex(bf_dev(xb), *dev_w, group=128)
        torch.cuda.synchronize()
        assert w4.kernel_status() == 0
        ref = oracle.gemm_bf16(xb, *ref_w, group=128)
        err = oracle.rel_err(values_of(bits_of(out)[:, cols]), ref)
        assert err <= TOL, (K, N, M, err)


def test_gemm_bf16_random_encodings():
    """Arbitrary valid codes, bfloat16 scales and zeros (not from the quantizer)."""
    K, N = 2048, 512
    rng = np.random.Generator(np.random.PCG64(151))
    packed = rng.integers(0, 2**32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    scales = synth.bf16_bits(rng.random((K // 128, N), dtype=np.float32) * np.float32(0.004)
                             + np.float32(0.0005))
    zeros = synth.bf16_bits(rng.integers(0, 16, size=(K // 128, N)).astype(np.float32))
    dev_w = (i32_dev(packed), bf_dev(scales), bf_dev(zeros))
    for M in (1, 7, 16, 40):
        xb = synth.activations_bf16(M, K, seed=152 + M)
        check_gemm(xb, dev_w, (packed, scales, zeros), 128)


@pytest.mark.parametrize("M,config", [
    (1, None), (16, None), (9, dict(path="decode", variant="registers", warps_n=2, warps_k=4)),
    (3, dict(path="decode", variant="tma")), (12, dict(path="decode", variant="tma", warps_k=16)),
    (64, dict(path="prefill", tile_m=64)), (128, dict(path="prefill", tile_m=128)),
    (300, dict(path="prefill", tile_m=256)),
])
def test_bf16_one_hot_is_exact(M, config):
    """x = e_k: one nonzero product 1.0 * Wdq, exact in fp32, so out equals the
    bfloat16 dequantized row bit for bit on every kernel."""
    K, N = 1024, 768
    Wb = synth.weight_bf16(K, N, seed=161, outliers=True)
    dev_w, ref_w = quantize_both(Wb, 128)
    wdq = oracle.dequant_bf16(*ref_w, group=128)
    ks = np.array([0, 1, 7, 8, 127, 128, 500, 1023, 640, 64, 333, 900, 17, 256, 1000, 2])
    if M > len(ks):
        ks = np.random.Generator(np.random.PCG64(M)).integers(0, K, M)
    xb = np.zeros((M, K), dtype=np.uint16)
    xb[np.arange(M), ks[:M]] = 0x3F80          # 1.0
    out = w4.gemm_ex(bf_dev(xb), *dev_w, group=128, config=config)
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    assert np.array_equal(bits_of(out), wdq[ks[:M]])


@pytest.mark.parametrize("M", [4, 300])
def test_bf16_dirty_output_and_determinism(M):
    """out is overwritten, never accumulated into; repeated calls give the
    same bits; x = 0 gives +0."""
    K, N = 1024, 512
    dev_w, _ = quantized(K, N, 128, 171, False)
    xb = synth.activations_bf16(M, K, seed=172)
    x = bf_dev(xb)
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    a = bits_of(w4.gemm_ex(x, *dev_w, group=128, out=out)).copy()
    b = bits_of(w4.gemm_ex(x, *dev_w, group=128, out=out)).copy()
    assert np.array_equal(a, b)
    z = w4.gemm_ex(torch.zeros_like(x), *dev_w, group=128, out=out)
    torch.cuda.synchronize()
    assert np.all(bits_of(z) == 0)


def test_bf16_rejected_where_not_built():
    """The variants without a bfloat16 kernel refuse it (nothing enqueued)."""
    dev_w, _ = quantized(512, 256, 128, 181, False)
    x = bf_dev(synth.activations_bf16(4, 512, seed=182))
    for cfg in (dict(path="decode", variant="warp"), dict(path="decode", variant="stream"),
                dict(path="prefill", variant="smem", tile_m=64)):
        with pytest.raises(w4.W4A16Error) as e:
            w4.gemm_ex(x, *dev_w, group=128, config=cfg)
        assert e.value.status == 2
