"""Parity of the stream decode kernel (W4A16_DECODE_STREAM) and of the
repacked (pre-permuted) weight layout with the fp64 oracle, through the C ABI.

Bars as in test_gpu_parity.py: repacked words bit-exact with the oracle's map;
GEMM outputs max |out - ref| / max(1, |ref|) <= 5e-3 elementwise; one-hot
activations give the dequantized row bit-exactly; repeated calls give
identical bits (the cross-CTA sum of a shared tile runs in a fixed order).
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
STREAM = dict(path="decode", variant="stream")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@functools.lru_cache(maxsize=6)
def quantized(K, N, group, seed, outliers=False):
    """Seeded weight quantized by both sides; bit-exactness asserted."""
    W = synth.weight(K, N, seed=seed, outliers=outliers)
    ref = oracle.quantize_pack(W, group)
    got = w4.quantize_pack(to_dev(W), group)
    torch.cuda.synchronize()
    assert np.array_equal(got[0].cpu().numpy().view(np.uint32), ref[0])
    assert np.array_equal(got[1].cpu().numpy().view(np.uint16), ref[1].view(np.uint16))
    assert np.array_equal(got[2].cpu().numpy().view(np.uint16), ref[2].view(np.uint16))
    return got, ref


def oracle_ref(x, ref_w, group):
    return oracle.gemm(x, *ref_w, group=group)


def check(out, x, ref_w, group, what):
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    err = oracle.rel_err(out.cpu().numpy(), oracle_ref(x, ref_w, group))
    assert err <= TOL, "rel err %.3g > %g (%s)" % (err, TOL, what)


# ------------------------------------------------------- natural layout
@pytest.mark.parametrize("split", [1, 2])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("K,N,outliers", [
    (512, 256, False), (4096, 4096, False), (2048, 768, False), (768, 2048, False),
    (4096, 14336, True), (14336, 4096, True),
])
def test_stream_decode_configs(K, N, outliers, M, split):
    """The benchmark shapes at full size: whole tiles per CTA (split 1) and
    stream-K shares with the cross-CTA sum (split 2)."""
    dev_w, ref_w = quantized(K, N, 128, synth.weight_seed(1) + K + N, outliers)
    x = synth.activations(M, K, seed=synth.x_seed(1, M) + K)
    out = w4.gemm_ex(to_dev(x), *dev_w, group=128, config=dict(STREAM, split_k=split))
    check(out, x, ref_w, 128, "K=%d N=%d M=%d split=%d" % (K, N, M, split))


@pytest.mark.parametrize("cfg", [
    dict(warps_n=1, split_k=1), dict(warps_n=1, split_k=2), dict(warps_n=2, split_k=1),
    dict(warps_n=2, split_k=2), dict(warps_n=4, split_k=1), dict(warps_n=4, split_k=2),
    dict(warps_n=4, split_k=2, ctas=7), dict(warps_n=1, split_k=2, ctas=37),
    dict(warps_n=2, split_k=2, ctas=200), dict(warps_n=2, split_k=1, ctas=5),
    dict(pdl=True),
], ids=lambda c: "-".join("%s%s" % (k, v) for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 3, 9, 16])
def test_stream_launch_shapes(cfg, M):
    """Every tile width, both work splits, grids from 5 to 200 CTAs (tiles
    shared by up to many CTAs), ragged N (1000 = 31 tiles of 32 + 8) and a
    ragged last stage (K = 1536: 1.5 stages of 1024 k at warps_n = 1)."""
    K, N = 1536, 1000
    try:
        w4.plan(M, N, K, 128, **dict(STREAM, **cfg))
    except w4.W4A16Error as e:
        # one-strip tiles at M > 8 need more shared memory than a CTA may use
        assert e.status == 2 and M > 8 and cfg.get("warps_n") == 1
        pytest.skip("configuration not offered: %s" % e)
    dev_w, ref_w = quantized(K, N, 128, 21)
    x = synth.activations(M, K, seed=22 + M)
    out = w4.gemm_ex(to_dev(x), *dev_w, group=128, config=dict(STREAM, **cfg))
    check(out, x, ref_w, 128, str(cfg))


@pytest.mark.parametrize("cfg", [
    dict(warps_n=1, split_k=1), dict(warps_n=2, split_k=2), dict(warps_n=4, split_k=1),
    dict(warps_n=4, split_k=2, ctas=11), dict(warps_n=2, split_k=2, ctas=150),
], ids=lambda c: "-".join("%s%s" % (k, v) for k, v in c.items()))
@pytest.mark.parametrize("M", [1, 5, 16])
def test_stream_tma_boxes_ragged(cfg, M):
    """N % 32 == 0 takes the TMA-box layout: N = 1120 is 35 strips, so the last
    tile of 2 or 4 strips runs past N (its box reads zeros there), and K = 2304
    leaves a partial last stage for every tile width."""
    K, N = 2304, 1120
    try:
        w4.plan(M, N, K, 128, **dict(STREAM, **cfg))
    except w4.W4A16Error as e:
        assert e.status == 2 and M > 8 and cfg.get("warps_n") == 1
        pytest.skip("configuration not offered: %s" % e)
    dev_w, ref_w = quantized(K, N, 128, 23)
    x = synth.activations(M, K, seed=24 + M)
    out = w4.gemm_ex(to_dev(x), *dev_w, group=128, config=dict(STREAM, **cfg))
    check(out, x, ref_w, 128, str(cfg))


@pytest.mark.parametrize("group", [32, 64, 256, 512, 1024])
@pytest.mark.parametrize("M", [1, 12])
@pytest.mark.parametrize("split", [1, 2])
def test_stream_groups(group, M, split):
    K, N = 2048, 384
    dev_w, ref_w = quantized(K, N, group, 31 + group, True)
    x = synth.activations(M, K, seed=32)
    out = w4.gemm_ex(to_dev(x), *dev_w, group=group, config=dict(STREAM, split_k=split))
    check(out, x, ref_w, group, "group=%d" % group)


@pytest.mark.parametrize("cfg", [dict(split_k=1), dict(split_k=2), dict(split_k=2, ctas=33)])
@pytest.mark.parametrize("M", [1, 16])
def test_stream_one_hot_is_exact(cfg, M):
    """x = e_k: a single nonzero product per output, so out equals the
    dequantized row bit-exactly, including through the cross-CTA sum (the
    other partials are exact zeros)."""
    K, N = 1024, 768
    W = synth.weight(K, N, seed=61, outliers=True)
    ref_w = oracle.quantize_pack(W, 128)
    dev_w = w4.quantize_pack(to_dev(W), 128)
    wdq = oracle.dequant(*ref_w, group=128).view(np.uint16)
    ks = np.array([0, 1, 7, 8, 127, 128, 500, 1023, 640, 64, 333, 900, 17, 256, 1000, 2])[:M]
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = 1.0
    out = w4.gemm_ex(to_dev(x), *dev_w, group=128, config=dict(STREAM, **cfg))
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), wdq[ks])


@pytest.mark.parametrize("cfg", [dict(split_k=1), dict(split_k=2), dict(split_k=2, ctas=61)])
def test_stream_zero_dirty_output_determinism(cfg):
    """Every output element is overwritten (NaN-filled out), x = 0 gives
    exact zeros, and repeated calls (the scratch and its arrival counters
    reused) give identical bits."""
    K, N, M = 4096, 2048, 5
    dev_w, _ = quantized(K, N, 128, 73)
    c = dict(STREAM, **cfg)
    out = torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)
    w4.gemm_ex(torch.zeros((M, K), dtype=torch.float16, device=DEV), *dev_w, out=out, config=c)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    x = to_dev(synth.activations(M, K, seed=74))
    first = w4.gemm_ex(x, *dev_w, config=c).clone()
    for _ in range(5):
        again = w4.gemm_ex(x, *dev_w, out=torch.full_like(first, float("nan")), config=c)
        torch.cuda.synchronize()
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    assert w4.kernel_status() == 0


def test_stream_bounded_wait_times_out_and_reports():
    """A stage that is armed but never loaded: the consumers' bounded wait
    gives up, the status word reads W4A16_ERR_TIMEOUT, and the next call (which
    reuses the scratch counters) is correct."""
    K, N, M = 2048, 1024, 4
    dev_w, ref_w = quantized(K, N, 128, 45)
    x = synth.activations(M, K, seed=46)
    assert w4.kernel_status() == 0
    w4.gemm_ex(to_dev(x), *dev_w, group=128,
               config=dict(STREAM, split_k=1, flags=w4.native.FLAG_TEST_TIMEOUT))
    assert w4.kernel_status() == 5
    assert w4.kernel_status() == 0
    out = w4.gemm_ex(to_dev(x), *dev_w, group=128, config=dict(STREAM, split_k=2))
    check(out, x, ref_w, 128, "after timeout")


@pytest.mark.parametrize("split", [1, 2])
@pytest.mark.parametrize("M", [1, 16])
def test_stream_pdl_chain_reads_the_previous_output(split, M):
    """A chain of square GEMMs where each call's x is the previous call's out,
    launched with programmatic dependent launch inside a CUDA graph: every
    link waits for its input (compare with the same chain run call by call)."""
    K = N = 1024
    dev_w, ref_w = quantized(K, N, 128, 91)
    x0 = to_dev(synth.activations(M, K, seed=92) * np.float16(0.5))
    cfg = dict(STREAM, split_k=split, pdl=True)
    bufs = [torch.empty((M, N), dtype=torch.float16, device=DEV) for _ in range(6)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        w4.gemm_ex(x0, *dev_w, out=bufs[0], config=cfg)     # warm (plans, scratch)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        prev = x0
        for b in bufs:
            w4.gemm_ex(prev, *dev_w, out=b, config=cfg)
            prev = b
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    assert w4.kernel_status() == 0
    prev = x0
    for b in bufs:
        ref = w4.gemm_ex(prev, *dev_w, config=dict(STREAM, split_k=split))
        torch.cuda.synchronize()
        assert torch.equal(ref.view(torch.int16), b.view(torch.int16))
        prev = ref


def test_stream_two_streams_concurrently():
    """Calls on two streams at once use separate scratch buffers: both give
    the single-stream bits."""
    K, N, M = 4096, 4096, 8
    dev_w, _ = quantized(K, N, 128, 95)
    cfg = dict(STREAM, split_k=2)
    xa = to_dev(synth.activations(M, K, seed=96))
    xb = to_dev(synth.activations(M, K, seed=97))
    ra = w4.gemm_ex(xa, *dev_w, config=cfg).clone()
    rb = w4.gemm_ex(xb, *dev_w, config=cfg).clone()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for _ in range(20):
        with torch.cuda.stream(sa):
            oa = w4.gemm_ex(xa, *dev_w, config=cfg)
        with torch.cuda.stream(sb):
            ob = w4.gemm_ex(xb, *dev_w, config=cfg)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    for oa, ob in outs:
        assert torch.equal(oa.view(torch.int16), ra.view(torch.int16))
        assert torch.equal(ob.view(torch.int16), rb.view(torch.int16))


def expert_set(E, K, N, group, seed):
    ws, refs = [], []
    for e in range(E):
        W = synth.weight(K, N, seed=seed + e)
        refs.append(oracle.quantize_pack(W, group))
        ws.append(w4.quantize_pack(to_dev(W), group))
    return ws, refs


@pytest.mark.parametrize("split", [1, 2])
@pytest.mark.parametrize("E,M", [(1, 1), (3, 5), (64, 1), (64, 16), (7, 9)])
@pytest.mark.parametrize("K,N", [(2048, 768), (768, 2048)])
def test_stream_grouped_matches_oracle_per_expert(E, M, K, N, split):
    ws, refs = expert_set(E, K, N, 128, 500 + K)
    xs = [synth.activations(M, K, seed=600 + e) for e in range(E)]
    outs = w4.gemm_grouped([to_dev(v) for v in xs], [w[0] for w in ws], [w[1] for w in ws],
                           [w[2] for w in ws], config=dict(STREAM, split_k=split))
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    for e in range(E):
        err = oracle.rel_err(outs[e].cpu().numpy(), oracle.gemm(xs[e], *refs[e]))
        assert err <= TOL, "expert %d rel err %.3g" % (e, err)


def test_stream_grouped_whole_tiles_equal_single_launches_bitwise():
    """With whole tiles per CTA every output tile is summed the same way in a
    grouped launch as in a single launch: identical bits."""
    E, K, N, M = 5, 2048, 768, 4
    ws, _ = expert_set(E, K, N, 128, 700)
    xs = [to_dev(synth.activations(M, K, seed=710 + e)) for e in range(E)]
    cfg = dict(STREAM, split_k=1, warps_n=2)
    outs = w4.gemm_grouped(xs, [w[0] for w in ws], [w[1] for w in ws], [w[2] for w in ws],
                           config=cfg)
    for e in range(E):
        single = w4.gemm_ex(xs[e], *ws[e], config=cfg)
        torch.cuda.synchronize()
        assert torch.equal(single.view(torch.int16), outs[e].view(torch.int16))


# ------------------------------------------------------- repacked layout
@pytest.mark.parametrize("K,N,group", [
    (256, 32, 128), (512, 256, 128), (4096, 4096, 128), (2048, 768, 32), (768, 2048, 64),
    (1024, 96, 256), (2048, 64, 512), (3072, 160, 1024), (14336, 4096, 128),
])
def test_repack_bit_exact(K, N, group):
    """w4a16_repack against the oracle's index map, word for word."""
    dev_w, ref_w = quantized(K, N, group, 800 + K + group)
    rep = w4.repack(*dev_w, group=group)
    torch.cuda.synchronize()
    ref = oracle.permute(*ref_w, group=group)
    assert rep.numel() == ref.size * 4 == w4.repacked_bytes(K, N, group)
    assert np.array_equal(rep.cpu().numpy().view(np.uint32), ref)


def test_repack_rejects_unsupported_shapes():
    dev_w, _ = quantized(512, 40, 128, 801)          # N % 32 != 0
    assert w4.repacked_bytes(512, 40, 128) == 0
    with pytest.raises(w4.W4A16Error) as e:
        w4.repack(*dev_w, group=128)
    assert e.value.status == 2


@pytest.mark.parametrize("cfg", [dict(), dict(variant="stream"), dict(split_k=1), dict(split_k=2),
                                 dict(warps_n=1, split_k=2), dict(warps_n=4, split_k=1),
                                 dict(split_k=2, ctas=45), dict(pdl=True)],
                         ids=lambda c: "-".join("%s%s" % (k, v) for k, v in c.items()) or "auto")
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("K,N,outliers", [
    (4096, 4096, False), (4096, 14336, True), (14336, 4096, True), (2048, 768, False),
    (768, 2048, False), (512, 256, False),
])
def test_gemm_repacked_decode_configs(K, N, outliers, M, cfg):
    if M > 8 and cfg.get("warps_n") == 1:
        pytest.skip("one-strip tiles at M > 8 need more shared memory than a CTA may use")
    dev_w, ref_w = quantized(K, N, 128, synth.weight_seed(1) + K + N, outliers)
    rep = w4.repack(*dev_w, group=128)
    x = synth.activations(M, K, seed=synth.x_seed(1, M) + K)
    out = w4.gemm_repacked(to_dev(x), rep, N, group=128, config=dict(cfg) or None)
    check(out, x, ref_w, 128, "repacked K=%d N=%d M=%d %s" % (K, N, M, cfg))


@pytest.mark.parametrize("group", [32, 64, 256, 512, 1024])
@pytest.mark.parametrize("M", [1, 12])
def test_gemm_repacked_groups(group, M):
    K, N = 2048, 384
    dev_w, ref_w = quantized(K, N, group, 31 + group, True)
    rep = w4.repack(*dev_w, group=group)
    x = synth.activations(M, K, seed=33)
    out = w4.gemm_repacked(to_dev(x), rep, N, group=group)
    check(out, x, ref_w, group, "repacked group=%d" % group)


@pytest.mark.parametrize("M", [17, 40])
def test_gemm_repacked_larger_m_in_chunks(M):
    K, N = 1024, 512
    dev_w, ref_w = quantized(K, N, 128, 41)
    rep = w4.repack(*dev_w, group=128)
    x = synth.activations(M, K, seed=42)
    out = w4.gemm_repacked(to_dev(x), rep, N, group=128)
    check(out, x, ref_w, 128, "repacked M=%d" % M)


@pytest.mark.parametrize("M", [1, 16])
def test_gemm_repacked_one_hot_is_exact(M):
    K, N = 1024, 768
    W = synth.weight(K, N, seed=61, outliers=True)
    ref_w = oracle.quantize_pack(W, 128)
    dev_w = w4.quantize_pack(to_dev(W), 128)
    rep = w4.repack(*dev_w, group=128)
    wdq = oracle.dequant(*ref_w, group=128).view(np.uint16)
    ks = np.array([0, 1, 7, 8, 127, 128, 500, 1023, 640, 64, 333, 900, 17, 256, 1000, 2])[:M]
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = 1.0
    out = w4.gemm_repacked(to_dev(x), rep, N, group=128, config=dict(split_k=2))
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), wdq[ks])


@pytest.mark.parametrize("E,M", [(64, 1), (64, 16), (3, 7)])
@pytest.mark.parametrize("K,N", [(2048, 768), (768, 2048)])
def test_gemm_grouped_repacked(E, M, K, N):
    ws, refs = expert_set(E, K, N, 128, 900 + K)
    reps = [w4.repack(*w, group=128) for w in ws]
    xs = [synth.activations(M, K, seed=950 + e) for e in range(E)]
    outs = w4.gemm_grouped_repacked([to_dev(v) for v in xs], reps, N, group=128)
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    for e in range(E):
        err = oracle.rel_err(outs[e].cpu().numpy(), oracle.gemm(xs[e], *refs[e]))
        assert err <= TOL, "expert %d rel err %.3g" % (e, err)
