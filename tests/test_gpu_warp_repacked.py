"""Parity of the warp-stream decode kernel on repacked weights
(w4a16_gemm_repacked / w4a16_gemm_grouped_repacked with W4A16_DECODE_WARP,
M <= 8) with the fp64 oracle: the decode workload shapes, every repacked group
size, grid sizes that give different runs per warp and split tiles, grouped
calls over many experts, one-hot exactness, dirty outputs, PDL chains and
run-to-run determinism; requests it cannot serve are refused."""
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
WARP = dict(path="decode", variant="warp")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@functools.lru_cache(maxsize=4)
def repacked(K, N, group, seed, outliers=False):
    W = synth.weight(K, N, seed=seed, outliers=outliers)
    ref_w = oracle.quantize_pack(W, group)
    dev_w = w4.quantize_pack(to_dev(W), group)
    rep = w4.repack(*dev_w, group=group)
    torch.cuda.synchronize()
    assert np.array_equal(rep.cpu().numpy().view(np.uint32), oracle.permute(*ref_w, group=group))
    return rep, ref_w


def check(out, x, ref_w, group, what):
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    err = oracle.rel_err(out.cpu().numpy(), oracle.gemm(x, *ref_w, group=group))
    assert err <= TOL, "rel err %.3g > %g (%s)" % (err, TOL, what)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("K,N,outliers", [
    (256, 32, False), (512, 256, False), (4096, 4096, False), (2048, 768, False),
    (768, 2048, False), (4096, 14336, True), (14336, 4096, True),
])
def test_warp_repacked_decode_configs(K, N, outliers, M):
    rep, ref_w = repacked(K, N, 128, synth.weight_seed(1) + K + N, outliers)
    x = synth.activations(M, K, seed=synth.x_seed(1, M) + K)
    xd = to_dev(x)
    out = w4.gemm_repacked(xd, rep, N, group=128, config=dict(WARP, pdl=True))
    check(out, x, ref_w, 128, "K=%d N=%d M=%d" % (K, N, M))
    if (K // 256) * (N // 32) >= 4 * torch.cuda.get_device_properties(DEV).multi_processor_count:
        # the default request takes this kernel here: the same bits
        auto = w4.gemm_repacked(xd, rep, N, group=128)
        torch.cuda.synchronize()
        assert torch.equal(auto.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("group", [32, 64, 256, 512, 1024])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_warp_repacked_groups(group, M):
    K, N = 2048, 384
    rep, ref_w = repacked(K, N, group, 31 + group, True)
    x = synth.activations(M, K, seed=33 + M)
    out = w4.gemm_repacked(to_dev(x), rep, N, group=group, config=WARP)
    check(out, x, ref_w, group, "group=%d M=%d" % (group, M))


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 19, 152, 300])
@pytest.mark.parametrize("M", [1, 4, 7])
def test_warp_repacked_grid_sizes(ctas, M):
    """Different grids give different tiles per CTA, runs per warp and split
    tiles (a run of blocks may cross a tile and a tile's blocks may be split
    between several warps); each is correct and repeats bit for bit."""
    K, N = 4096, 1024
    rep, ref_w = repacked(K, N, 128, 321, True)
    x = synth.activations(M, K, seed=322 + M)
    cfg = dict(WARP, ctas=ctas)
    a = w4.gemm_repacked(to_dev(x), rep, N, group=128, config=cfg)
    check(a, x, ref_w, 128, "ctas=%d" % ctas)
    a = a.clone()
    b = w4.gemm_repacked(to_dev(x), rep, N, group=128, config=cfg)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_warp_repacked_one_hot_is_exact(M):
    K, N = 1024, 768
    W = synth.weight(K, N, seed=61, outliers=True)
    ref_w = oracle.quantize_pack(W, 128)
    rep = w4.repack(*w4.quantize_pack(to_dev(W), 128), group=128)
    wdq = oracle.dequant(*ref_w, group=128).view(np.uint16)
    ks = np.array([0, 255, 7, 8, 127, 128, 500, 1023, 640, 64, 333, 900, 17, 256, 1000, 2])[:M]
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = 1.0
    out = w4.gemm_repacked(to_dev(x), rep, N, group=128, config=WARP)
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), wdq[ks])


def expert_set(E, K, N, group, seed):
    reps, refs = [], []
    for e in range(E):
        W = synth.weight(K, N, seed=seed + e)
        refs.append(oracle.quantize_pack(W, group))
        reps.append(w4.repack(*w4.quantize_pack(to_dev(W), group), group=group))
    return reps, refs


@pytest.mark.parametrize("E,M", [(64, 1), (64, 4), (64, 8), (3, 3), (5, 6), (1, 2)])
@pytest.mark.parametrize("K,N", [(2048, 768), (768, 2048)])
def test_warp_repacked_grouped(E, M, K, N):
    """Tiles of all experts are split between the CTAs in one launch; every
    expert's result matches the oracle."""
    reps, refs = expert_set(E, K, N, 128, 900 + K)
    xs = [synth.activations(M, K, seed=950 + e) for e in range(E)]
    xd = [to_dev(v) for v in xs]
    outs = w4.gemm_grouped_repacked(xd, reps, N, group=128, config=dict(WARP, pdl=True))
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    for e in range(E):
        err = oracle.rel_err(outs[e].cpu().numpy(), oracle.gemm(xs[e], *refs[e]))
        assert err <= TOL, "expert %d rel err %.3g" % (e, err)
    if E * (K // 256) * (N // 32) >= 4 * torch.cuda.get_device_properties(DEV).multi_processor_count:
        # the default request takes this kernel here: the same bits
        auto = w4.gemm_grouped_repacked(xd, reps, N, group=128)
        torch.cuda.synchronize()
        assert torch.equal(auto.view(torch.int16), outs.view(torch.int16))


def test_warp_repacked_dirty_output_zero_input_and_chains():
    K, N = 4096, 2048
    rep, ref_w = repacked(K, N, 128, 331, False)
    x = to_dev(synth.activations(8, K, seed=332))
    out = torch.full((8, N), 5.0, dtype=torch.float16, device=DEV)
    w4.gemm_repacked(torch.zeros_like(x), rep, N, group=128, out=out, config=WARP)
    torch.cuda.synchronize()
    assert torch.all(out.view(torch.int16) == 0)
    outs = [torch.full((8, N), 9.0, dtype=torch.float16, device=DEV) for _ in range(6)]
    for o in outs:
        w4.gemm_repacked(x, rep, N, group=128, out=o, config=dict(WARP, pdl=True))
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    ref = oracle.gemm(x.cpu().numpy(), *ref_w, group=128)
    assert oracle.rel_err(outs[0].cpu().numpy(), ref) <= TOL


def test_warp_repacked_refusals():
    K, N = 1024, 4096
    rep, _ = repacked(K, N, 128, 341, False)
    x9 = to_dev(synth.activations(9, K, seed=342))
    with pytest.raises(w4.W4A16Error) as e:              # M > 8
        w4.gemm_repacked(x9, rep, N, group=128, config=WARP)
    assert e.value.status == 2
    x1 = to_dev(synth.activations(1, K, seed=343))
    with pytest.raises(w4.W4A16Error) as e:              # 128 tiles on one CTA
        w4.gemm_repacked(x1, rep, N, group=128, config=dict(WARP, ctas=1))
    assert e.value.status == 2
    # the default request at M = 9 takes the stream kernel and still answers
    out = w4.gemm_repacked(x9, rep, N, group=128)
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0 and out.shape == (9, N)
