"""Parity of the warp-stream decode kernel (W4A16_DECODE_WARP, M <= 4) with the
fp64 oracle: every decode workload shape at M = 1..4, other group sizes, ragged
N and K, different grid sizes (so different runs per warp and different split
tiles), one-hot exactness, dirty outputs and run-to-run determinism."""
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
def quantized(K, N, group, seed, outliers=False):
    W = synth.weight(K, N, seed=seed, outliers=outliers)
    ref_w = oracle.quantize_pack(W, group)
    dev_w = w4.quantize_pack(to_dev(W), group)
    torch.cuda.synchronize()
    assert np.array_equal(dev_w[0].cpu().numpy().view(np.uint32), ref_w[0])
    return dev_w, ref_w


def check(x, dev_w, ref_w, group, config):
    M, K = x.shape
    try:
        w4.plan(M, dev_w[0].shape[1], K, group, **config)
    except w4.W4A16Error:
        # group 32 at M = 4: two ring slots per warp do not fit (checked in
        # test_warp_plan_and_refusals); other kernels serve it
        pytest.skip("warp-stream kernel does not serve this shape")
    out = w4.gemm_ex(to_dev(x), *dev_w, group=group, config=config)
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    err = oracle.rel_err(out.cpu().numpy(), oracle.gemm(x, *ref_w, group=group))
    assert err <= TOL, "rel err %.3g (M=%d, %s)" % (err, x.shape[0], config)
    return out


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("K,N,outliers", [
    (512, 256, False), (4096, 4096, False), (2048, 768, False), (768, 2048, False),
    (4096, 14336, True), (14336, 4096, True),
])
def test_warp_decode_configs(K, N, outliers, M):
    dev_w, ref_w = quantized(K, N, 128, synth.weight_seed(1) + K + N, outliers)
    x = synth.activations(M, K, seed=synth.x_seed(1, M) + K)
    check(x, dev_w, ref_w, 128, dict(WARP, pdl=True))


@pytest.mark.parametrize("group", [32, 64, 256, 512, 1024])
@pytest.mark.parametrize("M", [1, 3])
def test_warp_other_groups(group, M):
    K, N = 2048, 520                 # N % 32 != 0: a ragged last column tile
    dev_w, ref_w = quantized(K, N, group, 301 + group, True)
    x = synth.activations(M, K, seed=302 + M)
    check(x, dev_w, ref_w, group, WARP)


@pytest.mark.parametrize("K,group", [(1088, 64), (576, 32), (1152, 128), (1280, 256), (768, 128)])
@pytest.mark.parametrize("M", [1, 4])
def test_warp_k_not_a_multiple_of_the_unit(K, group, M):
    """K % 512 != 0: the last unit of a tile is partly past K and reads zeros
    (and its last x box may lie wholly past K)."""
    N = 264
    dev_w, ref_w = quantized(K, N, group, 311 + K, False)
    x = synth.activations(M, K, seed=312 + M)
    check(x, dev_w, ref_w, group, WARP)


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 19, 152])
@pytest.mark.parametrize("M", [1, 4])
def test_warp_grid_sizes(ctas, M):
    """Different grids give different tiles per CTA, runs per warp and split
    tiles; each is correct and each repeats bit for bit."""
    K, N = 4096, 1024
    dev_w, ref_w = quantized(K, N, 128, 321, True)
    x = synth.activations(M, K, seed=322 + M)
    cfg = dict(WARP, ctas=ctas)
    a = check(x, dev_w, ref_w, 128, cfg).clone()
    b = w4.gemm_ex(to_dev(x), *dev_w, group=128, config=cfg)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M", [1, 2, 4])
def test_warp_one_hot_is_exact(M):
    K, N = 1024, 768
    W = synth.weight(K, N, seed=61, outliers=True)
    ref_w = oracle.quantize_pack(W, 128)
    dev_w = w4.quantize_pack(to_dev(W), 128)
    wdq = oracle.dequant(*ref_w, group=128).view(np.uint16)
    ks = np.array([0, 1, 7, 8, 127, 128, 500, 1023, 640, 64, 333, 900, 17, 256, 1000, 2])[:M]
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = 1.0
    out = w4.gemm_ex(to_dev(x), *dev_w, group=128, config=WARP)
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    assert np.array_equal(out.cpu().numpy().view(np.uint16), wdq[ks])


def test_warp_dirty_output_zero_input_and_chains():
    """out is overwritten; x = 0 gives +0; a PDL chain of calls on rotating
    weights and outputs gives every call's own result."""
    K, N = 4096, 2048
    dev_w, ref_w = quantized(K, N, 128, 331, False)
    x = to_dev(synth.activations(4, K, seed=332))
    out = torch.full((4, N), 5.0, dtype=torch.float16, device=DEV)
    w4.gemm_ex(torch.zeros_like(x), *dev_w, group=128, out=out, config=WARP)
    torch.cuda.synchronize()
    assert torch.all(out.view(torch.int16) == 0)
    outs = [torch.full((4, N), 9.0, dtype=torch.float16, device=DEV) for _ in range(6)]
    for o in outs:
        w4.gemm_ex(x, *dev_w, group=128, out=o, config=dict(WARP, pdl=True))
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    ref = oracle.gemm(x.cpu().numpy(), *ref_w, group=128)
    assert oracle.rel_err(outs[0].cpu().numpy(), ref) <= TOL


def test_warp_plan_and_refusals():
    p = w4.plan(4, 4096, 4096, path="decode", variant="warp")
    assert (p["path"], p["variant"]) == (1, 4)
    for bad in (dict(M=4, N=4092, K=4096, group=128),    # N % 8 != 0
                dict(M=4, N=4096, K=4032, group=192),    # not a power-of-two group
                dict(M=5, N=4096, K=4096, group=128),    # M > 4
                dict(M=4, N=4096, K=4096, group=32)):    # ring slots do not fit
        with pytest.raises(w4.W4A16Error):
            w4.plan(bad["M"], bad["N"], bad["K"], bad["group"], path="decode", variant="warp")
