"""The host side of a call: prepared GEMM calls, the per-thread plan cache and
the tensor-map cache give the same bits as fresh calls, follow new contents of
x, and keep requests with different configurations apart."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_codes_gb300 as w4
from weight_only_int4_codes_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.fixture(scope="module")
def weights():
    K, N = 2048, 1024
    W = synth.weight(K, N, seed=201, outliers=True)
    return W, w4.quantize_pack(to_dev(W), 128), oracle.quantize_pack(W, 128)


@pytest.mark.parametrize("M,config", [
    (1, None), (4, dict(pdl=True)), (16, dict(path="decode", variant="registers")),
    (8, dict(path="decode", variant="tma", pdl=True)), (8, dict(path="decode", variant="stream")),
    (64, None), (300, dict(path="prefill", tile_m=256)),
])
def test_prepared_call_matches_fresh_calls(weights, M, config):
    _, dev_w, ref_w = weights
    K = dev_w[0].shape[0] * 8
    x = to_dev(synth.activations(M, K, seed=202 + M))
    ref = w4.gemm_ex(x, *dev_w, group=128, config=config).clone()
    out = torch.empty_like(ref)
    call = w4.prepare_gemm(x, *dev_w, group=128, out=out, config=config)
    for _ in range(3):
        out.fill_(3.0)
        assert call() is out
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # new contents in x are seen by the same prepared call
    x2 = synth.activations(M, K, seed=203 + M)
    x.copy_(to_dev(x2))
    call()
    torch.cuda.synchronize()
    assert w4.kernel_status() == 0
    err = oracle.rel_err(out.cpu().numpy(), oracle.gemm(x2, *ref_w, group=128))
    assert err <= 5e-3


def test_plan_cache_keeps_requests_apart(weights):
    """Alternating requests on one shape (the cache key holds the request):
    each configuration still gives its own, correct, result."""
    _, dev_w, ref_w = weights
    K = dev_w[0].shape[0] * 8
    xh = synth.activations(4, K, seed=211)
    x = to_dev(xh)
    ref = oracle.gemm(xh, *ref_w, group=128)
    cfgs = [None, dict(path="decode", variant="registers", split_k=2, warps_k=4, warps_n=1),
            dict(path="decode", variant="tma", warps_n=4), dict(path="prefill", tile_m=16)]
    outs = {}
    for rnd in range(3):
        for i, c in enumerate(cfgs):
            o = w4.gemm_ex(x, *dev_w, group=128, config=c)
            torch.cuda.synchronize()
            assert oracle.rel_err(o.cpu().numpy(), ref) <= 5e-3, c
            if rnd == 0:
                outs[i] = o.clone()
            else:
                assert torch.equal(o.view(torch.int16), outs[i].view(torch.int16)), c


def test_tensor_map_cache_follows_the_pointer(weights):
    """Two weight copies at different addresses through the TMA variant, called
    alternately: the cached tensor maps never mix them up."""
    W, dev_w, ref_w = weights
    K = dev_w[0].shape[0] * 8
    other_W = synth.weight(K, dev_w[0].shape[1], seed=221)
    other = w4.quantize_pack(to_dev(other_W), 128)
    other_ref = oracle.quantize_pack(other_W, 128)
    xh = synth.activations(2, K, seed=222)
    x = to_dev(xh)
    cfg = dict(path="decode", variant="tma")
    for _ in range(3):
        for d, r in ((dev_w, ref_w), (other, other_ref)):
            o = w4.gemm_ex(x, *d, group=128, config=cfg)
            torch.cuda.synchronize()
            assert oracle.rel_err(o.cpu().numpy(), oracle.gemm(xh, *r, group=128)) <= 5e-3


def test_prepared_call_bf16_and_errors(weights):
    K, N = 1024, 512
    Wb = synth.weight_bf16(K, N, seed=231)
    packed, scales, zeros = w4.quantize_pack_bf16(
        torch.from_numpy(Wb.view(np.int16)).view(torch.bfloat16).to(DEV), 128)
    x = torch.from_numpy(synth.activations_bf16(3, K, seed=232).view(np.int16)).view(
        torch.bfloat16).to(DEV)
    ref = w4.gemm_ex(x, packed, scales, zeros, group=128).clone()
    call = w4.prepare_gemm(x, packed, scales, zeros, group=128)
    out = call()
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16 and torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # a request the library refuses is reported when the prepared call runs
    bad = w4.prepare_gemm(x, packed, scales, zeros, group=128, config=dict(variant="warp",
                                                                           path="decode"))
    with pytest.raises(w4.W4A16Error) as e:
        bad()
    assert e.value.status == 2


def test_concurrent_host_threads(weights):
    """Four host threads, each with its own stream, issue GEMMs of different
    shapes and variants at once (ctypes releases the interpreter lock during
    the C call, so the plan, tensor-map and scratch caches are exercised
    concurrently); every result equals the single-threaded one bit for bit."""
    import threading
    _, dev_w, _ = weights
    K = dev_w[0].shape[0] * 8
    cases = [(1, dict(path="decode", variant="tma", pdl=True)),
             (3, dict(path="decode", variant="registers")),
             (2, dict(path="decode", variant="warp")),
             (8, dict(path="decode", variant="stream")),
             (64, None)]
    xs = {M: to_dev(synth.activations(M, K, seed=240 + M)) for M, _ in cases}
    ref = {}
    for M, cfg in cases:
        ref[M] = w4.gemm_ex(xs[M], *dev_w, group=128, config=cfg).clone()
    torch.cuda.synchronize()
    errors = []

    def worker(tid):
        try:
            s = torch.cuda.Stream()
            outs = {M: torch.empty_like(ref[M]) for M, _ in cases}
            calls = [w4.prepare_gemm(xs[M], *dev_w, group=128, out=outs[M], config=cfg)
                     for M, cfg in cases]
            with torch.cuda.stream(s):
                for it in range(40):
                    for c in calls[tid % len(calls):] + calls[:tid % len(calls)]:
                        c(s)
                    if it % 10 == 9:
                        s.synchronize()
                        for M, _ in cases:
                            if not torch.equal(outs[M].view(torch.int16), ref[M].view(torch.int16)):
                                errors.append((tid, it, M))
            s.synchronize()
        except Exception as e:        # reported below, on the main thread
            errors.append((tid, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors[:5]
    assert w4.kernel_status() == 0
