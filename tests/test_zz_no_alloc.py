"""w4a16_gemm_noalloc: the decode GEMM for callers that may not allocate GPU
memory (a runtime limited to memory reserved at start-up, a real-time loop
that cannot afford an allocation, an application whose own allocator owns all
memory).  Its scratch is a fixed array inside the library.  Called through the
C ABI, two calls in a row must match the existing entry point (w4a16_gemm)
within the GEMM tolerance; the second call also shows that what the first call
left in the shared scratch does not leak into the next result.

This file's name sorts last so that a run stopping at the first failure has
run every other test before it."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_int4_codes_gb300 as w4
from weight_only_int4_codes_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("K,N,M", [(4096, 4096, 1), (14336, 4096, 8), (4096, 1000, 16)])
def test_noalloc_matches_gemm_on_two_calls_in_a_row(K, N, M):
    W = synth.weight(K, N, seed=1200 + K + N)
    packed, scales, zeros = w4.quantize_pack(torch.from_numpy(W).cuda(), 128)
    outs = []
    for call in range(2):
        x = torch.from_numpy(synth.activations(M, K, seed=1300 + call + M)).cuda()
        got = w4.gemm_noalloc(x, packed, scales, zeros, 128)
        ref = w4.gemm(x, packed, scales, zeros, 128)
        torch.cuda.synchronize()
        assert w4.kernel_status() == 0
        err = oracle.rel_err(got.cpu().numpy(), ref.cpu().numpy().astype(np.float64))
        assert err <= TOL, "call %d: rel err %.3g against w4a16_gemm" % (call, err)
        outs.append(got.cpu())
    assert not torch.equal(outs[0], outs[1])      # two different inputs, two results


def test_noalloc_rejects_a_shape_beyond_its_scratch():
    """N = 2^20 columns need more tile counters than the fixed scratch holds:
    the call is refused before anything is enqueued."""
    lib = w4.native.load_library()
    st = lib.w4a16_gemm_noalloc(16, 16, 16, 16, 16, 1, 1 << 20, 128, 128, None)
    assert st == 2
    assert b"scratch" in lib.w4a16_last_error()
