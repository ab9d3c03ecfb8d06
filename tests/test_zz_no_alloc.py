"""The W4A16 GEMV entry point that allocates nothing.

Some callers cannot allocate device memory when they run a layer (a runtime
that forbids allocation after start-up, code inside a memory pool it does not
own, a host with a fixed footprint).  qlin_w4a16_gemv_noalloc serves them with
a fixed scratch array inside the library instead of a caller workspace.  This
file checks, through the C ABI, that two calls in a row give the same output
as the workspace-taking GEMV, within the parity tolerance used everywhere
else.  It is collected last so that a stop-at-first-failure run has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import W4A16Linear

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (4, 4096, 14336), (16, 28672, 4096), (3, 512, 512)])
def test_noalloc_matches_workspace_gemv(M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    Wh = syn.make_weight(N, K, seed=M + N)
    Xh = syn.make_act(M, K, seed=M + K + 1)
    W = torch.from_numpy(Wh.view(np.int16)).cuda()
    X = torch.from_numpy(Xh.view(np.int16)).cuda()
    lin = W4A16Linear(W)
    ref = lin(X, path=q.PATH_GEMV).float()
    # the tolerance's scale: ||x_m|| * ||deq(w_n)|| (dequantised rows from the oracle)
    xn = torch.from_numpy(np.linalg.norm(syn.bf16_bits_to_f32(Xh).astype(np.float64), axis=1)).cuda()
    wn = torch.from_numpy(np.linalg.norm(oracle.dequant_w4(oracle.quantize_w4(Wh)), axis=1)).cuda()
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        q.qlin_w4a16_gemv_noalloc(X, lin.codes, lin.scales, lin.zeros, Y.view(torch.int16), M, N, K, 128)
        err = ((Y.double() - ref.double()).abs() / (xn[:, None] * wn[None, :])).max().item()
        assert err <= TOL
        assert torch.equal(Y.float(), ref)       # same kernel, same split order: identical bits
    assert q.qlin_get_device_error() == 0


def test_noalloc_rejects_oversize():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QlinError) as e:       # K % 256 != 0: the CUDA-core GEMV needs ~15.7 MiB of partial sums
        q.qlin_w4a16_gemv_noalloc(t, t, t, t, t, 16, 16384, 28800, 128)
    assert e.value.status == 4
