"""The W4A16 GEMV entry point that allocates nothing.

Some callers cannot allocate device memory when they run a layer (a runtime
that forbids allocation after start-up, code inside a memory pool it does not
own, a host with a fixed footprint).  qlin_w4a16_gemv_noalloc serves them with
a fixed scratch array inside the library instead of a caller workspace.

The array is only used when the call runs the CUDA-core GEMV (K % 256 != 0)
with its K range split: the cases below are chosen so, and the dispatch query
confirms it (split count > 1 and a non-zero workspace that the array stands in
for).  Each output is compared with the oracle element by element and, bit
for bit, with the workspace-taking call (the same kernel with the same split
order).  Different shapes run back to back, twice each, so every call finds the
array holding the previous call's counters and partial sums.  The K % 256 == 0
cases run the tensor-core small-M kernel, which needs no scratch at all.

This file is collected last, so that a stop-at-first-failure run has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import W4A16Linear

from _parity import check_w4, host_f64, to_dev

pytestmark = pytest.mark.gpu

# (M, N, K): K % 256 != 0 -> CUDA-core GEMV with its partial sums in the array
SCRATCH_CASES = [(1, 4096, 4224), (4, 6144, 4224), (16, 4096, 4224), (3, 512, 4224)]


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()


def _case(M, N, K, seed):
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1)
    return W, X, oracle.quantize_w4(W), W4A16Linear(to_dev(W))


def test_noalloc_scratch_path_matches_oracle_and_workspace_call():
    _need_gpu()
    cases = []
    for i, (M, N, K) in enumerate(SCRATCH_CASES):
        plan = q.qlin_plan_info(q.OP_W4A16_GEMM, M, N, K, 128, q.PATH_GEMV)
        assert plan["kernel"] == q.KERNEL_W4A16_GEMV and plan["splits"] > 1 and plan["ws_bytes"] > 0, plan
        W, X, wq, lin = _case(M, N, K, seed=900 + i)
        ref = lin(to_dev(X), path=q.PATH_GEMV).clone()   # the same kernel with a caller workspace
        cases.append((M, N, K, X, wq, lin, ref))
    torch.cuda.synchronize()
    for _ in range(2):                                   # each shape twice, all shapes back to back
        for M, N, K, X, wq, lin, ref in cases:
            Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            q.qlin_w4a16_gemv_noalloc(to_dev(X), lin.codes, lin.scales, lin.zeros, Y.view(torch.int16), M, N, K,
                                      128)
            torch.cuda.synchronize()
            assert torch.equal(Y, ref), (M, N, K)       # same kernel, same split order: identical bits
            check_w4(host_f64(Y), X, wq, full=True, tm=16, seed=M)
    assert q.qlin_get_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (16, 28672, 4096)])
def test_noalloc_tensor_core_kernel_matches_oracle(M, N, K):
    _need_gpu()
    plan = q.qlin_plan_info(q.OP_W4A16_GEMM, M, N, K, 128, q.PATH_GEMV)
    assert plan["kernel"] == q.KERNEL_W4A16_MMA and plan["ws_bytes"] == 0
    W, X, wq, lin = _case(M, N, K, seed=M + N)
    ref = lin(to_dev(X), path=q.PATH_GEMV)
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        q.qlin_w4a16_gemv_noalloc(to_dev(X), lin.codes, lin.scales, lin.zeros, Y.view(torch.int16), M, N, K, 128)
        torch.cuda.synchronize()
        assert torch.equal(Y, ref)
        check_w4(host_f64(Y), X, wq, full=True, tm=16, seed=M)
    assert q.qlin_get_device_error() == 0


def test_noalloc_rejects_oversize():
    _need_gpu()
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QlinError) as e:       # K % 256 != 0: the CUDA-core GEMV needs ~15.7 MiB of partial sums
        q.qlin_w4a16_gemv_noalloc(t, t, t, t, t, 16, 16384, 28800, 128)
    assert e.value.status == 4
