"""Per-channel W4A16 scales (G = K: one scale and zero-point per weight row,
[LP] S4 "per-channel") on the GPU against the oracle, through the C ABI.

Packing (codes, the row scales and zero-points in the tile layout) is
bit-exact; GEMM outputs stay within
    |Y - Y_ref| <= 2e-3 * ||X[m, :]||_2 * ||W_deq[n, :]||_2
on both kernels: the small-M register-MMA kernel (every element) and the
tcgen05 kernel (every element up to 32 tokens, whole tiles beyond).
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import W4A16Linear

from _parity import bias_bits, check_w4, host_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    q.load()
    yield
    assert q.qlin_get_device_error() == 0


@pytest.mark.parametrize("N,K,sym", [(256, 1024, False), (512, 4096, True), (4096, 14336, False), (128, 128, False)])
def test_pack_per_channel_bit_exact(N, K, sym):
    W = syn.make_weight(N, K, seed=N + K)
    W[1, :] = 0                                      # a degenerate row: s = 1, z = 0 (symmetric: 8)
    wq = oracle.quantize_w4(W, G=K, symmetric=sym)
    c_ref, s_ref, z_ref = oracle.pack_tile(wq)
    lin = W4A16Linear(to_dev(W), G=K, symmetric=sym)
    torch.cuda.synchronize()
    assert np.array_equal(lin.codes.cpu().numpy(), c_ref)
    assert np.array_equal(lin.scales.cpu().numpy().view(np.uint16), s_ref)
    assert np.array_equal(lin.zeros.cpu().numpy(), z_ref)
    assert lin.packed_bytes() == N * K // 2 + 2 * N + N // 2


# (M, N, K, path, act, expected kernel)
CASES = [
    (1, 4096, 4096, q.PATH_AUTO, q.ACT_NONE, q.KERNEL_W4A16_MMA),
    (4, 4096, 14336, q.PATH_AUTO, q.ACT_NONE, q.KERNEL_W4A16_MMA),
    (16, 6144, 4096, q.PATH_AUTO, q.ACT_SILU, q.KERNEL_W4A16_MMA),
    (32, 4096, 4096, q.PATH_AUTO, q.ACT_NONE, q.KERNEL_W4A16_MMA),
    (5, 512, 1024, q.PATH_TC, q.ACT_NONE, q.KERNEL_W4A16_TC),
    (64, 4096, 14336, q.PATH_AUTO, q.ACT_GELU, q.KERNEL_W4A16_TC),
    (128, 14336, 4096, q.PATH_AUTO, q.ACT_NONE, q.KERNEL_W4A16_TC),
    (512, 14336, 4096, q.PATH_AUTO, q.ACT_NONE, q.KERNEL_W4A16_TC),
    (2048, 4096, 4096, q.PATH_AUTO, q.ACT_NONE, q.KERNEL_W4A16_TC),
]


@pytest.mark.parametrize("M,N,K,path,act,kernel", CASES)
def test_gemm_per_channel(M, N, K, path, act, kernel):
    plan = q.qlin_plan_info(q.OP_W4A16_GEMM, M, N, K, K, path)
    assert plan["kernel"] == kernel, plan
    seed = M + N + K
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    wq = oracle.quantize_w4(W, G=K)
    bias = bias_bits(N, seed) if act else None
    lin = W4A16Linear(to_dev(W), G=K, bias=None if bias is None else to_dev(bias).view(torch.bfloat16))
    Y = host_f64(lin(to_dev(X), path=path, act=act))
    check_w4(Y, X, wq, full=M <= 32, tm=max(plan["tokens_per_tile"], 64), seed=seed, bias=bias, act=act)


def test_per_channel_cuda_core_gemv_is_rejected():
    # K % 256 != 0 on the small-M path runs the CUDA-core GEMV, which takes G = 128 only
    K, N = 4224, 512
    lin = W4A16Linear(to_dev(syn.make_weight(N, K, seed=1)), G=K)
    X = to_dev(syn.make_act(4, K, seed=2))
    with pytest.raises(q.QlinError) as e:
        lin(X, path=q.PATH_GEMV)
    assert e.value.status == 2
    Y = host_f64(lin(X, path=q.PATH_TC))           # the tensor-core kernel takes it
    check_w4(Y, syn.make_act(4, K, seed=2), oracle.quantize_w4(syn.make_weight(N, K, seed=1), G=K), full=True,
             tm=16, seed=0)
