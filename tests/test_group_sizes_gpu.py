"""GPU parity of W4A16 at group sizes G = 32 and 64 ([LP] S4 per-group
granularity, S5 b_eff = 4 + 16/G), through the C ABI.

Bar as for G = 128: packed codes / scales / zero-points bit-exact against the
oracle's tile layout; |Y - Y_ref| <= 2e-3 ||X[m]|| ||deq(W)[n]|| on the
small-M kernel (M <= 32) and the tcgen05 kernel.
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    q.load()
    yield
    assert q.qlin_get_device_error() == 0


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def norm_err(Y, Yref, xn, wn):
    return float((np.abs(Y - Yref) / (xn[:, None] * wn[None, :])).max())


@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("N,K,sym", [(256, 1024, False), (384, 512, True), (4096, 4096, False)])
def test_pack_w4_bit_exact_other_groups(G, N, K, sym):
    W = syn.make_weight(N, K, seed=N + K + G, outlier_frac=0.01)
    W[:2, :G] = 0  # degenerate all-zero groups
    wq = oracle.quantize_w4(W, G=G, symmetric=sym)
    c_ref, s_ref, z_ref = oracle.pack_tile(wq)
    layer = W4A16Linear(to_dev(W), G=G, symmetric=sym)
    torch.cuda.synchronize()
    assert np.array_equal(layer.codes.cpu().numpy(), c_ref)
    assert np.array_equal(layer.scales.cpu().numpy().view(np.uint16), s_ref)
    assert np.array_equal(layer.zeros.cpu().numpy(), z_ref)


@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("M,path", [(1, q.PATH_GEMV), (5, q.PATH_GEMV), (16, q.PATH_GEMV), (32, q.PATH_GEMV),
                                    (17, q.PATH_TC), (100, q.PATH_TC), (300, q.PATH_TC)])
def test_w4a16_other_groups_m_sweep(G, M, path):
    N, K = 256, 1024
    W = syn.make_weight(N, K, seed=M + G)
    X = syn.make_act(M, K, seed=M + G + 1)
    wq = oracle.quantize_w4(W, G=G)
    Y = W4A16Linear(to_dev(W), G=G)(to_dev(X).view(torch.bfloat16), path=path)
    Y = Y.float().cpu().numpy().astype(np.float64)
    Yref = oracle.w4a16_full(X, wq)
    xn = np.linalg.norm(syn.bf16_bits_to_f32(X).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.dequant_w4(wq), axis=1)
    assert norm_err(Y, Yref, xn, wn) <= TOL


@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("M,N,K", [(4, 4096, 14336), (16, 28672, 4096), (256, 4096, 4096)])
def test_w4a16_other_groups_llama_sampled(G, M, N, K):
    W = syn.make_weight(N, K, seed=N + G)
    X = syn.make_act(M, K, seed=K + G)
    wq = oracle.quantize_w4(W, G=G)
    Y = W4A16Linear(to_dev(W), G=G)(to_dev(X).view(torch.bfloat16)).float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(G + M)
    ms, ns = rng.integers(0, M, 1500), rng.integers(0, N, 1500)
    ref = oracle.w4a16_at(X, wq, ms, ns)
    xn = np.linalg.norm(syn.bf16_bits_to_f32(X).astype(np.float64), axis=1)[ms]
    wn = np.linalg.norm(oracle.dequant_w4(oracle.W4Quant(wq.q[ns], wq.s[ns], wq.z[ns], G, False, 0)), axis=1)
    assert float((np.abs(Y[ms, ns] - ref) / (xn * wn)).max()) <= TOL


def test_other_groups_rejected_where_unsupported():
    N, K = 256, 4224  # K % 256 != 0: only the CUDA-core GEMV serves small M there, and it takes G = 128 only
    lin = W4A16Linear(torch.zeros((N, K), dtype=torch.bfloat16, device="cuda"), G=64)
    X = torch.zeros((2, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q.QlinError) as e:
        lin(X, path=q.PATH_GEMV)
    assert e.value.status == 2  # QLIN_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(q.QlinError) as e:
        q.qlin_w4_packed_sizes(N, 4096, 48)
    assert e.value.status == 2


@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("M,path", [(3, q.PATH_GEMV), (24, q.PATH_GEMV), (100, q.PATH_TC)])
def test_w4a16_other_groups_with_fused_epilogue(G, M, path):
    N, K = 256, 1024
    W = syn.make_weight(N, K, seed=M + 3 * G)
    X = syn.make_act(M, K, seed=M + 3 * G + 1)
    wq = oracle.quantize_w4(W, G=G)
    b32 = np.random.default_rng(G).normal(0.0, 0.5, N).astype(np.float32)
    bias = (b32.view(np.uint32) >> 16).astype(np.uint16)  # BF16 by truncation: any BF16 values will do
    lin = W4A16Linear(to_dev(W), G=G, bias=to_dev(bias).view(torch.bfloat16))
    Y = lin(to_dev(X).view(torch.bfloat16), path=path, act=q.ACT_SILU).float().cpu().numpy().astype(np.float64)
    Yref = oracle.epilogue(oracle.w4a16_full(X, wq), bias, oracle.ACT_SILU)
    xn = np.linalg.norm(syn.bf16_bits_to_f32(X).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.dequant_w4(wq), axis=1)
    bound = 1.13 * TOL * xn[:, None] * wn[None, :] + 2.0 ** -8 * np.abs(Yref)
    assert (np.abs(Y - Yref) <= bound).all()
