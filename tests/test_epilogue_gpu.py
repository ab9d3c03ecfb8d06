"""GPU parity of the fused output epilogue (bias + activation) against the oracle.

Y = bf16(act(acc + bias[n])) on every kernel path of both GEMMs.  Bar: the
GEMM bound carried through the activation (slope <= 1.13 for GELU, 1.10 for
SiLU, 1 for ReLU) plus the BF16 rounding of the output:
    |Y - Y_ref| <= 1.13 * 2e-3 * ||X_deq[m]|| * ||W_deq[n]|| + 2^-8 |Y_ref|
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import W4A16Linear, W8A8Linear

pytestmark = pytest.mark.gpu

TOL = 2e-3
SLOPE = 1.13
ACTS = [q.ACT_NONE, q.ACT_RELU, q.ACT_SILU, q.ACT_GELU]


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


def check(Y, Yref, xn, wn):
    bound = SLOPE * TOL * xn[:, None] * wn[None, :] + 2.0 ** -8 * np.abs(Yref)
    bad = np.abs(Y - Yref) > bound
    assert not bad.any(), (np.argwhere(bad)[:4], Y[bad][:4], Yref[bad][:4])


def _bias(N, seed):
    # magnitudes comparable with the outputs, so that the bias shifts the activation's operating point
    b = (np.random.default_rng(seed).normal(0.0, 0.5, N)).astype(np.float32)
    return (b.view(np.uint32) >> 16).astype(np.uint16) + ((b.view(np.uint32) >> 15) & 1).astype(np.uint16)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M,N,K,path", [(1, 512, 1024, q.PATH_GEMV), (5, 512, 1024, q.PATH_GEMV),
                                        (16, 512, 1024, q.PATH_GEMV), (32, 512, 1024, q.PATH_GEMV),
                                        (3, 256, 4224, q.PATH_GEMV), (100, 512, 1024, q.PATH_TC),
                                        (300, 256, 1024, q.PATH_TC), (64, 256, 8192, q.PATH_TC)])
def test_w4a16_fused_epilogue(M, N, K, path, act):
    W = syn.make_weight(N, K, seed=M + N + act)
    X = syn.make_act(M, K, seed=M + K + act)
    wq = oracle.quantize_w4(W)
    bias = _bias(N, seed=N + act) if act != q.ACT_RELU or M % 2 else None
    lin = W4A16Linear(to_dev(W), bias=to_dev(bias).view(torch.bfloat16) if bias is not None else None)
    Y = lin(to_dev(X).view(torch.bfloat16), path=path, act=act).float().cpu().numpy().astype(np.float64)
    Yref = oracle.epilogue(oracle.w4a16_full(X, wq), bias, act)
    xn = np.linalg.norm(syn.bf16_bits_to_f32(X).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.dequant_w4(wq), axis=1)
    check(Y, Yref, xn, wn)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M,N,K,path", [(1, 512, 1024, q.PATH_TC), (16, 512, 1024, q.PATH_TC),
                                        (300, 256, 1024, q.PATH_TC), (64, 256, 8192, q.PATH_TC),
                                        (4, 512, 1024, q.PATH_GEMV)])
def test_w8a8_fused_epilogue(M, N, K, path, act):
    W = syn.make_weight(N, K, seed=M + N + 7 * act)
    X = syn.make_act(M, K, seed=M + K + 7 * act, token_outlier_frac=0.01)
    Xq_r, sx_r = oracle.quant_fp8_rows(X)
    Wq_r, sw_r = oracle.quant_fp8_tensor(W)
    bias = _bias(N, seed=N + 3 * act)
    lin = W8A8Linear(to_dev(W), bias=to_dev(bias).view(torch.bfloat16))
    Y = lin(to_dev(X).view(torch.bfloat16), path=path, act=act).float().cpu().numpy().astype(np.float64)
    Yref = oracle.epilogue(oracle.w8a8_full(Xq_r, sx_r, Wq_r, sw_r), bias, act)
    tab = oracle.e4m3_table()
    xn = np.linalg.norm(tab[Xq_r] * np.asarray(sx_r, np.float64)[:, None], axis=1)
    wn = np.linalg.norm(tab[Wq_r] * float(np.asarray(sw_r).reshape(-1)[0]), axis=1)
    check(Y, Yref, xn, wn)


def test_fused_rejects_bad_arguments():
    N, K, M = 256, 512, 2
    lin = W4A16Linear(torch.zeros((N, K), dtype=torch.bfloat16, device="cuda"))
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q.QlinError) as e:
        q.qlin_w4a16_gemm_fused(X.view(torch.int16), lin.codes, lin.scales, lin.zeros, Y.view(torch.int16), M, N, K,
                                128, None, 4, None, 0, q.PATH_AUTO)
    assert e.value.status == 1  # QLIN_ERR_INVALID_VALUE: unknown activation
    b = torch.zeros(N + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q.QlinError) as e:
        q.qlin_w4a16_gemm_fused(X.view(torch.int16), lin.codes, lin.scales, lin.zeros, Y.view(torch.int16), M, N, K,
                                128, b[1:].data_ptr(), q.ACT_RELU, None, 0, q.PATH_AUTO)
    assert e.value.status == 3  # QLIN_ERR_MISALIGNED: bias not 16-byte aligned
