"""The five workload configurations against the oracle on the GPU, through the C ABI.

C1  W4A16 tiny: M=1, K=N=512, G=128 asymmetric, no outliers, seed 0.
C2  W4A16 Llama-3-8B decode layers (K=4096: N=6144, 4096, 28672; K=14336: N=4096)
    at M = 1, 4, 16, 1 % of input channels x20.
C3  Batch-sweep crossover: K=4096 N=14336 and K=14336 N=4096, M = 1, 2, 4 ... 512,
    W4A16 and W8A8 (per-tensor weight scale, per-token activation scale) on the
    same seeded weights.
C4  W8A8 FP8 prefill: M = 2048 and 8192 on the four C2 shapes, 0.1 % of tokens x50.
C5  Llama-3-70B layers (K=8192: N=10240, 8192, 57344; K=28672: N=8192): W4A16 at
    M = 1, 64, 256 and W8A8 at M = 256, 4096.

Every call goes through the default (AUTO) dispatch, as a user's would.  Up to
M = 512 on the C3 shapes and up to M = 32 elsewhere every output element is
compared with the oracle; beyond that whole tiles are (first, last and a random
middle tile of tokens, with the tile holding an outlier token added, x first,
last and middle 128-row weight tiles).
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import W4A16Linear, W8A8Linear

from _parity import check_w4, check_w8, host_f64, to_dev

pytestmark = pytest.mark.gpu

C2_SHAPES = [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]   # (K, N)
C3_SHAPES = [(4096, 14336), (14336, 4096)]
C5_SHAPES = [(8192, 10240), (8192, 8192), (8192, 57344), (28672, 8192)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    q.load()
    yield
    _weights.cache_clear()
    assert q.qlin_get_device_error() == 0


@functools.lru_cache(maxsize=2)
def _weights(K, N, seed, w4=True, w8=True):
    """Seeded BF16 weights with their oracle quantisations and device layers (one
    shape at a time is kept, so the large shapes do not pile up on the device)."""
    W = syn.make_weight(N, K, seed=seed)
    dW = to_dev(W)
    out = {"W": W}
    if w4:
        out["wq"] = oracle.quantize_w4(W)
        out["lin4"] = W4A16Linear(dW)
    if w8:
        out["Wq"], out["sw"] = oracle.quant_fp8_tensor(W)
        out["lin8"] = W8A8Linear(dW)
    del dW
    torch.cuda.synchronize()
    return out


def _run_w4(d, K, N, M, seed, full):
    X = syn.make_act(M, K, seed=seed)
    Y = host_f64(d["lin4"](to_dev(X)))
    plan = q.qlin_plan_info(q.OP_W4A16_GEMM, M, N, K)
    return check_w4(Y, X, d["wq"], full=full, tm=max(plan["tokens_per_tile"], 64), seed=seed)


def _run_w8(d, K, N, M, seed, full, token_outliers=0.0):
    X = syn.make_act(M, K, seed=seed, token_outlier_frac=token_outliers)
    Xq, sx = oracle.quant_fp8_rows(X)
    lin = d["lin8"]
    dXq, dsx = lin.quant_act(to_dev(X))
    # the device quantiser is bit-exact with the oracle's
    assert np.array_equal(dXq.cpu().numpy(), Xq) and np.array_equal(dsx.cpu().numpy()[:M], sx)
    Y = host_f64(lin.gemm(dXq, dsx))
    plan = q.qlin_plan_info(q.OP_W8A8_GEMM, M, N, K)
    extra = syn.outlier_indices(M, token_outliers, seed)
    return check_w8(Y, Xq, sx, d["Wq"], d["sw"], full=full, tm=max(plan["tokens_per_tile"], 64), seed=seed,
                    extra_m=extra[:1])


def test_c1_tiny():
    K = N = 512
    W = syn.make_weight(N, K, seed=0, outlier_frac=0.0)
    X = syn.make_act(1, K, seed=0)
    wq = oracle.quantize_w4(W)
    lin = W4A16Linear(to_dev(W))
    c_ref, s_ref, z_ref = oracle.pack_tile(wq)
    assert np.array_equal(lin.codes.cpu().numpy(), c_ref)
    assert np.array_equal(lin.scales.cpu().numpy().view(np.uint16), s_ref)
    assert np.array_equal(lin.zeros.cpu().numpy(), z_ref)
    Y = host_f64(lin(to_dev(X)))
    check_w4(Y, X, wq, full=True, tm=16, seed=0)


@pytest.mark.parametrize("K,N", C2_SHAPES)
def test_c2_llama8b_decode(K, N):
    d = _weights(K, N, seed=K + N, w8=False)
    c_ref, s_ref, z_ref = oracle.pack_tile(d["wq"])       # packing is bit-exact at full size
    assert np.array_equal(d["lin4"].codes.cpu().numpy(), c_ref)
    assert np.array_equal(d["lin4"].scales.cpu().numpy().view(np.uint16), s_ref)
    assert np.array_equal(d["lin4"].zeros.cpu().numpy(), z_ref)
    for M in (1, 4, 16):
        _run_w4(d, K, N, M, seed=M + K, full=True)


@pytest.mark.parametrize("K,N", C3_SHAPES)
@pytest.mark.parametrize("variant", ["w4a16", "w8a8"])
def test_c3_crossover_sweep(K, N, variant):
    d = _weights(K, N, seed=3 * K + N)
    for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
        if variant == "w4a16":
            _run_w4(d, K, N, M, seed=M + 11, full=True)
        else:
            _run_w8(d, K, N, M, seed=M + 13, full=True)


@pytest.mark.parametrize("K,N", C2_SHAPES)
def test_c4_fp8_prefill(K, N):
    d = _weights(K, N, seed=5 * K + N, w4=False)
    for M in (2048, 8192):
        _run_w8(d, K, N, M, seed=M + 17, full=False, token_outliers=0.001)


@pytest.mark.parametrize("K,N", C5_SHAPES)
def test_c5_llama70b(K, N):
    d = _weights(K, N, seed=7 * K + N)
    for M in (1, 64, 256):
        _run_w4(d, K, N, M, seed=M + 19, full=M <= 32)
    for M in (256, 4096):
        _run_w8(d, K, N, M, seed=M + 23, full=False)
