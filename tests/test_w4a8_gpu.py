"""W4A8 on the GPU against the oracle, through the C ABI.

The packed INT4 weights of qlin_pack_w4 (G = 128) times the per-token E4M3
activations of qlin_quant_act_fp8; the oracle's reference is the fp64 product of
the dequantised operands (sx[m] e4m3(Xq) and s (q - z)).  Bar:
    |Y - Y_ref| <= 2e-3 * ||X_deq[m, :]||_2 * ||W_deq[n, :]||_2
on every element up to 32 tokens (and on the crossover shapes up to 512),
on whole tiles beyond; the Llama-3-70B layers at M = 1, 64 and 256.  Each case asserts through the dispatch query which token
tile and split count it reaches.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import W4A8Linear

from _parity import blocks, check, host_f64, to_dev, w4_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    q.load()
    yield
    assert q.qlin_get_device_error() == 0


def _check_w4a8(Y, Xq, sx, wq, ms_ns):
    tab = oracle.e4m3_table()
    for ms, ns in ms_ns:
        sub = w4_rows(wq, ns)
        ref = oracle.w4a8_full(Xq[ms], sx[ms], sub)
        xn = np.linalg.norm(tab[Xq[ms]] * sx[ms].astype(np.float64)[:, None], axis=1)
        wn = np.linalg.norm(oracle.dequant_w4(sub), axis=1)
        check(Y[np.ix_(ms, ns)], ref, xn, wn, 0, "tile m%d n%d" % (ms[0], ns[0]))


def _run(M, N, K, seed, full, sym=False, W=None, wq=None, lin=None):
    if W is None:
        W = syn.make_weight(N, K, seed=seed)
        wq = oracle.quantize_w4(W, symmetric=sym)
        lin = W4A8Linear(to_dev(W), symmetric=sym)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    Xq_r, sx_r = oracle.quant_fp8_rows(X)
    Xq, sx = lin.quant_act(to_dev(X))
    Y = host_f64(lin.gemm(Xq, sx))
    plan = q.qlin_plan_info(q.OP_W4A8_GEMM, M, N, K)
    sel = [(np.arange(M), np.arange(N))] if full else blocks(M, N, plan["tokens_per_tile"], 128, seed)
    _check_w4a8(Y, Xq_r, sx_r, wq, sel)
    return plan


# (id, M, N, K, token tile, split count)
CASES = [
    ("bn16_m1", 1, 512, 1024, 16, 1),
    ("bn16_split", 4, 4096, 4096, 16, 3),
    ("bn16_m16_split", 16, 4096, 4096, 16, 3),
    ("bn32", 32, 512, 1024, 32, 1),
    ("bn64", 100, 4096, 4096, 64, 1),
    ("bn64_split", 64, 4096, 14336, 64, 2),
    ("bn64_ragged", 300, 512, 1024, 64, 1),
    ("bn64_prefill", 2048, 28672, 4096, 64, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_w4a8_gemm(case):
    name, M, N, K, bn, splits = case
    plan = q.qlin_plan_info(q.OP_W4A8_GEMM, M, N, K)
    assert plan["kernel"] == q.KERNEL_W4A8_TC
    assert (plan["tokens_per_tile"], plan["splits"]) == (bn, splits), plan
    _run(M, N, K, seed=M + N + K, full=M <= 32)


def test_w4a8_symmetric():
    _run(16, 512, 2048, seed=5, full=True, sym=True)


@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096)])
def test_w4a8_crossover_shapes(K, N):
    W = syn.make_weight(N, K, seed=3 * K + N)
    wq = oracle.quantize_w4(W)
    lin = W4A8Linear(to_dev(W))
    for M in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512):
        _run(M, N, K, seed=M + 41, full=True, W=W, wq=wq, lin=lin)


@pytest.mark.parametrize("K,N", [(8192, 10240), (8192, 8192), (8192, 57344), (28672, 8192)])
def test_w4a8_llama70b(K, N):
    """The Llama-3-70B layers at the W4A16 batch points (M = 1, 64, 256): every
    element at one token, whole tiles beyond."""
    W = syn.make_weight(N, K, seed=11 * K + N)
    wq = oracle.quantize_w4(W)
    lin = W4A8Linear(to_dev(W))
    for M in (1, 64, 256):
        _run(M, N, K, seed=M + 53, full=M == 1, W=W, wq=wq, lin=lin)
    del lin
    torch.cuda.empty_cache()


def test_w4a8_deterministic_and_workspace_left_zero():
    M, N, K = 16, 4096, 4096
    lin = W4A8Linear(to_dev(syn.make_weight(N, K, seed=7)))
    Xq, sx = lin.quant_act(to_dev(syn.make_act(M, K, seed=8)))
    a = lin.gemm(Xq, sx).clone()
    b = lin.gemm(Xq, sx).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert int(torch.count_nonzero(lin.ws.buf)) == 0


def test_w4a8_rejects_other_group_sizes():
    t = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QlinError) as e:
        q.qlin_w4a8_gemm(t, t, t, t, t, t, 1, 128, 128, 64, None, 0)
    assert e.value.status == 2
