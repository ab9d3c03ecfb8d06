"""GPU parity of the fused output epilogue (bias + activation) against the oracle.

Y = bf16(act(acc + bias[n])) on every kernel path of the W4A16 and W8A8 GEMMs,
and on every tile kind of the MXFP8, MXFP4, NVFP4 and W4A8 GEMMs.  Bar: the
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
from precision_quantized_linear_gb300.layers import (MXFP4Linear, MXFP8Linear, NVFP4Linear, W4A8Linear, W4A16Linear,
                                                      W8A8BlockLinear, W8A8Linear)

from _parity import blocks, w4_rows

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


# ------------------------------------------------------------------ block formats and W4A8
# The same epilogue on the MXFP8, MXFP4, NVFP4 and W4A8 GEMMs, on every tile
# kind they plan: the single token block of up to 32 tokens, 64- / 128-token
# tiles, split K ranges (the reduction applies it), and the 256-token tiles of
# the block formats, whose epilogue drains the single accumulator into
# registers before writing.  (M, N, K, activation, bias); the dispatch query
# asserts the tile each case is meant to reach.
FMT_CASES = [(16, 512, 1024, q.ACT_SILU, True), (100, 512, 1024, q.ACT_GELU, True),
             (8, 512, 14336, q.ACT_RELU, False), (2048, 4096, 4096, q.ACT_NONE, True)]
FMT_OPS = {"mxfp8": q.OP_MXFP8_GEMM, "mxfp4": q.OP_MXFP4_GEMM, "nvfp4": q.OP_NVFP4_GEMM, "w4a8": q.OP_W4A8_GEMM,
           "w8a8b": q.OP_W8A8_BLOCK_GEMM}
# token tile each (format, M) of FMT_CASES is planned onto
FMT_TILE = {"mxfp8": {16: 32, 100: 64, 8: 32, 2048: 256}, "mxfp4": {16: 32, 100: 128, 8: 32, 2048: 256},
            "nvfp4": {16: 32, 100: 128, 8: 32, 2048: 256}, "w4a8": {16: 16, 100: 64, 8: 16, 2048: 64},
            "w8a8b": {16: 16, 100: 128, 8: 16, 2048: 128}}


def _fmt_oracle(fmt, X, W):
    """(reference of rows ms x columns ns, X dequantised row norms, W dequantised norms of rows ns)."""
    if fmt == "mxfp8":
        Xq, xs = oracle.quant_mxfp8_rows(X)
        Wq, ws = oracle.quant_mxfp8_rows(W)
        xn = np.linalg.norm(oracle.mx_dequant(Xq, xs), axis=1)
        return (lambda ms, ns: oracle.w8a8_mx_full(Xq[ms], xs[ms], Wq[ns], ws[ns]), xn,
                lambda ns: np.linalg.norm(oracle.mx_dequant(Wq[ns], ws[ns]), axis=1))
    if fmt == "mxfp4":
        Xq, xs = oracle.quant_mxfp4_rows(X)
        Wq, ws = oracle.quant_mxfp4_rows(W)
        xn = np.linalg.norm(oracle.mxfp4_dequant(Xq, xs), axis=1)
        return (lambda ms, ns: oracle.w4a4_mx_full(Xq[ms], xs[ms], Wq[ns], ws[ns]), xn,
                lambda ns: np.linalg.norm(oracle.mxfp4_dequant(Wq[ns], ws[ns]), axis=1))
    if fmt == "nvfp4":
        sgx, sgw = oracle.nvfp4_global_scale(X), oracle.nvfp4_global_scale(W)
        Xq, xs = oracle.quant_nvfp4_rows(X, sgx)
        Wq, ws = oracle.quant_nvfp4_rows(W, sgw)
        xn = np.linalg.norm(oracle.nvfp4_dequant(Xq, xs, sgx), axis=1)
        return (lambda ms, ns: oracle.w4a4_nv_full(Xq[ms], xs[ms], sgx, Wq[ns], ws[ns], sgw), xn,
                lambda ns: np.linalg.norm(oracle.nvfp4_dequant(Wq[ns], ws[ns], sgw), axis=1))
    if fmt == "w8a8b":  # 1 x 128 token blocks (sx [K/128][M]), 128 x 128 weight blocks (sw [N/128][K/128])
        tab = oracle.e4m3_table()
        Xq, sx = oracle.quant_fp8_act_blocks(X)
        Wq, sw = oracle.quant_fp8_weight_blocks(W)
        xn = np.linalg.norm(tab[Xq] * np.repeat(sx.T.astype(np.float64), 128, axis=1), axis=1)
        swr = lambda ns: sw[ns[0] // 128: ns[-1] // 128 + 1]  # the scale rows of whole 128-row tiles ns
        return (lambda ms, ns: oracle.w8a8_blocks_full(Xq[ms], sx[:, ms], Wq[ns], swr(ns)), xn,
                lambda ns: np.linalg.norm(tab[Wq[ns]] * np.repeat(np.repeat(swr(ns).astype(np.float64), 128, axis=0),
                                                                 128, axis=1), axis=1))
    Xq, sx = oracle.quant_fp8_rows(X)
    wq = oracle.quantize_w4(W)
    xn = np.linalg.norm(oracle.e4m3_table()[Xq] * sx.astype(np.float64)[:, None], axis=1)
    return (lambda ms, ns: oracle.w4a8_full(Xq[ms], sx[ms], w4_rows(wq, ns)), xn,
            lambda ns: np.linalg.norm(oracle.dequant_w4(w4_rows(wq, ns)), axis=1))


@pytest.mark.parametrize("fmt", list(FMT_OPS))
@pytest.mark.parametrize("case", FMT_CASES, ids=["m%d_n%d_k%d" % c[:3] for c in FMT_CASES])
def test_block_formats_fused_epilogue(fmt, case):
    M, N, K, act, with_bias = case
    plan = q.qlin_plan_info(FMT_OPS[fmt], M, N, K)
    assert plan["tokens_per_tile"] == FMT_TILE[fmt][M] and (plan["splits"] > 1) == (K == 14336), plan
    seed = M + N + K + act + len(fmt)
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    bias = _bias(N, seed=seed + 2) if with_bias else None
    dbias = to_dev(bias).view(torch.bfloat16) if bias is not None else None
    dW, dX = to_dev(W).view(torch.bfloat16), to_dev(X).view(torch.bfloat16)
    lin = {"mxfp8": MXFP8Linear, "mxfp4": MXFP4Linear, "nvfp4": NVFP4Linear, "w4a8": W4A8Linear,
           "w8a8b": W8A8BlockLinear}[fmt](dW, bias=dbias)
    Y = lin(dX, act=act).float().cpu().numpy().astype(np.float64)
    ref, xn, wn_of = _fmt_oracle(fmt, X, W)
    sel = [(np.arange(M), np.arange(N))] if M * N <= 1 << 16 else blocks(M, N, plan["tokens_per_tile"], 128, seed)
    for ms, ns in sel:
        Yref = oracle.epilogue(ref(ms, ns), None if bias is None else bias[ns], act)
        check(Y[np.ix_(ms, ns)], Yref, xn[ms], wn_of(ns))


def test_block_scaled_fused_epilogue_token_major_split():
    """Block-scaled FP8 at 128 tokens runs token-major (thread = token, bias per
    column); with two K ranges the reduction applies the epilogue."""
    M, N, K, act = 100, 512, 14336, q.ACT_SILU
    plan = q.qlin_plan_info(q.OP_W8A8_BLOCK_GEMM, M, N, K)
    assert (plan["tokens_per_tile"], plan["splits"]) == (128, 2), plan
    W = syn.make_weight(N, K, seed=91)
    X = syn.make_act(M, K, seed=92, token_outlier_frac=0.01)
    bias = _bias(N, seed=93)
    lin = W8A8BlockLinear(to_dev(W).view(torch.bfloat16), bias=to_dev(bias).view(torch.bfloat16))
    Y = lin(to_dev(X).view(torch.bfloat16), act=act).float().cpu().numpy().astype(np.float64)
    ref, xn, wn_of = _fmt_oracle("w8a8b", X, W)
    ns = np.arange(N)
    check(Y, oracle.epilogue(ref(np.arange(M), ns), bias, act), xn, wn_of(ns))

