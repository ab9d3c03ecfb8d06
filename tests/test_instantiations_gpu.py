"""Every tensor-core kernel instantiation against the oracle, reached on purpose.

The tcgen05 GEMM is compiled per (token tile BN, K blocks per stage, block
scaling, weight rows per tile, fused epilogue); which one a call runs is decided
by the planner.  Each case below names the instantiation it is meant to reach,
asserts through the dispatch query (qlin_plan_info) that the call plans onto
it, runs the call through the C ABI and compares the output with the oracle:
every element up to 32 tokens, otherwise whole tiles (first, last and a
random middle tile of tokens x first, last and middle 128-row weight tiles).
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import W4A16Linear, W8A8BlockLinear, W8A8Linear

from _parity import bias_bits, check, check_w4, check_w8, host_f64, to_dev, tile_starts

pytestmark = pytest.mark.gpu

NONE, SILU, GELU = q.ACT_NONE, q.ACT_SILU, q.ACT_GELU


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    q.load()
    yield
    assert q.qlin_get_device_error() == 0


def _plan(op, M, N, K, path):
    return q.qlin_plan_info(op, M, N, K, 128, path)


# (id, M, N, K, act, expected plan fields) -- W4A16 on QLIN_PATH_TC:
# tc_gemm_kernel<BN, W4 = true, KPS, BS = false, WN = 128, EPI = act != none>
W4_TC = [
    ("bn16_kps4", 16, 512, 1024, NONE, dict(tokens_per_tile=16, kblocks_per_stage=4, a_in_tmem=1, splits=1)),
    ("bn16_kps4_split", 1, 512, 4096, NONE, dict(tokens_per_tile=16, kblocks_per_stage=4, splits=2)),
    ("bn16_kps2", 9, 512, 4224, NONE, dict(tokens_per_tile=16, kblocks_per_stage=2, splits=3)),
    ("bn32_kps4", 20, 512, 1024, NONE, dict(tokens_per_tile=32, kblocks_per_stage=4)),
    ("bn32_kps4_split", 20, 6144, 4096, NONE, dict(tokens_per_tile=32, kblocks_per_stage=4, splits=2)),
    ("bn32_kps2", 20, 6144, 4224, NONE, dict(tokens_per_tile=32, kblocks_per_stage=2, splits=2)),
    ("bn64", 40, 14336, 1024, NONE, dict(tokens_per_tile=64, kblocks_per_stage=2, splits=1)),
    ("bn64_split", 40, 6144, 8192, NONE, dict(tokens_per_tile=64, splits=3)),
    ("bn128", 300, 4096, 1024, NONE, dict(tokens_per_tile=128, kblocks_per_stage=2, a_in_tmem=1, splits=1)),
    ("bn128_split", 100, 6144, 14336, NONE, dict(tokens_per_tile=128, kblocks_per_stage=2, splits=3)),
    ("bn256", 160, 14336, 4096, NONE, dict(tokens_per_tile=256, kblocks_per_stage=1, a_in_tmem=0, splits=1)),
    ("bn16_kps4_epi", 5, 512, 1024, SILU, dict(tokens_per_tile=16, kblocks_per_stage=4)),
    ("bn16_kps2_epi", 3, 512, 4224, GELU, dict(tokens_per_tile=16, kblocks_per_stage=2)),
    ("bn32_kps4_epi", 20, 6144, 4096, GELU, dict(tokens_per_tile=32, kblocks_per_stage=4, splits=2)),
    ("bn32_kps2_epi", 20, 6144, 4224, SILU, dict(tokens_per_tile=32, kblocks_per_stage=2)),
    ("bn64_split_epi", 40, 6144, 8192, SILU, dict(tokens_per_tile=64, splits=3)),
    ("bn128_epi", 300, 4096, 1024, GELU, dict(tokens_per_tile=128, kblocks_per_stage=2)),
    ("bn128_split_epi", 100, 6144, 14336, SILU, dict(tokens_per_tile=128, splits=3)),
    ("bn256_epi", 160, 14336, 4096, SILU, dict(tokens_per_tile=256, splits=1)),
]


@pytest.mark.parametrize("case", W4_TC, ids=[c[0] for c in W4_TC])
def test_w4a16_tc_instantiation(case):
    name, M, N, K, act, want = case
    plan = _plan(q.OP_W4A16_GEMM, M, N, K, q.PATH_TC)
    assert plan["kernel"] == q.KERNEL_W4A16_TC
    for k, v in want.items():
        assert plan[k] == v, (name, k, plan)
    seed = M * 7 + N + K + act
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    wq = oracle.quantize_w4(W)
    bias = bias_bits(N, seed) if act else None
    lin = W4A16Linear(to_dev(W), bias=None if bias is None else to_dev(bias).view(torch.bfloat16))
    Y = host_f64(lin(to_dev(X), path=q.PATH_TC, act=act))
    check_w4(Y, X, wq, full=M <= 32, tm=plan["tokens_per_tile"], seed=seed, bias=bias, act=act)


# W8A8 on QLIN_PATH_TC: tc_gemm_kernel<BN, W4 = false, 1, BS = false, 128, EPI>
W8_TC = [
    ("bn16", 16, 512, 1024, NONE, dict(tokens_per_tile=16)),
    ("bn16_split", 4, 4096, 4096, NONE, dict(tokens_per_tile=16, splits=3)),
    ("bn32", 32, 512, 1024, NONE, dict(tokens_per_tile=32)),
    ("bn64", 64, 4096, 4096, NONE, dict(tokens_per_tile=64, splits=1)),
    ("bn64_split", 64, 4096, 14336, NONE, dict(tokens_per_tile=64, splits=2)),
    ("bn128", 128, 14336, 4096, NONE, dict(tokens_per_tile=128, splits=1)),
    ("bn256", 512, 14336, 4096, NONE, dict(tokens_per_tile=256, splits=1)),
    ("bn16_epi", 7, 512, 1024, GELU, dict(tokens_per_tile=16)),
    ("bn32_epi", 30, 512, 1024, SILU, dict(tokens_per_tile=32)),
    ("bn64_split_epi", 64, 4096, 14336, SILU, dict(tokens_per_tile=64, splits=2)),
    ("bn128_epi", 128, 14336, 4096, GELU, dict(tokens_per_tile=128)),
    ("bn256_epi", 512, 14336, 4096, SILU, dict(tokens_per_tile=256)),
]


@pytest.mark.parametrize("case", W8_TC, ids=[c[0] for c in W8_TC])
def test_w8a8_tc_instantiation(case):
    name, M, N, K, act, want = case
    plan = _plan(q.OP_W8A8_GEMM, M, N, K, q.PATH_TC)
    assert plan["kernel"] == q.KERNEL_W8A8_TC
    for k, v in want.items():
        assert plan[k] == v, (name, k, plan)
    seed = M * 5 + N + 3 * K + act
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    Xq, sx = oracle.quant_fp8_rows(X)
    Wq, sw = oracle.quant_fp8_tensor(W)
    bias = bias_bits(N, seed) if act else None
    lin = W8A8Linear(to_dev(W), bias=None if bias is None else to_dev(bias).view(torch.bfloat16))
    Y = host_f64(lin(to_dev(X), path=q.PATH_TC, act=act))
    check_w8(Y, Xq, sx, Wq, sw, full=M <= 32, tm=plan["tokens_per_tile"], seed=seed, bias=bias, act=act)


# Block-scaled W8A8: tc_gemm_kernel<BN, false, 1, BS = true, WN, false>
BLOCK_TC = [
    ("bn16", 16, 512, 1024, dict(tokens_per_tile=16, rows_per_tile=128)),
    ("bn16_split", 5, 4096, 4096, dict(tokens_per_tile=16, splits=3)),
    ("bn32", 32, 512, 1024, dict(tokens_per_tile=32, rows_per_tile=128)),
    ("bn64", 64, 4096, 4096, dict(tokens_per_tile=64, splits=3)),
    ("bn128_wn128", 200, 4096, 4096, dict(tokens_per_tile=128, rows_per_tile=128, splits=1)),
    ("bn128_wn128_split", 100, 4096, 14336, dict(tokens_per_tile=128, rows_per_tile=128, splits=2)),
    ("bn128_wn256", 256, 28672, 4096, dict(tokens_per_tile=128, rows_per_tile=256, splits=1)),
]


@pytest.mark.parametrize("case", BLOCK_TC, ids=[c[0] for c in BLOCK_TC])
def test_w8a8_block_tc_instantiation(case):
    name, M, N, K, want = case
    plan = _plan(q.OP_W8A8_BLOCK_GEMM, M, N, K, q.PATH_AUTO)
    assert plan["kernel"] == q.KERNEL_W8A8_BLOCK_TC
    for k, v in want.items():
        assert plan[k] == v, (name, k, plan)
    seed = M + N + K
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    Xq_r, sx_r = oracle.quant_fp8_act_blocks(X)
    Wq_r, sw_r = oracle.quant_fp8_weight_blocks(W)
    lin = W8A8BlockLinear(to_dev(W))
    Xq, sx = lin.quant_act(to_dev(X))
    Y = host_f64(lin.gemm(Xq, sx))
    tab = oracle.e4m3_table()
    tm = plan["tokens_per_tile"]
    mblocks = [np.arange(M)] if M <= 32 else [np.arange(m0, min(M, m0 + tm)) for m0 in tile_starts(M, tm, seed)]
    nblocks = [np.arange(n0, n0 + 128) for n0 in tile_starts(N, 128, seed + 1)]
    for ms in mblocks:
        for ns in nblocks:
            kb = K // 128
            xs = sx_r[:, ms]                                   # [K/128][m]
            ws = sw_r[ns // 128]                               # [n][K/128]
            ref = np.zeros((ms.size, ns.size))
            for b in range(kb):
                part = oracle.gemm_nt_f64(np.ascontiguousarray(tab[Xq_r[ms, b * 128:(b + 1) * 128]]),
                                          np.ascontiguousarray(tab[Wq_r[ns, b * 128:(b + 1) * 128]]))
                ref += part * xs[b].astype(np.float64)[:, None] * ws[:, b].astype(np.float64)[None, :]
            xd = tab[Xq_r[ms]] * np.repeat(xs.T.astype(np.float64), 128, axis=1)
            wd = tab[Wq_r[ns]] * np.repeat(ws.astype(np.float64), 128, axis=1)
            check(Y[np.ix_(ms, ns)], ref, np.linalg.norm(xd, axis=1), np.linalg.norm(wd, axis=1), 0,
                  "tile m%d n%d" % (ms[0], ns[0]))


@pytest.mark.parametrize("M", [1, 3, 7])
def test_w8a8_gemv_k_not_256(M):
    # K % 256 != 0 on the small-M path: the CUDA-core E4M3 GEMV with its split-K sums in the workspace
    N, K = 512, 4224
    plan = _plan(q.OP_W8A8_GEMM, M, N, K, q.PATH_GEMV)
    assert plan["kernel"] == q.KERNEL_W8A8_GEMV
    W = syn.make_weight(N, K, seed=M + 70)
    X = syn.make_act(M, K, seed=M + 71)
    Xq, sx = oracle.quant_fp8_rows(X)
    Wq, sw = oracle.quant_fp8_tensor(W)
    Y = host_f64(W8A8Linear(to_dev(W))(to_dev(X), path=q.PATH_GEMV))
    check_w8(Y, Xq, sx, Wq, sw, full=True, tm=16, seed=M)
