"""MXFP8 on the GPU against the oracle, through the C ABI.

The quantiser (E4M3 codes, E8M0 block scales in the scale-atom layout) is
bit-exact with the oracle's MX quantiser; the GEMM, whose block scales are
applied by the tensor cores (tcgen05 kind::mxf8f6f4 with hardware block
scaling), stays within
    |Y - Y_ref| <= 2e-3 * ||X_deq[m, :]||_2 * ||W_deq[n, :]||_2
of the oracle's fp64 product of the MX-dequantised operands: on every element
up to 32 tokens, on whole tiles beyond (first, last and a random middle tile of
tokens x first, last and middle 128-row weight tiles).  Each GEMM case asserts
through the dispatch query which token tile and split count it reaches.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import MXFP8Linear

from _parity import blocks, check, host_f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    q.build()
    q.load()
    yield
    assert q.qlin_get_device_error() == 0


@pytest.mark.parametrize("R,K", [(1, 128), (7, 512), (33, 384), (300, 4096), (4096, 4096), (129, 14336)])
def test_quant_mxfp8_bit_exact(R, K):
    X = syn.make_act(R, K, seed=R + K, token_outlier_frac=0.01)
    X[0, :32] = 0                                 # an all-zero block: scale code 0
    X[R // 2, 64:96] = syn.f32_to_bf16_bits(np.full(32, 1e-39, np.float32))  # subnormal block: clamped exponent
    codes_r, scales_r = oracle.quant_mxfp8_rows(X)
    codes = torch.empty((R, K), dtype=torch.uint8, device="cuda")
    atoms = torch.full((q.qlin_mx_scale_bytes(R, K),), 0xAB, dtype=torch.uint8, device="cuda")
    q.qlin_quant_mxfp8(to_dev(X), R, K, codes, atoms)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), codes_r)
    assert np.array_equal(atoms.cpu().numpy(), oracle.mx_scales_atoms(scales_r))   # padding rows written as 0


# (id, M, N, K, token tile, split count)
GEMM_CASES = [
    ("bn32_m1", 1, 512, 1024, 32, 1),
    ("bn32_split", 16, 4096, 4096, 32, 3),
    ("bn32_m32", 32, 512, 1024, 32, 1),
    ("bn64", 100, 4096, 4096, 64, 1),
    ("bn64_split", 64, 4096, 14336, 64, 2),
    ("bn64_ragged", 300, 512, 1024, 64, 1),
    ("bn128", 128, 14336, 4096, 128, 1),
    ("bn128_ragged", 300, 4096, 4096, 128, 1),
    ("bn256_prefill", 2048, 4096, 4096, 256, 1),
    ("bn256_prefill_gateup", 2048, 28672, 4096, 256, 1),
    ("bn256_odd_atoms", 300, 14336, 4096, 256, 1),   # 3 token atoms: the last tile's second atom is past M
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=[c[0] for c in GEMM_CASES])
def test_mxfp8_gemm(case):
    name, M, N, K, bn, splits = case
    plan = q.qlin_plan_info(q.OP_MXFP8_GEMM, M, N, K)
    assert plan["kernel"] == q.KERNEL_MXFP8_TC
    assert (plan["tokens_per_tile"], plan["splits"]) == (bn, splits), plan
    seed = M + 3 * N + K
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    Xq_r, xs_r = oracle.quant_mxfp8_rows(X)
    Wq_r, ws_r = oracle.quant_mxfp8_rows(W)
    lin = MXFP8Linear(to_dev(W))
    Xq, xs = lin.quant_act(to_dev(X))
    torch.cuda.synchronize()
    assert np.array_equal(lin.Wq.cpu().numpy(), Wq_r) and np.array_equal(Xq.cpu().numpy(), Xq_r)
    Y = host_f64(lin.gemm(Xq, xs))
    sel = [(np.arange(M), np.arange(N))] if M <= 32 else blocks(M, N, bn, 128, seed)
    for ms, ns in sel:
        xd = oracle.mx_dequant(Xq_r[ms], xs_r[ms])
        wd = oracle.mx_dequant(Wq_r[ns], ws_r[ns])
        ref = oracle.w8a8_mx_full(Xq_r[ms], xs_r[ms], Wq_r[ns], ws_r[ns])
        check(Y[np.ix_(ms, ns)], ref, np.linalg.norm(xd, axis=1), np.linalg.norm(wd, axis=1), 0,
              "%s tile m%d n%d" % (name, ms[0], ns[0]))


def test_mxfp8_gemm_deterministic_and_workspace_left_zero():
    M, N, K = 16, 4096, 4096                      # split K: partial sums through the workspace
    lin = MXFP8Linear(to_dev(syn.make_weight(N, K, seed=3)))
    Xq, xs = lin.quant_act(to_dev(syn.make_act(M, K, seed=4)))
    a = lin.gemm(Xq, xs).clone()
    b = lin.gemm(Xq, xs).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert int(torch.count_nonzero(lin.ws.buf)) == 0


def test_mxfp8_rejects_bad_arguments():
    t = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QlinError) as e:
        q.qlin_quant_mxfp8(t, 1, 96, t, t)       # K % 128 != 0
    assert e.value.status == 2
    with pytest.raises(q.QlinError) as e:
        q.qlin_mxfp8_gemm(t, t, t, t, t, 1, 100, 128, None, 0)   # N % 128 != 0
    assert e.value.status == 2
    with pytest.raises(q.QlinError) as e:
        q.qlin_mxfp8_gemm(t, t[1:], t, t, t, 1, 128, 128, None, 0)   # misaligned scales
    assert e.value.status == 3
