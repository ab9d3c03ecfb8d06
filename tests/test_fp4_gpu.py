"""FP4 (E2M1, [LP] S10) on the GPU against the oracle, through the C ABI.

MXFP4 (E8M0 scale per 32 columns, tcgen05 kind::mxf4) and NVFP4 (E4M3 scale
per 16 columns plus an FP32 scale per tensor, tcgen05 kind::mxf4nvf4).  The
quantisers (packed E2M1 codes, the scale atoms, the NVFP4 tensor scale) are
bit-exact with the oracle's; the GEMMs, whose block scales are applied by the
tensor cores, stay within
    |Y - Y_ref| <= 2e-3 * ||X_deq[m, :]||_2 * ||W_deq[n, :]||_2
of the oracle's fp64 product of the dequantised operands: on every element up
to 32 tokens, on whole tiles beyond (first, last and a random middle tile of
tokens x first, last and middle 128-row weight tiles).  Each GEMM case asserts
through the dispatch query which token tile and split count it reaches.
"""
import numpy as np
import pytest
import torch

import oracle
import precision_quantized_linear_gb300 as q
from precision_quantized_linear_gb300 import synthetic as syn
from precision_quantized_linear_gb300.layers import MXFP4Linear, NVFP4Linear

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


def _edge_rows(X, R):
    """An all-zero block, a block below 2^-126 and a block of tiny negative values."""
    X[0, :32] = 0
    X[R // 2, 64:96] = syn.f32_to_bf16_bits(np.full(32, 1e-39, np.float32))
    X[R - 1, 32:64] = syn.f32_to_bf16_bits(np.linspace(-1e-3, -1e-6, 32).astype(np.float32))
    X[R - 1, 32] = syn.f32_to_bf16_bits(np.array([5.0], np.float32))[0]   # the same block: -tiny / X rounds to -0
    return X


@pytest.mark.parametrize("R,K", [(1, 256), (7, 512), (300, 4096), (129, 14336), (4096, 4096)])
def test_quant_mxfp4_bit_exact(R, K):
    X = _edge_rows(syn.make_act(R, K, seed=R + K, token_outlier_frac=0.01), R)
    codes_r, scales_r = oracle.quant_mxfp4_rows(X)
    codes = torch.full((R, K // 2), 0xAB, dtype=torch.uint8, device="cuda")
    atoms = torch.full((q.qlin_mx_scale_bytes(R, K),), 0xAB, dtype=torch.uint8, device="cuda")
    q.qlin_quant_mxfp4(to_dev(X), R, K, codes, atoms)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), oracle.pack_fp4(codes_r))
    assert np.array_equal(atoms.cpu().numpy(), oracle.mx_scales_atoms(scales_r))   # padding rows written as 0


@pytest.mark.parametrize("R,K", [(1, 256), (300, 4096), (4096, 14336)])
def test_nvfp4_tensor_scale_bit_exact(R, K):
    X = syn.make_act(R, K, seed=3 * R + K, token_outlier_frac=0.01)
    sg = torch.full((4,), -1.0, dtype=torch.float32, device="cuda")
    q.qlin_nvfp4_tensor_scale(to_dev(X), R * K, sg)
    torch.cuda.synchronize()
    assert np.float32(sg[0].item()) == np.float32(oracle.nvfp4_global_scale(X))
    q.qlin_nvfp4_tensor_scale(to_dev(np.zeros((R, K), np.uint16)), R * K, sg)   # all zero: 1
    torch.cuda.synchronize()
    assert sg[0].item() == 1.0


@pytest.mark.parametrize("R,K", [(1, 256), (7, 512), (300, 4096), (129, 14336), (4096, 4096)])
def test_quant_nvfp4_bit_exact(R, K):
    X = _edge_rows(syn.make_act(R, K, seed=R + 2 * K, token_outlier_frac=0.01), R)
    X[R // 3, 128:144] = syn.f32_to_bf16_bits(np.full(16, 1e-4, np.float32))   # a block whose E4M3 scale is 0
    Xd = to_dev(X)
    sg = torch.empty(4, dtype=torch.float32, device="cuda")
    q.qlin_nvfp4_tensor_scale(Xd, R * K, sg)
    codes = torch.full((R, K // 2), 0xAB, dtype=torch.uint8, device="cuda")
    atoms = torch.full((q.qlin_nvfp4_scale_bytes(R, K),), 0xAB, dtype=torch.uint8, device="cuda")
    q.qlin_quant_nvfp4(Xd, R, K, sg, codes, atoms)
    torch.cuda.synchronize()
    sg_r = oracle.nvfp4_global_scale(X)
    assert np.float32(sg[0].item()) == np.float32(sg_r)
    codes_r, scales_r = oracle.quant_nvfp4_rows(X, sg_r)
    assert np.array_equal(codes.cpu().numpy(), oracle.pack_fp4(codes_r))
    assert np.array_equal(atoms.cpu().numpy(), oracle.mx_scales_atoms(scales_r))


def test_quant_nvfp4_rounding_ties():
    """Quotients v / (sb sg) exactly on the E2M1 rounding midpoints (0.25, 0.75,
    1.25, 1.75, 2.5, 3.5, 5: ties to even) and one BF16 step either side of
    them, with block scales 1, 0.5 and 448 and the tensor scale 1: the
    quantiser's codes against the oracle's."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    K = 256
    rows = []
    for den in (1.0, 0.5, 2.0):            # block amax 6 den -> E4M3 scale den (exact), tensor scale 1
        for off in (-1, 0, 1):             # BF16 steps off the midpoint
            v = (mids * den).astype(np.float32)
            b = syn.f32_to_bf16_bits(v).astype(np.int32) + off
            blk = np.concatenate([syn.f32_to_bf16_bits(np.array([6.0 * den], np.float32)).astype(np.int32), b,
                                  b | 0x8000, [0]]).astype(np.uint16)   # amax, the 7 values, their negatives, 0
            row = np.zeros(K, np.uint16)
            row[:16] = blk
            row[16:32] = blk ^ 0x8000
            rows.append(row)
    X = np.stack(rows)
    X[0, 64] = syn.f32_to_bf16_bits(np.array([2688.0], np.float32))[0]   # tensor amax 2688: sg = 1
    R = X.shape[0]
    Xd = to_dev(X)
    sg = torch.empty(4, dtype=torch.float32, device="cuda")
    q.qlin_nvfp4_tensor_scale(Xd, R * K, sg)
    codes = torch.empty((R, K // 2), dtype=torch.uint8, device="cuda")
    atoms = torch.empty((q.qlin_nvfp4_scale_bytes(R, K),), dtype=torch.uint8, device="cuda")
    q.qlin_quant_nvfp4(Xd, R, K, sg, codes, atoms)
    torch.cuda.synchronize()
    sg_r = oracle.nvfp4_global_scale(X)
    assert np.float32(sg_r) == np.float32(1.0)
    codes_r, scales_r = oracle.quant_nvfp4_rows(X, sg_r)
    assert np.array_equal(codes.cpu().numpy(), oracle.pack_fp4(codes_r))
    assert np.array_equal(atoms.cpu().numpy(), oracle.mx_scales_atoms(scales_r))


# (id, M, N, K, token tile, split count)
GEMM_CASES = [
    ("bn32_m1", 1, 512, 1024, 32, 1),
    ("bn32_split", 1, 512, 4096, 32, 4),
    ("bn32_m16", 16, 4096, 4096, 32, 1),
    ("bn32_m8_split", 8, 4096, 14336, 32, 3),
    ("bn32_m32", 32, 512, 1024, 32, 1),
    ("bn128_m40", 40, 512, 1024, 128, 1),          # 33 .. 64 tokens: a 128-token tile (no 64-token FP4 tiles)
    ("bn128_split", 40, 512, 53248, 128, 3),
    ("bn128", 100, 14336, 4096, 128, 1),
    ("bn128_ragged", 300, 512, 1024, 128, 1),
    ("bn256_prefill", 2048, 4096, 4096, 256, 1),
    ("bn256_prefill_gateup", 2048, 28672, 4096, 256, 1),
    ("bn256_odd_atoms", 300, 14336, 8192, 256, 1),   # 3 token atoms: the last tile's second atom is past M
]


def _operands(M, N, K, seed):
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    return W, X


@pytest.mark.parametrize("case", GEMM_CASES, ids=[c[0] for c in GEMM_CASES])
def test_mxfp4_gemm(case):
    name, M, N, K, bn, splits = case
    plan = q.qlin_plan_info(q.OP_MXFP4_GEMM, M, N, K)
    assert plan["kernel"] == q.KERNEL_MXFP4_TC
    assert (plan["tokens_per_tile"], plan["splits"]) == (bn, splits), plan
    seed = M + 5 * N + K
    W, X = _operands(M, N, K, seed)
    Xq_r, xs_r = oracle.quant_mxfp4_rows(X)
    Wq_r, ws_r = oracle.quant_mxfp4_rows(W)
    lin = MXFP4Linear(to_dev(W))
    Xq, xs = lin.quant_act(to_dev(X))
    torch.cuda.synchronize()
    assert np.array_equal(lin.Wq.cpu().numpy(), oracle.pack_fp4(Wq_r))
    assert np.array_equal(Xq.cpu().numpy(), oracle.pack_fp4(Xq_r))
    Y = host_f64(lin.gemm(Xq, xs))
    sel = [(np.arange(M), np.arange(N))] if M <= 32 else blocks(M, N, bn, 128, seed)
    for ms, ns in sel:
        xd = oracle.mxfp4_dequant(Xq_r[ms], xs_r[ms])
        wd = oracle.mxfp4_dequant(Wq_r[ns], ws_r[ns])
        ref = oracle.w4a4_mx_full(Xq_r[ms], xs_r[ms], Wq_r[ns], ws_r[ns])
        check(Y[np.ix_(ms, ns)], ref, np.linalg.norm(xd, axis=1), np.linalg.norm(wd, axis=1), 0,
              "%s tile m%d n%d" % (name, ms[0], ns[0]))


@pytest.mark.parametrize("case", GEMM_CASES, ids=[c[0] for c in GEMM_CASES])
def test_nvfp4_gemm(case):
    name, M, N, K, bn, splits = case
    plan = q.qlin_plan_info(q.OP_NVFP4_GEMM, M, N, K)
    assert plan["kernel"] == q.KERNEL_NVFP4_TC
    assert (plan["tokens_per_tile"], plan["splits"]) == (bn, splits), plan
    seed = M + 7 * N + K
    W, X = _operands(M, N, K, seed)
    sgx, sgw = oracle.nvfp4_global_scale(X), oracle.nvfp4_global_scale(W)
    Xq_r, xs_r = oracle.quant_nvfp4_rows(X, sgx)
    Wq_r, ws_r = oracle.quant_nvfp4_rows(W, sgw)
    lin = NVFP4Linear(to_dev(W))
    Xq, xs, sgx_d = lin.quant_act(to_dev(X))
    torch.cuda.synchronize()
    assert np.float32(sgx_d[0].item()) == np.float32(sgx) and np.float32(lin.sgw[0].item()) == np.float32(sgw)
    assert np.array_equal(lin.Wq.cpu().numpy(), oracle.pack_fp4(Wq_r))
    assert np.array_equal(Xq.cpu().numpy(), oracle.pack_fp4(Xq_r))
    Y = host_f64(lin.gemm(Xq, xs, sgx_d))
    sel = [(np.arange(M), np.arange(N))] if M <= 32 else blocks(M, N, bn, 128, seed)
    for ms, ns in sel:
        xd = oracle.nvfp4_dequant(Xq_r[ms], xs_r[ms], sgx)
        wd = oracle.nvfp4_dequant(Wq_r[ns], ws_r[ns], sgw)
        ref = oracle.w4a4_nv_full(Xq_r[ms], xs_r[ms], sgx, Wq_r[ns], ws_r[ns], sgw)
        check(Y[np.ix_(ms, ns)], ref, np.linalg.norm(xd, axis=1), np.linalg.norm(wd, axis=1), 0,
              "%s tile m%d n%d" % (name, ms[0], ns[0]))


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_fp4_gemm_deterministic_and_workspace_left_zero(fmt):
    M, N, K = 8, 4096, 14336                      # split K: partial sums through the workspace
    W = to_dev(syn.make_weight(N, K, seed=11))
    X = to_dev(syn.make_act(M, K, seed=12))
    if fmt == "mxfp4":
        lin = MXFP4Linear(W)
        ops = lin.quant_act(X)
    else:
        lin = NVFP4Linear(W)
        ops = lin.quant_act(X)
    a = lin.gemm(*ops).clone()
    b = lin.gemm(*ops).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert int(torch.count_nonzero(lin.ws.buf)) == 0


def test_fp4_rejects_bad_arguments():
    t = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    f = torch.ones(4, dtype=torch.float32, device="cuda")
    with pytest.raises(q.QlinError) as e:
        q.qlin_quant_mxfp4(t, 1, 128, t, t)       # K % 256 != 0
    assert e.value.status == 2
    with pytest.raises(q.QlinError) as e:
        q.qlin_quant_nvfp4(t, 1, 384, f, t, t)    # K % 256 != 0
    assert e.value.status == 2
    with pytest.raises(q.QlinError) as e:
        q.qlin_mxfp4_gemm(t, t, t, t, t, 1, 128, 384, None, 0)   # K % 256 != 0
    assert e.value.status == 2
    with pytest.raises(q.QlinError) as e:
        q.qlin_nvfp4_gemm(t, t, f, t, t, f, t, 1, 100, 256, None, 0)   # N % 128 != 0
    assert e.value.status == 2
    with pytest.raises(q.QlinError) as e:
        q.qlin_mxfp4_gemm(t, t[1:], t, t, t, 1, 128, 256, None, 0)   # misaligned scales
    assert e.value.status == 3
    with pytest.raises(q.QlinError) as e:
        q.qlin_nvfp4_tensor_scale(t, 12, f)     # n % 8 != 0
    assert e.value.status == 2
