"""GPU parity of libqlin against the CPU oracle, through the C ABI.

Bar (from the problem statement): packed codes / scales / zero-points and the
FP8 codes and scales are bit-exact; GEMM outputs satisfy
    |Y - Y_ref| <= 2e-3 * ||X_deq[m, :]||_2 * ||W_deq[n, :]||_2
against the oracle's fp64 result on the same quantised operands.
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


def bf16_out(Y: torch.Tensor) -> np.ndarray:
    return Y.float().cpu().numpy().astype(np.float64)


def norm_err(Y, Yref, xnorm, wnorm):
    den = xnorm[:, None] * wnorm[None, :]
    num = np.abs(Y - Yref)
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.where(den > 0, num / den, np.where(num == 0, 0.0, np.inf))
    return float(r.max()) if r.size else 0.0


# ------------------------------------------------------------------ packing

@pytest.mark.parametrize("N,K,sym,outl", [(512, 512, False, 0.0), (256, 1024, True, 0.01), (384, 2048, False, 0.01),
                                          (4096, 4096, False, 0.01), (4096, 14336, False, 0.01)])
def test_pack_w4_bit_exact(N, K, sym, outl):
    W = syn.make_weight(N, K, seed=N + K, outlier_frac=outl)
    W[:2, :128] = 0                     # degenerate all-zero groups
    wq = oracle.quantize_w4(W, G=128, symmetric=sym)
    c_ref, s_ref, z_ref = oracle.pack_tile(wq)
    layer = W4A16Linear(to_dev(W), symmetric=sym)
    torch.cuda.synchronize()
    assert np.array_equal(layer.codes.cpu().numpy(), c_ref)
    assert np.array_equal(layer.scales.cpu().numpy().view(np.uint16), s_ref)
    assert np.array_equal(layer.zeros.cpu().numpy(), z_ref)


# ------------------------------------------------------------------ FP8 quantisers

@pytest.mark.parametrize("M,K", [(1, 512), (7, 4096), (33, 14336), (2048, 4096)])
def test_quant_act_fp8_bit_exact(M, K):
    X = syn.make_act(M, K, seed=M * 7 + K, token_outlier_frac=0.01)
    X[M // 2, :] = 0
    Xq_ref, sx_ref = oracle.quant_fp8_rows(X)
    Xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    q.qlin_quant_act_fp8(to_dev(X), M, K, Xq, sx)
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))


@pytest.mark.parametrize("N,K", [(128, 512), (4096, 4096)])
def test_quant_w_fp8_bit_exact(N, K):
    W = syn.make_weight(N, K, seed=N + 3 * K)
    Wq_ref, sw_ref = oracle.quant_fp8_tensor(W)
    layer = W8A8Linear(to_dev(W))
    torch.cuda.synchronize()
    assert np.array_equal(layer.Wq.cpu().numpy(), Wq_ref)
    assert layer.sw.cpu().numpy()[0] == np.float32(sw_ref)


# ------------------------------------------------------------------ W4A16 GEMM

def _w4_full_case(M, N, K, path, seed, sym=False):
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.01)
    wq = oracle.quantize_w4(W, G=128, symmetric=sym)
    layer = W4A16Linear(to_dev(W), symmetric=sym)
    Y = bf16_out(layer(to_dev(X), path=path))
    Yref = oracle.w4a16_full(X, wq)
    xn = np.linalg.norm(syn.bf16_bits_to_f32(X).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.dequant_w4(wq), axis=1)
    return Y, Yref, xn, wn


def test_w4a16_tiny_config_both_paths():
    """M=1, K=512, N=512, G=128 asymmetric, seed 0."""
    for path in (q.PATH_GEMV, q.PATH_TC, q.PATH_AUTO):
        W = syn.make_weight(512, 512, seed=0, outlier_frac=0.0)
        X = syn.make_act(1, 512, seed=0)
        wq = oracle.quantize_w4(W)
        Y = bf16_out(W4A16Linear(to_dev(W))(to_dev(X), path=path))
        Yref = oracle.w4a16_full(X, wq)
        xn = np.linalg.norm(syn.bf16_bits_to_f32(X).astype(np.float64), axis=1)
        wn = np.linalg.norm(oracle.dequant_w4(wq), axis=1)
        assert norm_err(Y, Yref, xn, wn) <= TOL, path


@pytest.mark.parametrize("path", [q.PATH_GEMV, q.PATH_TC])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 16, 17, 33, 64, 100, 129, 256, 300])
def test_w4a16_m_sweep(path, M):
    Y, Yref, xn, wn = _w4_full_case(M, 256, 1024, path, seed=100 + M)
    assert norm_err(Y, Yref, xn, wn) <= TOL


@pytest.mark.parametrize("path", [q.PATH_GEMV, q.PATH_TC])
def test_w4a16_symmetric_and_deep_k(path):
    Y, Yref, xn, wn = _w4_full_case(16, 384, 4096, path, seed=5, sym=True)
    assert norm_err(Y, Yref, xn, wn) <= TOL


def _sampled_w4(M, N, K, path, seed, nsamp=1500):
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1)
    wq = oracle.quantize_w4(W)
    layer = W4A16Linear(to_dev(W))
    Y = bf16_out(layer(to_dev(X), path=path))
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, nsamp)
    ns = rng.integers(0, N, nsamp)
    ms[:2], ns[:2] = [M - 1, 0], [N - 1, 0]
    ref = oracle.w4a16_at(X, wq, ms, ns)
    xn = np.linalg.norm(syn.bf16_bits_to_f32(X).astype(np.float64), axis=1)[ms]
    deq_rows = oracle.dequant_w4(oracle.W4Quant(wq.q[ns], wq.s[ns], wq.z[ns], 128, False, 0))
    wn = np.linalg.norm(deq_rows, axis=1)
    err = np.abs(Y[ms, ns] - ref) / (xn * wn)
    return float(err.max()), layer, X


@pytest.mark.parametrize("K,N", [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a16_llama8b_decode_sampled(K, N, M):
    err, _, _ = _sampled_w4(M, N, K, q.PATH_AUTO, seed=K + N + M)
    assert err <= TOL


@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096), (8192, 10240)])
@pytest.mark.parametrize("M", [17, 24, 32])
def test_w4a16_mid_m_small_kernel_sampled(K, N, M):
    # 17 <= M <= 32 on the register-level MMA kernel (four token blocks), split-K clusters
    err, _, _ = _sampled_w4(M, N, K, q.PATH_GEMV, seed=K + N + M)
    assert err <= TOL


def test_w4a16_deterministic_split_k():
    _, layer, X = _sampled_w4(4, 4096, 14336, q.PATH_AUTO, seed=9, nsamp=10)
    Xd = to_dev(X)
    a = layer(Xd).clone()
    b = layer(Xd).clone()
    assert torch.equal(a, b)
    a = layer(Xd, path=q.PATH_TC).clone()
    b = layer(Xd, path=q.PATH_TC).clone()
    assert torch.equal(a, b)


# ------------------------------------------------------------------ W8A8 GEMM

def _w8_case(M, N, K, path, seed, nsamp=None):
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.001 if M >= 1000 else 0.05)
    Xq, sx = oracle.quant_fp8_rows(X)
    Wq, sw = oracle.quant_fp8_tensor(W)
    layer = W8A8Linear(to_dev(W))
    Y = bf16_out(layer(to_dev(X), path=path))
    tab = oracle.e4m3_table()
    if nsamp is None:
        Yref = oracle.w8a8_full(Xq, sx, Wq, sw)
        xn = np.linalg.norm(tab[Xq] * sx.astype(np.float64)[:, None], axis=1)
        wn = np.linalg.norm(tab[Wq] * float(sw), axis=1)
        return norm_err(Y, Yref, xn, wn)
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, nsamp)
    ns = rng.integers(0, N, nsamp)
    ref = oracle.w8a8_at(Xq, sx, Wq, sw, ms, ns)
    xn = np.linalg.norm(tab[Xq[ms]] * sx.astype(np.float64)[ms, None], axis=1)
    wn = np.linalg.norm(tab[Wq[ns]] * float(sw), axis=1)
    return float((np.abs(Y[ms, ns] - ref) / (xn * wn)).max())


@pytest.mark.parametrize("path", [q.PATH_GEMV, q.PATH_TC])
@pytest.mark.parametrize("M", [1, 2, 4, 5, 16, 17, 64, 200, 256, 257])
def test_w8a8_m_sweep(path, M):
    assert _w8_case(M, 256, 1024, path, seed=300 + M) <= TOL


@pytest.mark.parametrize("K,N", [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_w8a8_small_m_mma_kernel_sampled(K, N, M):
    # the register-level E4M3 MMA kernel (one or two token blocks, split-K clusters)
    assert _w8_case(M, N, K, q.PATH_GEMV, seed=K + N + M, nsamp=1500) <= TOL


@pytest.mark.parametrize("M,K,N", [(2048, 4096, 6144), (2048, 14336, 4096)])
def test_w8a8_prefill_sampled(M, K, N):
    assert _w8_case(M, N, K, q.PATH_AUTO, seed=M + K + N, nsamp=1500) <= TOL


# ------------------------------------------------------------------ boundary on device

def test_shared_workspace_mixed_shapes():
    """One workspace shared by calls of different shapes and kernels, twice over:
    each output equals the one computed with a private workspace, and the shared
    buffer is left all zero (the split-K counters, the work queue and the
    partial sums are all cleared by the calls that used them)."""
    w4 = [(1, 28672, 4096), (16, 4096, 14336), (4, 6144, 4096), (3, 512, 640), (64, 4096, 4096)]
    cases = []
    for i, (M, N, K) in enumerate(w4):
        lin = W4A16Linear(to_dev(syn.make_weight(N, K, seed=40 + i)))
        X = to_dev(syn.make_act(M, K, seed=50 + i))
        cases.append(("w4", M, N, K, lin, X, lin(X).clone()))
    lin8 = W8A8Linear(to_dev(syn.make_weight(4096, 4096, seed=60)))
    X8 = to_dev(syn.make_act(4, 4096, seed=61))
    Xq8, sx8 = lin8.quant_act(X8)
    cases.append(("w8", 4, 4096, 4096, lin8, (Xq8, sx8), lin8.gemm(Xq8, sx8).clone()))
    need = max(q.qlin_workspace_size(q.OP_W4A16_GEMM if c[0] == "w4" else q.OP_W8A8_GEMM, c[1], c[2], c[3])
               for c in cases)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        outs = []
        for kind, M, N, K, lin, X, _ in cases:
            Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            if kind == "w4":
                q.qlin_w4a16_gemm(X, lin.codes, lin.scales, lin.zeros, Y.view(torch.int16), M, N, K, 128, ws,
                                  ws.numel())
            else:
                q.qlin_w8a8_fp8_gemm(X[0], X[1], lin.Wq, lin.sw, Y.view(torch.int16), M, N, K, ws, ws.numel())
            outs.append(Y)
        torch.cuda.synchronize()
        for (kind, M, N, K, _, _, ref), Y in zip(cases, outs):
            assert torch.equal(Y, ref), (kind, M, N, K)
        assert int(torch.count_nonzero(ws)) == 0
    assert q.qlin_get_device_error() == 0


def test_workspace_too_small_and_empty():
    # K = 4224 is not a multiple of 256: the CUDA-core GEMV serves M = 4 and
    # keeps its split-K partial sums in the workspace
    K = 4224
    W = syn.make_weight(4096, K, seed=1)
    layer = W4A16Linear(to_dev(W))
    X = to_dev(syn.make_act(4, K, seed=2))
    Y = torch.empty((4, 4096), dtype=torch.bfloat16, device="cuda")
    need = q.qlin_workspace_size(q.OP_W4A16_GEMM, 4, 4096, K)
    assert need > 0
    with pytest.raises(q.QlinError) as e:
        q.qlin_w4a16_gemm(X, layer.codes, layer.scales, layer.zeros, Y.view(torch.int16), 4, 4096, K, 128,
                          None, 0)
    assert e.value.status == 4
    q.qlin_w4a16_gemm(X, layer.codes, layer.scales, layer.zeros, Y.view(torch.int16), 0, 4096, K, 128, None, 0)
    # the small-M tensor-core kernel adds its split-K sums in distributed shared memory: no workspace
    X4 = to_dev(syn.make_act(4, 4096, seed=3))
    lin = W4A16Linear(to_dev(syn.make_weight(4096, 4096, seed=4)))
    Y4 = torch.empty((4, 4096), dtype=torch.bfloat16, device="cuda")
    q.qlin_w4a16_gemm_ex(X4, lin.codes, lin.scales, lin.zeros, Y4.view(torch.int16), 4, 4096, 4096, 128, None, 0,
                         q.PATH_GEMV)
    torch.cuda.synchronize()
    assert torch.equal(Y4, lin(X4, path=q.PATH_GEMV))
    assert q.qlin_get_device_error() == 0


# ------------------------------------------------------------------ FP8 block scaling

from precision_quantized_linear_gb300.layers import W8A8BlockLinear  # noqa: E402


@pytest.mark.parametrize("M,K", [(1, 128), (7, 512), (300, 4096)])
def test_quant_act_fp8_blocks_bit_exact(M, K):
    X = syn.make_act(M, K, seed=M + K, token_outlier_frac=0.01)
    X[0, :128] = 0                                # an all-zero block
    q_ref, s_ref = oracle.quant_fp8_act_blocks(X)
    Xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    sx = torch.empty((K // 128, M), dtype=torch.float32, device="cuda")
    q.qlin_quant_act_fp8_blocks(to_dev(X), M, K, Xq, sx)
    torch.cuda.synchronize()
    assert np.array_equal(Xq.cpu().numpy(), q_ref)
    assert np.array_equal(sx.cpu().numpy(), s_ref)


@pytest.mark.parametrize("N,K", [(128, 128), (384, 1024), (4096, 4096)])
def test_quant_w_fp8_blocks_bit_exact(N, K):
    W = syn.make_weight(N, K, seed=N + K)
    W[:128, :128] = 0
    q_ref, s_ref = oracle.quant_fp8_weight_blocks(W)
    lin = W8A8BlockLinear(to_dev(W))
    torch.cuda.synchronize()
    assert np.array_equal(lin.Wq.cpu().numpy(), q_ref)
    assert np.array_equal(lin.sw.cpu().numpy(), s_ref)


def _w8b_case(M, N, K, seed, nsamp=None):
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.001)
    Xq_r, sx_r = oracle.quant_fp8_act_blocks(X)
    Wq_r, sw_r = oracle.quant_fp8_weight_blocks(W)
    lin = W8A8BlockLinear(to_dev(W))
    Xq, sx = lin.quant_act(to_dev(X))
    Y = bf16_out(lin.gemm(Xq, sx))
    assert np.array_equal(Xq.cpu().numpy(), Xq_r) and np.array_equal(sx.cpu().numpy()[:, :M], sx_r)
    tab = oracle.e4m3_table()
    xd = tab[Xq_r] * np.repeat(sx_r.T.astype(np.float64), 128, axis=1)
    wd = tab[Wq_r] * np.repeat(np.repeat(sw_r.astype(np.float64), 128, axis=0), 128, axis=1)
    xn, wn = np.linalg.norm(xd, axis=1), np.linalg.norm(wd, axis=1)
    if nsamp is None:
        ref = oracle.w8a8_blocks_full(Xq_r, sx_r, Wq_r, sw_r)
        return norm_err(Y, ref, xn, wn)
    rng = np.random.default_rng(seed)
    ms, ns = rng.integers(0, M, nsamp), rng.integers(0, N, nsamp)
    ref = oracle.w8a8_blocks_at(Xq_r, sx_r, Wq_r, sw_r, ms, ns)
    err = np.abs(Y[ms, ns] - ref) / (xn[ms] * wn[ns])
    return float(err.max())


@pytest.mark.parametrize("M", [1, 5, 16, 17, 64, 100, 129, 300])
def test_w8a8_block_gemm_m_sweep(M):
    assert _w8b_case(M, 512, 1024, seed=M + 31) <= TOL


@pytest.mark.parametrize("M,N,K", [(4, 4096, 4096), (16, 4096, 14336), (2048, 4096, 4096)])
def test_w8a8_block_gemm_llama_sampled(M, N, K):
    assert _w8b_case(M, N, K, seed=M + N, nsamp=1500) <= TOL


def test_w8a8_block_gemm_deterministic():
    W = syn.make_weight(512, 4096, seed=5)
    X = syn.make_act(3, 4096, seed=6)
    lin = W8A8BlockLinear(to_dev(W))
    a = lin(to_dev(X)).clone()
    b = lin(to_dev(X)).clone()
    assert torch.equal(a, b)
