"""qlin oracle -- TEST INFRASTRUCTURE ONLY.

A plain CPU statement (C, fp64 accumulation) of the quantized linear layer
Y = X . deq(W)^T in its two variants, used to check the CUDA library.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the product package never does, and the two
share no code.  Every function cites the passage of the source pages it
follows (see ``qlin_oracle.c`` for the list):

  [LP] "Low-precision LLM inference: FP8/INT8/INT4/FP4 kernels and
       calibration" -- S2 uniform quantisation, S3 symmetric/asymmetric,
       S4 granularity, S5 effective bits, S7 E4M3, S8 FP8 current scaling,
       S10 FP4 E2M1 and the block formats (MXFP8 and MXFP4 after the OCP
       Microscaling spec v1.0, NVFP4 after its vendor's two-level recipe:
       ``quant_mxfp8_rows``, ``quant_mxfp4_rows``, ``quant_nvfp4_rows``
       below), S22 accumulator precision, S23/S24 fused
       bias / activation epilogue (``epilogue`` below).
  [TP] "Quantization throughput by batch size: why W4A16 is overtaken by
       W8A8" -- the arithmetic-intensity roofline (``roofline_*`` below).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force, exhaustive code tables and library
routines; no function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlin_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liborc.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE rounding: no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.orc_f16_to_f64.restype = ctypes.c_double
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f32_to_f16_rn.restype = ctypes.c_uint16
        lib.orc_f32_to_f16_rn.argtypes = [ctypes.c_float]
        lib.orc_e4m3_to_f64.restype = ctypes.c_double
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_f32_to_e4m3_rn_sat.restype = ctypes.c_uint8
        lib.orc_f32_to_e4m3_rn_sat.argtypes = [ctypes.c_float]
        lib.orc_quantize_w4.restype = ctypes.c_int
        lib.orc_quantize_w4.argtypes = [_p, _i64, _i64, ctypes.c_int, ctypes.c_int, _p, _p, _p]
        lib.orc_dequant_w4.restype = None
        lib.orc_dequant_w4.argtypes = [_p, _p, _p, _i64, _i64, ctypes.c_int, _p]
        lib.orc_pack_canonical.restype = None
        lib.orc_pack_canonical.argtypes = [_p, _p, _i64, _i64, ctypes.c_int, _p, _p]
        lib.orc_quant_mxfp8_rows.restype = None
        lib.orc_quant_mxfp8_rows.argtypes = [_p, _i64, _i64, _p, _p]
        lib.orc_w8a8_mx_at.restype = None
        lib.orc_w8a8_mx_at.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p]
        lib.orc_pack_tile.restype = None
        lib.orc_pack_tile.argtypes = [_p, _p, _p, _i64, _i64, _i64, _p, _p, _p]
        lib.orc_quant_fp8_rows.restype = None
        lib.orc_quant_fp8_rows.argtypes = [_p, _i64, _i64, _p, _p]
        lib.orc_quant_fp8_tensor.restype = None
        lib.orc_quant_fp8_tensor.argtypes = [_p, _i64, _i64, _p, _p]
        lib.orc_quant_fp8_act_blocks.restype = None
        lib.orc_quant_fp8_act_blocks.argtypes = [_p, _i64, _i64, _p, _p]
        lib.orc_quant_fp8_weight_blocks.restype = None
        lib.orc_quant_fp8_weight_blocks.argtypes = [_p, _i64, _i64, _p, _p]
        lib.orc_w8a8_blocks_at.restype = None
        lib.orc_w8a8_blocks_at.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p]
        lib.orc_gemm_nt_f64.restype = None
        lib.orc_gemm_nt_f64.argtypes = [_p, _p, _i64, _i64, _i64, _p]
        lib.orc_w4a16_at.restype = None
        lib.orc_w4a16_at.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, ctypes.c_int,
                                     _p, _p, _i64, _p]
        lib.orc_w4a8_at.restype = None
        lib.orc_w4a8_at.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _i64, _p]
        lib.orc_w8a8_at.restype = None
        lib.orc_w8a8_at.argtypes = [_p, _p, _p, ctypes.c_float, _i64, _i64, _i64,
                                    _p, _p, _i64, _p]
        lib.orc_e2m1_to_f64.restype = ctypes.c_double
        lib.orc_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_f32_to_e2m1_rn_sat.restype = ctypes.c_uint8
        lib.orc_f32_to_e2m1_rn_sat.argtypes = [ctypes.c_float]
        lib.orc_quant_mxfp4_rows.restype = None
        lib.orc_quant_mxfp4_rows.argtypes = [_p, _i64, _i64, _p, _p]
        lib.orc_w4a4_mx_at.restype = None
        lib.orc_w4a4_mx_at.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p]
        lib.orc_nvfp4_global_scale.restype = ctypes.c_float
        lib.orc_nvfp4_global_scale.argtypes = [_p, _i64]
        lib.orc_quant_nvfp4_rows.restype = None
        lib.orc_quant_nvfp4_rows.argtypes = [_p, _i64, _i64, ctypes.c_float, _p, _p]
        lib.orc_w4a4_nv_at.restype = None
        lib.orc_w4a4_nv_at.argtypes = [_p, _p, ctypes.c_float, _p, _p, ctypes.c_float, _i64, _i64, _i64,
                                       _p, _p, _i64, _p]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_set_num_threads.restype = None
        lib.orc_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (n >= 1)."""
    _load().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- formats

def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values (bf16 is the top half of binary32)."""
    return (np.ascontiguousarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f16_to_f64(h: int) -> float:
    return float(_load().orc_f16_to_f64(int(h)))


def f32_to_f16_rn(x: float) -> int:
    return int(_load().orc_f32_to_f16_rn(float(x)))


def e4m3_to_f64(c: int) -> float:
    """[LP] S7: E4M3 (OCP fn variant) decode."""
    return float(_load().orc_e4m3_to_f64(int(c)))


def f32_to_e4m3(x: float) -> int:
    """[LP] S7/S8: round-to-nearest-even encode with saturation to +-448."""
    return int(_load().orc_f32_to_e4m3_rn_sat(float(x)))


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 E4M3 codes (NaN for the two NaN codes)."""
    return np.array([e4m3_to_f64(c) for c in range(256)], dtype=np.float64)


def f16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    uniq, inv = np.unique(flat, return_inverse=True)
    vals = np.array([lib.orc_f16_to_f64(int(u)) for u in uniq], dtype=np.float64)
    return vals[inv].reshape(np.shape(h))


# ---------------------------------------------------------------- INT4 W4A16

class W4Quant:
    """Result of the per-group INT4 quantiser: one code per weight, unpacked."""

    def __init__(self, q, s, z, G, symmetric, overflow):
        self.q = q            # [N, K] uint8, stored code 0..15
        self.s = s            # [N, K/G] uint16, binary16 bits
        self.z = z            # [N, K/G] uint8, stored zero nibble
        self.G = G
        self.symmetric = symmetric
        self.overflow = overflow


def quantize_w4(W_bf16: np.ndarray, G: int = 128, symmetric: bool = False) -> W4Quant:
    """[LP] S2-S4: q = clamp(round(x/s)+z, 0, 15) per group of G weights along K."""
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    N, K = W.shape
    assert K % G == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty((N, K // G), np.uint16)
    z = np.empty((N, K // G), np.uint8)
    ov = _load().orc_quantize_w4(_ptr(W), N, K, G, int(bool(symmetric)), _ptr(q), _ptr(s), _ptr(z))
    return W4Quant(q, s, z, G, bool(symmetric), int(ov))


def dequant_w4(wq: W4Quant) -> np.ndarray:
    """[LP] S2: x_hat = s (q - z), exact in double."""
    N, K = wq.q.shape
    out = np.empty((N, K), np.float64)
    _load().orc_dequant_w4(_ptr(wq.q), _ptr(wq.s), _ptr(wq.z), N, K, wq.G, _ptr(out))
    return out


def pack_canonical(wq: W4Quant):
    """Canonical layout: codes [N][K/2] (low nibble = even k), zeros [N][K/2G]."""
    N, K = wq.q.shape
    ng = K // wq.G
    codes = np.empty((N, K // 2), np.uint8)
    zeros = np.empty(((N * ng + 1) // 2,), np.uint8)
    _load().orc_pack_canonical(_ptr(wq.q), _ptr(wq.z), N, K, wq.G, _ptr(codes), _ptr(zeros))
    return codes, wq.s.copy(), zeros


def pack_tile(wq: W4Quant):
    """Tile layout, format version 2 (128 x 64 tiles, G = 32, 64, 128, or K for one
    group per row): codes, scales, zeros as flat arrays."""
    N, K = wq.q.shape
    G = wq.G
    assert (G in (32, 64, 128) or G == K) and N % 128 == 0 and K % 128 == 0
    codes = np.empty((N * K // 2,), np.uint8)
    scales = np.empty((N * K // G,), np.uint16)
    zeros = np.empty((N * K // G // 2,), np.uint8)
    _load().orc_pack_tile(_ptr(wq.q), _ptr(wq.s), _ptr(wq.z), N, K, G,
                          _ptr(codes), _ptr(scales), _ptr(zeros))
    return codes, scales, zeros


def w4a16_full(X_bf16: np.ndarray, wq: W4Quant) -> np.ndarray:
    """Y = X . deq(W)^T in double: dequantise, then a plain fp64 GEMM."""
    X = bf16_bits_to_f32(X_bf16).astype(np.float64)
    Wd = dequant_w4(wq)
    return gemm_nt_f64(X, Wd)


def w4a16_at(X_bf16: np.ndarray, wq: W4Quant, ms: np.ndarray, ns: np.ndarray) -> np.ndarray:
    """Y[m_i, n_i] for sampled pairs, each an fp64 dot product over K."""
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    M, K = X.shape
    N = wq.q.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_w4a16_at(_ptr(X), _ptr(wq.q), _ptr(wq.s), _ptr(wq.z), M, N, K, wq.G,
                         _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out


# ---------------------------------------------------------------- FP8 W8A8

def quant_fp8_rows(X_bf16: np.ndarray):
    """[LP] S4 per-token + S8 current scaling: s_x[m] = amax_m / 448, Xq = E4M3(X / s_x)."""
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    M, K = X.shape
    Xq = np.empty((M, K), np.uint8)
    sx = np.empty((M,), np.float32)
    _load().orc_quant_fp8_rows(_ptr(X), M, K, _ptr(Xq), _ptr(sx))
    return Xq, sx


def quant_fp8_tensor(W_bf16: np.ndarray):
    """[LP] S4 per-tensor + S8: s_w = amax(W) / 448, Wq = E4M3(W / s_w)."""
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    N, K = W.shape
    Wq = np.empty((N, K), np.uint8)
    sw = np.empty((1,), np.float32)
    _load().orc_quant_fp8_tensor(_ptr(W), N, K, _ptr(Wq), _ptr(sw))
    return Wq, float(sw[0])


def e4m3_decode_array(c: np.ndarray) -> np.ndarray:
    return e4m3_table()[np.asarray(c, dtype=np.uint8)]


def w8a8_full(Xq, sx, Wq, sw) -> np.ndarray:
    """Y = diag(s_x) (dec(Xq) . dec(Wq)^T) s_w in double."""
    tab = e4m3_table()
    A = tab[Xq]
    B = tab[Wq]
    Y = gemm_nt_f64(np.ascontiguousarray(A), np.ascontiguousarray(B))
    return Y * np.asarray(sx, np.float64)[:, None] * float(sw)


def w8a8_at(Xq, sx, Wq, sw, ms, ns) -> np.ndarray:
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    M, K = Xq.shape
    N = Wq.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_w8a8_at(_ptr(Xq), _ptr(sx), _ptr(Wq), float(sw), M, N, K,
                        _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out


# ---------------------------------------------------------------- W4A8

def w4a8_full(Xq, sx, wq: W4Quant) -> np.ndarray:
    """[LP] S1 W4A8: Y = (diag(sx) dec(Xq)) . deq(W)^T in double, deq(W) = s (q - z)
    of the INT4 quantiser and Xq / sx of the per-token E4M3 quantiser."""
    A = e4m3_table()[np.asarray(Xq, np.uint8)] * np.asarray(sx, np.float64)[:, None]
    return gemm_nt_f64(np.ascontiguousarray(A), dequant_w4(wq))


def w4a8_at(Xq, sx, wq: W4Quant, ms, ns) -> np.ndarray:
    """Y[m_i, n_i] of w4a8_full for sampled pairs, each a plain loop over K in C."""
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    M, K = Xq.shape
    N = wq.q.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_w4a8_at(_ptr(Xq), _ptr(sx), _ptr(wq.q), _ptr(wq.s), _ptr(wq.z), M, N, K, wq.G,
                        _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out


# ---------------------------------------------------------------- GEMM

def gemm_nt_f64(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """[LP] S22: Y = A . B^T accumulated in double (plain loops in C)."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    Y = np.empty((M, N), np.float64)
    _load().orc_gemm_nt_f64(_ptr(A), _ptr(B), M, N, K, _ptr(Y))
    return Y


# ---------------------------------------------------------------- bytes and roofline

def w4_bits_per_weight(N: int, K: int, G: int = 128, with_zeros: bool = False) -> float:
    """[LP] S5: effective bits from the packed buffer sizes (codes + scales [+ zeros])."""
    codes = N * K // 2
    scales = N * (K // G) * 2
    zeros = (N * (K // G) + 1) // 2
    total = codes + scales + (zeros if with_zeros else 0)
    return 8.0 * total / (N * K)


def roofline_transition_batch(ridge_flop_per_byte: float, bytes_per_weight: float) -> float:
    """[TP] arithmetic intensity of a decode GEMM, AI(B) = 2B / bytes_per_weight;
    the compute-bound transition is the batch where AI reaches the ridge."""
    return ridge_flop_per_byte * bytes_per_weight / 2.0


# ---------------------------------------------------------------- FP8 block scaling

def quant_fp8_act_blocks(X_bf16: np.ndarray):
    """[LP] S8 block scaling, 1 x 128 activation blocks: Xq [M][K] E4M3 and
    sx [K/128][M] (block-major), each block's scale amax / 448."""
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    M, K = X.shape
    assert K % 128 == 0
    Xq = np.empty((M, K), np.uint8)
    sx = np.empty((K // 128, M), np.float32)
    _load().orc_quant_fp8_act_blocks(_ptr(X), M, K, _ptr(Xq), _ptr(sx))
    return Xq, sx


def quant_fp8_weight_blocks(W_bf16: np.ndarray):
    """[LP] S8 block scaling, 128 x 128 weight blocks: Wq [N][K] E4M3 and
    sw [N/128][K/128]."""
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    N, K = W.shape
    assert N % 128 == 0 and K % 128 == 0
    Wq = np.empty((N, K), np.uint8)
    sw = np.empty((N // 128, K // 128), np.float32)
    _load().orc_quant_fp8_weight_blocks(_ptr(W), N, K, _ptr(Wq), _ptr(sw))
    return Wq, sw


def w8a8_blocks_full(Xq, sx, Wq, sw) -> np.ndarray:
    """Y = sum over K blocks b of diag(sx[b]) (dec(Xq_b) . dec(Wq_b)^T) sw[:, b] in double."""
    tab = e4m3_table()
    A = tab[Xq]
    B = tab[Wq]
    M, K = A.shape
    N = B.shape[0]
    Y = np.zeros((M, N), np.float64)
    for b in range(K // 128):
        part = gemm_nt_f64(np.ascontiguousarray(A[:, b * 128:(b + 1) * 128]),
                           np.ascontiguousarray(B[:, b * 128:(b + 1) * 128]))
        Y += part * np.asarray(sx[b], np.float64)[:, None] * np.repeat(np.asarray(sw[:, b], np.float64), 128)[None, :]
    return Y


def w8a8_blocks_at(Xq, sx, Wq, sw, ms, ns) -> np.ndarray:
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    M, K = Xq.shape
    N = Wq.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_w8a8_blocks_at(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), M, N, K, _ptr(ms), _ptr(ns), ms.size,
                               _ptr(out))
    return out


ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU = 0, 1, 2, 3


def epilogue(Y: np.ndarray, bias_bf16, act: int) -> np.ndarray:
    """[LP] S23/S24 fused epilogue, in double: act(Y[m][n] + bias[n]).

    bias_bf16: BF16 bit patterns [N] or None.  act: ReLU max(v, 0); SiLU
    v * sigmoid(v) = v / (1 + e^-v); GELU v * Phi(v), Phi the standard normal
    distribution function, Phi(v) = (1 + erf(v / sqrt 2)) / 2.
    """
    import math

    V = np.array(Y, dtype=np.float64, copy=True)
    if bias_bf16 is not None:
        V = V + bf16_bits_to_f32(np.asarray(bias_bf16, np.uint16)).astype(np.float64)[None, :]
    if act == ACT_RELU:
        return np.maximum(V, 0.0)
    if act == ACT_SILU:
        return V / (1.0 + np.exp(-V))
    if act == ACT_GELU:
        phi = np.vectorize(lambda v: 0.5 * (1.0 + math.erf(v / math.sqrt(2.0))))(V) if V.size else V
        return V * phi
    assert act == ACT_NONE
    return V


def quant_mxfp8_rows(X_bf16: np.ndarray):
    """MXFP8 (OCP MX v1.0, named in [LP] S10): per row, blocks of 32 elements share a
    power-of-two scale 2^e (E8M0 byte e + 127, e = floor(log2 amax) - 8, clamped to
    [-127, 127]); codes E4M3(v / 2^e), RNE, saturating.  Returns codes [R][K] uint8 and
    scales [R][K/32] uint8."""
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    R, K = X.shape
    assert K % 32 == 0
    codes = np.empty((R, K), np.uint8)
    scales = np.empty((R, K // 32), np.uint8)
    _load().orc_quant_mxfp8_rows(_ptr(X), R, K, _ptr(codes), _ptr(scales))
    return codes, scales


def mx_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantised MX values in double: e4m3(code) * 2^(scale - 127) per 32-block."""
    tab = e4m3_table()
    return tab[codes] * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)


def mx_scales_atoms(scales: np.ndarray) -> np.ndarray:
    """The MX scales [R][K/32] in the "scale atom" layout the library's MXFP8 calls
    take, written from its description: atoms of 512 bytes, atom (R0, c) at
    ((R0 * (K/128)) + c) * 512 for rows 128 R0 .. +127 and columns 128 c .. +127;
    row r (mod 128) keeps the scales of its 32-column blocks kk = 0..3 at
    16 (r % 32) + 4 (r / 32) + kk; rows past R are 0.  Flat uint8 array."""
    sc = np.asarray(scales, dtype=np.uint8)
    R, nb = sc.shape
    assert nb % 4 == 0
    nc = nb // 4
    nr = (R + 127) // 128
    out = np.zeros(nr * nc * 512, np.uint8)
    for r in range(R):
        r0, rr = divmod(r, 128)
        for c in range(nc):
            base = (r0 * nc + c) * 512 + 16 * (rr % 32) + 4 * (rr // 32)
            out[base:base + 4] = sc[r, 4 * c:4 * c + 4]
    return out


def w8a8_mx_full(Xq, xs, Wq, ws) -> np.ndarray:
    """Y = dequant(Xq, xs) . dequant(Wq, ws)^T in double (dense product of the MX-dequantised operands)."""
    return gemm_nt_f64(np.ascontiguousarray(mx_dequant(Xq, xs)), np.ascontiguousarray(mx_dequant(Wq, ws)))


def w8a8_mx_at(Xq, xs, Wq, ws, ms, ns) -> np.ndarray:
    """Y[m_i, n_i] = sum over 32-blocks of both block scales times the block's E4M3 dot product, in double."""
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    xs = np.ascontiguousarray(xs, dtype=np.uint8)
    ws = np.ascontiguousarray(ws, dtype=np.uint8)
    M, K = Xq.shape
    N = Wq.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_w8a8_mx_at(_ptr(Xq), _ptr(xs), _ptr(Wq), _ptr(ws), M, N, K, _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out


# ---- FP4 ([LP] S10): E2M1 elements, MXFP4 and NVFP4 block formats

def e2m1_to_f64(c: int) -> float:
    return _load().orc_e2m1_to_f64(c)


def f32_to_e2m1(x: float) -> int:
    """binary32 -> E2M1 code: nearest magnitude, ties to the even code, saturating at 6, sign kept."""
    return _load().orc_f32_to_e2m1_rn_sat(x)


def e2m1_table() -> np.ndarray:
    """The 16 E2M1 codes' values (bit 3 the sign)."""
    return np.array([e2m1_to_f64(c) for c in range(16)], np.float64)


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte along a row: column 2i in the low nibble, 2i + 1 in the high one."""
    c = np.asarray(codes, np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out


def quant_mxfp4_rows(X_bf16: np.ndarray):
    """MXFP4 (OCP MX v1.0, named in [LP] S10): per row, blocks of 32 elements share a
    power-of-two scale 2^e (E8M0 byte e + 127, e = floor(log2 amax) - 2, clamped to
    [-127, 127]); codes E2M1(v / 2^e), nearest, ties to even, saturating.  Returns codes
    [R][K] (one per byte) and scales [R][K/32] uint8."""
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    R, K = X.shape
    assert K % 32 == 0
    codes = np.empty((R, K), np.uint8)
    scales = np.empty((R, K // 32), np.uint8)
    _load().orc_quant_mxfp4_rows(_ptr(X), R, K, _ptr(codes), _ptr(scales))
    return codes, scales


def mxfp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """e2m1(code) * 2^(scale - 127) per 32-block, in double."""
    return e2m1_table()[codes] * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)


def w4a4_mx_full(Xq, xs, Wq, ws) -> np.ndarray:
    """Y = mxfp4_dequant(Xq, xs) . mxfp4_dequant(Wq, ws)^T in double."""
    return gemm_nt_f64(np.ascontiguousarray(mxfp4_dequant(Xq, xs)), np.ascontiguousarray(mxfp4_dequant(Wq, ws)))


def w4a4_mx_at(Xq, xs, Wq, ws, ms, ns) -> np.ndarray:
    """Y[m_i, n_i] = sum over 32-blocks of both block scales times the block's E2M1 dot product, in double."""
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    xs = np.ascontiguousarray(xs, dtype=np.uint8)
    ws = np.ascontiguousarray(ws, dtype=np.uint8)
    M, K = Xq.shape
    N = Wq.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_w4a4_mx_at(_ptr(Xq), _ptr(xs), _ptr(Wq), _ptr(ws), M, N, K, _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out


def nvfp4_global_scale(X_bf16: np.ndarray) -> float:
    """NVFP4 per-tensor scale: amax(|X|) / (6 * 448) as a binary32 division; 1.0 when that is 0."""
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    return float(np.float32(_load().orc_nvfp4_global_scale(_ptr(X), X.size)))


def quant_nvfp4_rows(X_bf16: np.ndarray, sg: float):
    """NVFP4 ([LP] S10 names it; the vendor's two-level recipe): blocks of 16 along a
    row, block scale sb = E4M3(amax_b / (6 sg)), codes E2M1(v / (sb sg)), each step one
    binary32 operation; a block whose scale is 0 stores code 0.  Returns codes [R][K]
    (one per byte) and scales [R][K/16] (E4M3 codes)."""
    X = np.ascontiguousarray(X_bf16, dtype=np.uint16)
    R, K = X.shape
    assert K % 16 == 0
    codes = np.empty((R, K), np.uint8)
    scales = np.empty((R, K // 16), np.uint8)
    _load().orc_quant_nvfp4_rows(_ptr(X), R, K, float(sg), _ptr(codes), _ptr(scales))
    return codes, scales


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray, sg: float) -> np.ndarray:
    """e2m1(code) * e4m3(sb) * sg per 16-block, in double."""
    return e2m1_table()[codes] * np.repeat(e4m3_table()[scales], 16, axis=1) * float(np.float32(sg))


def w4a4_nv_full(Xq, xs, sgx, Wq, ws, sgw) -> np.ndarray:
    """Y = nvfp4_dequant(Xq, xs, sgx) . nvfp4_dequant(Wq, ws, sgw)^T in double."""
    return gemm_nt_f64(np.ascontiguousarray(nvfp4_dequant(Xq, xs, sgx)),
                       np.ascontiguousarray(nvfp4_dequant(Wq, ws, sgw)))


def w4a4_nv_at(Xq, xs, sgx, Wq, ws, sgw, ms, ns) -> np.ndarray:
    """Y[m_i, n_i] = sgx sgw * sum over 16-blocks of both E4M3 block scales times the block's E2M1 dot product."""
    Xq = np.ascontiguousarray(Xq, dtype=np.uint8)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    xs = np.ascontiguousarray(xs, dtype=np.uint8)
    ws = np.ascontiguousarray(ws, dtype=np.uint8)
    M, K = Xq.shape
    N = Wq.shape[0]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.shape, np.float64)
    _load().orc_w4a4_nv_at(_ptr(Xq), _ptr(xs), float(sgx), _ptr(Wq), _ptr(ws), float(sgw), M, N, K,
                           _ptr(ms), _ptr(ns), ms.size, _ptr(out))
    return out
