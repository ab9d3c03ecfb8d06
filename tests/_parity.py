"""Helpers of the GPU parity tests: inputs on the device, oracle references on
full outputs or on whole tiles, and the bound of the problem statement

    |Y - Y_ref| <= 2e-3 * ||X_deq[m, :]||_2 * ||W_deq[n, :]||_2

(times the activation's largest slope, plus the BF16 rounding of the output,
when a fused epilogue is applied).  References come from the oracle applied to
the same quantised operands: for a tile, the oracle's product of the tile's
token rows and weight rows (the same definition, restricted to a sub-block).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from precision_quantized_linear_gb300 import synthetic as syn

TOL = 2e-3
SLOPE = {0: 1.0, 1: 1.0, 2: 1.10, 3: 1.13}  # largest slope of none / ReLU / SiLU / GELU


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f64(Y: torch.Tensor) -> np.ndarray:
    return Y.float().cpu().numpy().astype(np.float64)


def bias_bits(N: int, seed: int) -> np.ndarray:
    """BF16 bias of magnitude comparable with the outputs (bits)."""
    b = np.random.default_rng(seed).normal(0.0, 0.5, N).astype(np.float32)
    return syn.f32_to_bf16_bits(b)


def tile_starts(total: int, tile: int, seed: int):
    """First, last and one random middle tile of `tile` along an axis of `total`."""
    n = (total + tile - 1) // tile
    picks = {0, n - 1}
    if n > 2:
        picks.add(int(np.random.default_rng(seed).integers(1, n - 1)))
    return sorted(t * tile for t in picks)


def blocks(M: int, N: int, tm: int, tn: int, seed: int, extra_m=()):
    """Index sets (ms, ns) of the checked tiles: first / last / middle token tile x
    first / last / middle weight-row tile; extra_m adds the token tiles holding those rows."""
    mstarts = set(tile_starts(M, tm, seed))
    for m in extra_m:
        mstarts.add((int(m) // tm) * tm)
    out = []
    for m0 in sorted(mstarts):
        ms = np.arange(m0, min(M, m0 + tm))
        for n0 in tile_starts(N, tn, seed + 1):
            out.append((ms, np.arange(n0, min(N, n0 + tn))))
    return out


def check(Y, Yref, xn, wn, act=0, where=""):
    bound = SLOPE[act] * TOL * xn[:, None] * wn[None, :]
    if act:
        bound = bound + 2.0 ** -8 * np.abs(Yref)
    err = np.abs(Y - Yref)
    bad = ~(err <= bound)
    assert not bad.any(), (where, np.argwhere(bad)[:4].tolist(), Y[bad][:4], Yref[bad][:4])
    with np.errstate(invalid="ignore", divide="ignore"):
        return float(np.nanmax(np.where(bound > 0, err / (bound / SLOPE[act]), 0.0))) if err.size else 0.0


# ------------------------------------------------------------------ W4A16

def w4_rows(wq: oracle.W4Quant, ns) -> oracle.W4Quant:
    return oracle.W4Quant(wq.q[ns], wq.s[ns], wq.z[ns], wq.G, wq.symmetric, 0)


def w4_ref(X, wq, ms, ns, bias=None, act=0):
    """Oracle Y[ms][:, ns] (after the epilogue) and the bound's row norms."""
    sub = w4_rows(wq, ns)
    Xs = np.ascontiguousarray(X[ms])
    Yr = oracle.w4a16_full(Xs, sub)
    if bias is not None or act:
        Yr = oracle.epilogue(Yr, None if bias is None else bias[ns], act)
    xn = np.linalg.norm(syn.bf16_bits_to_f32(Xs).astype(np.float64), axis=1)
    wn = np.linalg.norm(oracle.dequant_w4(sub), axis=1)
    return Yr, xn, wn


def check_w4(Y, X, wq, full: bool, tm: int, seed: int, bias=None, act=0, chunk=4096, extra_m=()):
    """Compare the device output Y (host f64 [M][N]) with the oracle: every
    element (in chunks of weight rows) or whole tiles."""
    M, N = Y.shape
    worst = 0.0
    if full:
        for n0 in range(0, N, chunk):
            ns = np.arange(n0, min(N, n0 + chunk))
            ms = np.arange(M)
            Yr, xn, wn = w4_ref(X, wq, ms, ns, bias, act)
            worst = max(worst, check(Y[:, ns], Yr, xn, wn, act, "rows %d.." % n0))
    else:
        for ms, ns in blocks(M, N, tm, 128, seed, extra_m):
            Yr, xn, wn = w4_ref(X, wq, ms, ns, bias, act)
            worst = max(worst, check(Y[np.ix_(ms, ns)], Yr, xn, wn, act, "tile m%d n%d" % (ms[0], ns[0])))
    return worst


# ------------------------------------------------------------------ W8A8

def w8_ref(Xq, sx, Wq, sw, ms, ns, bias=None, act=0):
    tab = oracle.e4m3_table()
    Xs, Ws = np.ascontiguousarray(Xq[ms]), np.ascontiguousarray(Wq[ns])
    sxs = np.ascontiguousarray(sx[ms])
    Yr = oracle.w8a8_full(Xs, sxs, Ws, sw)
    if bias is not None or act:
        Yr = oracle.epilogue(Yr, None if bias is None else bias[ns], act)
    xn = np.linalg.norm(tab[Xs] * sxs.astype(np.float64)[:, None], axis=1)
    wn = np.linalg.norm(tab[Ws] * float(sw), axis=1)
    return Yr, xn, wn


def check_w8(Y, Xq, sx, Wq, sw, full: bool, tm: int, seed: int, bias=None, act=0, chunk=4096, extra_m=()):
    M, N = Y.shape
    worst = 0.0
    if full:
        for n0 in range(0, N, chunk):
            ns = np.arange(n0, min(N, n0 + chunk))
            Yr, xn, wn = w8_ref(Xq, sx, Wq, sw, np.arange(M), ns, bias, act)
            worst = max(worst, check(Y[:, ns], Yr, xn, wn, act, "rows %d.." % n0))
    else:
        for ms, ns in blocks(M, N, tm, 128, seed, extra_m):
            Yr, xn, wn = w8_ref(Xq, sx, Wq, sw, ms, ns, bias, act)
            worst = max(worst, check(Y[np.ix_(ms, ns)], Yr, xn, wn, act, "tile m%d n%d" % (ms[0], ns[0])))
    return worst
