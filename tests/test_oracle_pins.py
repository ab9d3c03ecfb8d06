"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests needs a GPU.  Each pin is independent of the oracle's own
code: closed forms, exhaustive code tables, brute force on tiny inputs,
library routines (numpy / torch casts and matmul) and values printed on the
pages (``tests/golden/page_values.json``).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from precision_quantized_linear_gb300 import synthetic as syn

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))


def _bf16(vals):
    return syn.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


# ------------------------------------------------------------------ formats

def test_f16_encode_matches_numpy_rne():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 1e-3,
        rng.standard_normal(20000).astype(np.float32) * 1e4,
        (rng.random(5000).astype(np.float32) * 6.1e-5),        # subnormal range
        np.float32([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 5.96e-8, 2.98e-8, 2.99e-8]),
    ])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    ours = np.array([oracle.f32_to_f16_rn(v) for v in x], dtype=np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_bits_to_f64(codes)
    ref = codes.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_decode_all_codes_vs_torch():
    tab = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    assert np.array_equal(tab[~np.isnan(tab)], ref[~np.isnan(ref)])
    # the format facts: max 448, smallest subnormal 2^-9, NaN only at S.1111.111
    assert np.nanmax(tab) == 448.0 and tab[0x7E] == 448.0
    assert tab[1] == 2.0 ** -9
    assert set(np.flatnonzero(np.isnan(tab))) == {0x7F, 0xFF}


def test_e4m3_roundtrip_every_code():
    tab = oracle.e4m3_table()
    for c in range(256):
        if np.isnan(tab[c]):
            continue
        assert oracle.f32_to_e4m3(tab[c]) == c, c


def test_e4m3_midpoints_round_to_even_and_saturate():
    tab = oracle.e4m3_table()
    pos = sorted({(tab[c], c) for c in range(0x7F)})
    for (v0, c0), (v1, c1) in zip(pos[:-1], pos[1:]):
        mid = np.float32((v0 + v1) / 2)
        if float(mid) != (v0 + v1) / 2:
            continue
        want = c0 if (c0 & 1) == 0 else c1
        assert oracle.f32_to_e4m3(mid) == want, (v0, v1)
        assert oracle.f32_to_e4m3(-mid) == want | 0x80
    for big in (448.0, 463.9, 464.0, 480.0, 1e4, 3e38):
        assert oracle.f32_to_e4m3(big) == 0x7E
        assert oracle.f32_to_e4m3(-big) == 0xFE


def test_e4m3_encode_is_nearest_code_brute_force():
    tab = oracle.e4m3_table()
    finite_pos = np.array([tab[c] for c in range(0x7F)])
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(3000) * 50, rng.standard_normal(3000) * 0.01]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    for v in x:
        c = oracle.f32_to_e4m3(v)
        d = np.abs(finite_pos - abs(float(v)))
        best = d.min()
        assert abs(tab[c & 0x7F] - abs(float(v))) == best
        if v != 0:
            assert (c >> 7) == (1 if v < 0 else 0)


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(50000) * 60).astype(np.float32)
    x = np.clip(x, -448, 448)
    ours = np.array([oracle.f32_to_e4m3(v) for v in x], dtype=np.uint8)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------ INT4 quantiser

def _group_grid_ok(Wf, wq, G):
    """Round-trip bound |x - x_hat| <= s/2 for every weight whose code is not clamped."""
    deq = oracle.dequant_w4(wq)
    s = oracle.f16_bits_to_f64(wq.s)
    N, K = Wf.shape
    s_full = np.repeat(s, G, axis=1)
    err = np.abs(Wf.astype(np.float64) - deq)
    return err, s_full, deq


def test_asymmetric_all_16_codes_and_exact_grid():
    G = 128
    # one group per row spanning a different range; linspace hits every code
    rows = []
    # the first two ranges are exact multiples of s = range/15 (every code appears);
    # the others leave z to rounding, so one end code may go unused
    for lo, hi in [(-3.0, 4.5), (-0.25, 0.125), (-1.0, 2.0), (-0.003, 0.001), (-50.0, 10.0),
                   (0.5, 3.0), (-4.0, -1.0)]:
        rows.append(np.linspace(lo, hi, G, dtype=np.float32))
    W = _bf16(np.stack(rows))
    Wf = syn.bf16_bits_to_f32(W)
    wq = oracle.quantize_w4(W, G=G, symmetric=False)
    for r in range(len(rows)):
        lo = min(Wf[r].min(), 0.0)
        hi = max(Wf[r].max(), 0.0)
        used = set(wq.q[r].tolist())
        if r < 2:
            assert used == set(range(16))
        elif lo < 0.0 < hi:
            assert len(used) >= 15
        else:
            assert len(used) >= 8
        # dequantised values lie exactly on the grid s (c - z), c in 0..15
        s = oracle.f16_to_f64(int(wq.s[r, 0]))
        z = int(wq.z[r, 0])
        deq = oracle.dequant_w4(wq)[r]
        grid = s * (np.arange(16) - z)
        assert np.all(np.isin(deq, grid))
        # zero is exactly representable: the grid contains 0
        assert 0.0 in grid
    err, s_full, _ = _group_grid_ok(Wf, wq, G)
    assert np.all(err <= s_full / 2 * (1 + 2 ** -20))


def test_asymmetric_round_trip_bound_random_groups():
    G = 128
    rng = np.random.default_rng(3)
    N, K = 16, 1024
    w = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    # groups of very different magnitude catch a wrong group index
    w *= (10.0 ** rng.integers(-2, 3, size=(N, K // G))).repeat(G, axis=1).astype(np.float32)
    W = _bf16(w)
    Wf = syn.bf16_bits_to_f32(W)
    wq = oracle.quantize_w4(W, G=G)
    err, s_full, deq = _group_grid_ok(Wf, wq, G)
    assert np.all(err <= s_full / 2 * (1 + 2 ** -20))
    # the nearest grid point is chosen: no other code is strictly closer
    s = s_full
    zf = np.repeat(wq.z.astype(np.float64), G, axis=1)
    for c in range(16):
        alt = s * (c - zf)
        assert np.all(np.abs(Wf - alt) >= err - s * 2 ** -20)


def test_symmetric_zero_point_and_extremes():
    G = 128
    rng = np.random.default_rng(4)
    W = _bf16(rng.standard_normal((8, 256)).astype(np.float32) * 0.05)
    Wf = syn.bf16_bits_to_f32(W).reshape(8, 2, G)
    wq = oracle.quantize_w4(W, G=G, symmetric=True)
    assert np.all(wq.z == 8)                       # logical zero-point 0, offset-binary storage
    codes = wq.q.reshape(8, 2, G).astype(int) - 8  # signed codes
    amax_pos = np.abs(Wf).argmax(axis=2)
    for n in range(8):
        for g in range(2):
            c = codes[n, g, amax_pos[n, g]]
            v = Wf[n, g, amax_pos[n, g]]
            assert c == (7 if v > 0 else -7)      # max|x| maps to +-qmax
    err, s_full, _ = _group_grid_ok(syn.bf16_bits_to_f32(W), wq, G)
    assert np.all(err <= s_full / 2 * (1 + 2 ** -20))


def test_degenerate_group_zero():
    W = _bf16(np.zeros((2, 128), np.float32))
    for sym in (False, True):
        wq = oracle.quantize_w4(W, G=128, symmetric=sym)
        assert np.all(wq.s == 0x3C00)
        assert np.all(oracle.dequant_w4(wq) == 0.0)


def test_scale_is_fp16_of_range_over_15():
    # one closed-form value: range [-1.5, 6.0] -> s = 7.5/15 = 0.5, z = 3
    v = np.zeros(128, np.float32)
    v[0], v[1] = -1.5, 6.0
    wq = oracle.quantize_w4(_bf16(v[None, :]), G=128)
    assert oracle.f16_to_f64(int(wq.s[0, 0])) == 0.5
    assert wq.z[0, 0] == 3
    assert wq.q[0, 0] == 0 and wq.q[0, 1] == 15 and wq.q[0, 2] == 3


# ------------------------------------------------------------------ packing

def test_canonical_pack_nibble_order():
    rng = np.random.default_rng(1)
    W = syn.make_weight(4, 256, seed=9, outlier_frac=0.0)
    wq = oracle.quantize_w4(W, G=128)
    codes, scales, zeros = oracle.pack_canonical(wq)
    lo = codes & 15
    hi = codes >> 4
    assert np.array_equal(lo, wq.q[:, 0::2])
    assert np.array_equal(hi, wq.q[:, 1::2])
    zflat = wq.z.ravel()
    assert np.array_equal(zeros & 15, zflat[0::2])
    assert np.array_equal(zeros >> 4, zflat[1::2])


def test_tile_pack_is_a_bijection_and_hand_positions():
    N, K = 256, 256
    # distinct code per (n, k) position modulo 16 is not unique; use single-hot probes
    q = np.zeros((N, K), np.uint8)
    s = np.full((N, K // 128), 0x3C00, np.uint16)
    z = np.zeros((N, K // 128), np.uint8)
    wq = oracle.W4Quant(q, s, z, 128, False, 0)
    seen = np.zeros(N * K, bool)
    rng = np.random.default_rng(2)
    for (n, k) in [(0, 0), (0, 1), (0, 2), (0, 7), (0, 8), (0, 16), (0, 25), (0, 32), (0, 63), (0, 64),
                   (1, 0), (127, 255), (128, 0), (255, 255)] + [tuple(x) for x in rng.integers(0, 256, (40, 2))]:
        q[:] = 0
        q[n, k] = 0xF
        codes, _, _ = oracle.pack_tile(wq)
        nz = np.flatnonzero(codes)
        assert nz.size == 1
        byte = nz[0]
        nib = 0 if codes[byte] == 0x0F else 1
        assert codes[byte] in (0x0F, 0xF0)
        pos = byte * 2 + nib
        assert not seen[pos]
        seen[pos] = True
        if (n, k) == (0, 0):
            assert (byte, nib) == (0, 0)
        if (n, k) == (0, 1):            # odd column 1 -> nibble position 4 -> byte 2, low
            assert (byte, nib) == (2, 0)
        if (n, k) == (0, 2):            # column 2 = 2t with t = 1 -> word 1, position 0
            assert (byte, nib) == (4, 0)
        if (n, k) == (0, 7):            # column 7 = 2*3 + 1 -> word 3, position 4 -> byte 14, low
            assert (byte, nib) == (14, 0)
        if (n, k) == (0, 8):            # column 8 = 8b -> word 0, position 1 -> byte 0, high
            assert (byte, nib) == (0, 1)
        if (n, k) == (0, 16):           # column 16 = 16a -> word 0, position 2 -> byte 1, low
            assert (byte, nib) == (1, 0)
        if (n, k) == (0, 25):           # column 25 = 16 + 8 + 1 -> word 0, position 7 -> byte 3, high
            assert (byte, nib) == (3, 1)
        if (n, k) == (0, 32):           # second half of the 64-column tile
            assert (byte, nib) == (2048, 0)
        if (n, k) == (1, 0):            # next row: 16 bytes on
            assert (byte, nib) == (16, 0)
        if (n, k) == (0, 64):           # next k tile of the same row tile
            assert (byte, nib) == (4096, 0)
        if (n, k) == (128, 0):          # next row tile: after K/64 = 4 tiles
            assert (byte, nib) == (4 * 4096, 0)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_tile_pack_roundtrip_full(G):
    N, K = 256, 512
    W = syn.make_weight(N, K, seed=3)
    wq = oracle.quantize_w4(W, G=G)
    codes, scales, zeros = oracle.pack_tile(wq)
    # unpack by the written description and compare with the unpacked codes
    c = codes.reshape(N // 128, K // 64, 2, 128, 4, 4)          # nb, kb, h, r, word t, byte
    nib = np.stack([c & 15, c >> 4], axis=-1).reshape(N // 128, K // 64, 2, 128, 4, 8)  # position p
    # position p = 2a + b + 4e of word t holds column c = 16a + 8b + 2t + e of the half
    cols = np.zeros((N // 128, K // 64, 2, 128, 32), np.uint8)
    for t in range(4):
        for p in range(8):
            a, b, e = (p & 3) >> 1, p & 1, p >> 2
            cols[..., 16 * a + 8 * b + 2 * t + e] = nib[..., t, p]
    un = cols.transpose(0, 3, 1, 2, 4).reshape(N, K)
    assert np.array_equal(un, wq.q)
    ng = K // G
    sc = scales.reshape(N // 128, ng, 128).transpose(0, 2, 1).reshape(N, ng)
    assert np.array_equal(sc, wq.s)
    zz = zeros.reshape(N // 128, ng, 64)
    zz = np.stack([zz & 15, zz >> 4], axis=-1).reshape(N // 128, ng, 128)
    assert np.array_equal(zz.transpose(0, 2, 1).reshape(N, ng), wq.z)


def test_effective_bits_from_buffers():
    gold = GOLDEN["effective_bits_int4_fp16_scale_g128"]
    N, K = 256, 512
    wq = oracle.quantize_w4(syn.make_weight(N, K, seed=1), G=128)
    codes, scales, zeros = oracle.pack_tile(wq)
    bits = 8.0 * (codes.nbytes + scales.nbytes) / (N * K)
    assert bits == gold["value"] == gold["b"] + gold["m"] / gold["G"]
    assert 8.0 * (codes.nbytes + scales.nbytes + zeros.nbytes) / (N * K) == 4.15625
    assert oracle.w4_bits_per_weight(N, K) == 4.125


@pytest.mark.parametrize("G", [32, 64])
def test_effective_bits_other_group_sizes(G):
    # the page's b_eff = b + m / G with its b and m, at the other group sizes
    gold = GOLDEN["effective_bits_int4_fp16_scale_g128"]
    N, K = 128, 512
    codes, scales, zeros = oracle.pack_tile(oracle.quantize_w4(syn.make_weight(N, K, seed=2), G=G))
    assert 8.0 * (codes.nbytes + scales.nbytes) / (N * K) == gold["b"] + gold["m"] / G
    assert 8.0 * zeros.nbytes / (N * K) == 4.0 / G


def test_8b_bytes_thought_experiment():
    gold = GOLDEN["model_8b_weight_gb"]
    p = gold["params"]
    assert p * 2 / 1e9 == gold["bf16"] and p * 1 / 1e9 == gold["int8"] and p * 0.5 / 1e9 == gold["int4"]
    # with FP16 scales per 128 and 4-bit zeros the resident bytes are above the ideal 4 GB
    packed = p * oracle.w4_bits_per_weight(4096, 4096, with_zeros=True) / 8 / 1e9
    assert 4.0 < packed < 4.2


# ------------------------------------------------------------------ FP8 quantisation

def test_fp8_per_token_scale_and_max_code():
    X = syn.make_act(9, 512, seed=4, token_outlier_frac=0.2)
    X[3, :] = 0                                   # all-zero row -> scale 1, codes 0
    Xq, sx = oracle.quant_fp8_rows(X)
    Xf = syn.bf16_bits_to_f32(X)
    tab = oracle.e4m3_table()
    for m in range(9):
        amax = np.abs(Xf[m]).max()
        if amax == 0:
            assert sx[m] == 1.0 and np.all(Xq[m] == 0)
            continue
        assert sx[m] == np.float32(amax) / np.float32(448.0)
        i = np.abs(Xf[m]).argmax()
        assert Xq[m, i] in (0x7E, 0xFE)
        dec = tab[Xq[m]] * sx[m]
        normal = np.abs(tab[Xq[m]]) >= 2.0 ** -6
        rel = np.abs(dec - Xf[m])[normal] / np.abs(Xf[m])[normal]
        assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)


def test_fp8_per_tensor_scale():
    W = syn.make_weight(64, 256, seed=2)
    Wq, sw = oracle.quant_fp8_tensor(W)
    Wf = syn.bf16_bits_to_f32(W)
    assert sw == np.float32(np.abs(Wf).max()) / np.float32(448.0)
    assert np.sum((Wq & 0x7F) == 0x7E) >= 1
    # exact power-of-two case: amax = 448 -> scale 1, codes equal the direct cast
    v = np.zeros((1, 128), np.float32)
    v[0, :] = np.linspace(-448, 448, 128, dtype=np.float32)
    Wq2, sw2 = oracle.quant_fp8_tensor(_bf16(v))
    assert sw2 == 1.0
    ref = torch.from_numpy(syn.bf16_bits_to_f32(_bf16(v))).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(Wq2, ref)


# ------------------------------------------------------------------ GEMM

def test_gemm_identity_pins_layout():
    K = 256
    W = syn.make_weight(384, K, seed=6)
    wq = oracle.quantize_w4(W, G=128)
    X = _bf16(np.eye(K, dtype=np.float32))
    Y = oracle.w4a16_full(X, wq)
    assert np.array_equal(Y, oracle.dequant_w4(wq).T)


def test_gemm_brute_force_tiny():
    M, N, K = 3, 8, 128
    W = syn.make_weight(N, K, seed=8)
    X = syn.make_act(M, K, seed=8)
    wq = oracle.quantize_w4(W, G=128)
    Y = oracle.w4a16_full(X, wq)
    Xf = syn.bf16_bits_to_f32(X).astype(np.float64)
    s = oracle.f16_bits_to_f64(wq.s)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += Xf[m, k] * (s[n, k // 128] * (int(wq.q[n, k]) - int(wq.z[n, k // 128])))
            assert abs(acc - Y[m, n]) <= 1e-12 * (1 + abs(acc))


def test_gemm_matches_library_matmul_and_sampled_path():
    M, N, K = 5, 256, 512
    W = syn.make_weight(N, K, seed=10)
    X = syn.make_act(M, K, seed=10)
    wq = oracle.quantize_w4(W, G=128)
    Y = oracle.w4a16_full(X, wq)
    ref = syn.bf16_bits_to_f32(X).astype(np.float64) @ oracle.dequant_w4(wq).T
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    ms = np.array([0, 4, 2, 1]), np.array([0, 255, 17, 128])
    assert np.allclose(oracle.w4a16_at(X, wq, *ms), Y[ms], rtol=1e-12, atol=1e-12)


def test_w8a8_reference_matches_library_and_sampled_path():
    M, N, K = 6, 128, 384
    X = syn.make_act(M, K, seed=12, token_outlier_frac=0.2)
    W = syn.make_weight(N, K, seed=12)
    Xq, sx = oracle.quant_fp8_rows(X)
    Wq, sw = oracle.quant_fp8_tensor(W)
    Y = oracle.w8a8_full(Xq, sx, Wq, sw)
    A = torch.from_numpy(Xq).view(torch.float8_e4m3fn).to(torch.float64)
    B = torch.from_numpy(Wq).view(torch.float8_e4m3fn).to(torch.float64)
    ref = (A @ B.T).numpy() * sx.astype(np.float64)[:, None] * sw
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-15)
    ms, ns = np.array([0, 5, 3]), np.array([7, 0, 127])
    assert np.allclose(oracle.w8a8_at(Xq, sx, Wq, sw, ms, ns), Y[ms, ns], rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------ roofline arithmetic

def test_roofline_transition_from_page_numbers():
    ridge = GOLDEN["ridge_h100_sxm_flop_per_byte"]["value"]
    t = GOLDEN["w4a16_transition_batch_h100"]
    b = oracle.roofline_transition_batch(ridge, t["bytes_per_weight"])
    assert b == 73.75 and round(b) == t["value"]
    d = GOLDEN["decode_bf16_ai_flop_per_byte"]
    assert 2 * d["batch"] / d["bytes_per_weight"] == d["value"]


# ---------------------------------------------------------------- FP8 block scaling ([LP] S8)

def test_fp8_act_blocks_reduce_to_per_token():
    """Each 1 x 128 block is quantised exactly as the per-token recipe would
    quantise a 128-column row holding just that block."""
    X = syn.make_act(5, 512, seed=21, token_outlier_frac=0.2)
    X[1, 128:256] = 0                       # an all-zero block: scale 1, codes 0
    Xq, sx = oracle.quant_fp8_act_blocks(X)
    assert sx.shape == (4, 5)
    for b in range(4):
        q_ref, s_ref = oracle.quant_fp8_rows(np.ascontiguousarray(X[:, b * 128:(b + 1) * 128]))
        assert np.array_equal(Xq[:, b * 128:(b + 1) * 128], q_ref)
        assert np.array_equal(sx[b], s_ref)
    assert sx[1, 1] == 1.0 and not Xq[1, 128:256].any()


def test_fp8_weight_blocks_reduce_to_per_tensor():
    """Each 128 x 128 block is quantised exactly as the per-tensor recipe would
    quantise that block as a tensor of its own."""
    W = syn.make_weight(256, 384, seed=22)
    W[128:, :128] = 0
    Wq, sw = oracle.quant_fp8_weight_blocks(W)
    assert sw.shape == (2, 3)
    for i in range(2):
        for b in range(3):
            blk = np.ascontiguousarray(W[i * 128:(i + 1) * 128, b * 128:(b + 1) * 128])
            q_ref, s_ref = oracle.quant_fp8_tensor(blk)
            assert np.array_equal(Wq[i * 128:(i + 1) * 128, b * 128:(b + 1) * 128], q_ref)
            assert sw[i, b] == s_ref
    assert sw[1, 0] == 1.0


def test_w8a8_blocks_reduce_to_per_token_per_tensor():
    """With every block scale of a token equal and one weight scale, the
    block-scaled product is the per-token / per-tensor W8A8 product."""
    rng = np.random.default_rng(23)
    M, N, K = 3, 256, 384
    Xq = rng.integers(0, 256, (M, K), dtype=np.uint8)
    Wq = rng.integers(0, 256, (N, K), dtype=np.uint8)
    Xq[(Xq & 0x7F) == 0x7F] = 0             # no NaN codes
    Wq[(Wq & 0x7F) == 0x7F] = 0
    sx_tok = np.array([0.5, 0.125, 2.0], np.float32)
    sx = np.repeat(sx_tok[None, :], K // 128, axis=0)
    sw = np.full((N // 128, K // 128), 0.25, np.float32)
    ref = oracle.w8a8_full(Xq, sx_tok, Wq, 0.25)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    got = oracle.w8a8_blocks_at(Xq, sx, Wq, sw, ms.ravel(), ns.ravel()).reshape(M, N)
    assert np.allclose(got, ref, rtol=1e-12, atol=0)
    full = oracle.w8a8_blocks_full(Xq, sx, Wq, sw)
    assert np.allclose(full, ref, rtol=1e-12, atol=0)


def test_w8a8_blocks_scales_enter_per_block():
    """Different scales per block: doubling one block's scale adds exactly that
    block's partial product once more (checked on a brute-force sum)."""
    rng = np.random.default_rng(24)
    M, N, K = 2, 128, 256
    Xq = rng.integers(0, 0x70, (M, K), dtype=np.uint8)
    Wq = rng.integers(0, 0x70, (N, K), dtype=np.uint8)
    sx = np.array([[1.0, 1.0], [1.0, 1.0]], np.float32)
    sw = np.array([[1.0, 1.0]], np.float32)
    base = oracle.w8a8_blocks_full(Xq, sx, Wq, sw)
    sx2 = sx.copy()
    sx2[1, 0] = 2.0                           # block 1, token 0
    got = oracle.w8a8_blocks_full(Xq, sx2, Wq, sw)
    tab = oracle.e4m3_table()
    part = np.array([[sum(tab[Xq[m, k]] * tab[Wq[n, k]] for k in range(128, 256)) for n in range(N)] for m in range(M)])
    assert np.allclose(got[0] - base[0], part[0], rtol=1e-12)
    assert np.array_equal(got[1], base[1])


def test_block_scaling_confines_an_outlier():
    """The reason for block scaling ([LP] S8): an outlier only coarsens its own
    block.  With one channel x4000, the per-token scale flushes some non-zero
    values of the other blocks to code 0 (below E4M3's smallest subnormal at
    that scale); the 1 x 128 block scales keep every one of them."""
    X = syn.make_act(4, 1024, seed=25)
    X32 = syn.bf16_bits_to_f32(X).astype(np.float64)
    X32[:, 5] *= 4000.0
    X = syn.f32_to_bf16_bits(X32.astype(np.float32))
    nonzero = syn.bf16_bits_to_f32(X)[:, 128:] != 0
    q1, _ = oracle.quant_fp8_rows(X)
    qb, _ = oracle.quant_fp8_act_blocks(X)
    flushed_tok = ((q1[:, 128:] & 0x7F) == 0) & nonzero
    flushed_blk = ((qb[:, 128:] & 0x7F) == 0) & nonzero
    assert flushed_tok.sum() > 0
    assert flushed_blk.sum() == 0


# ---- fused epilogue ([LP] S23 / S24): act(Y + bias[n])

def test_epilogue_activations_at_closed_form_points():
    ln3 = math.log(3.0)  # sigmoid(ln 3) = 3/4 exactly
    z975 = 1.959963984540054  # the standard normal 0.975 quantile: Phi(z) = 0.975
    v = np.array([[ln3, -ln3, z975, -z975, 1.0, 0.0, 40.0, -40.0, 2.5, -2.5]])
    silu = oracle.epilogue(v, None, oracle.ACT_SILU)[0]
    gelu = oracle.epilogue(v, None, oracle.ACT_GELU)[0]
    relu = oracle.epilogue(v, None, oracle.ACT_RELU)[0]
    assert silu[0] == pytest.approx(0.75 * ln3, rel=1e-15) and silu[1] == pytest.approx(-0.25 * ln3, rel=1e-15)
    assert gelu[2] == pytest.approx(0.975 * z975, rel=1e-14) and gelu[3] == pytest.approx(-0.025 * z975, rel=1e-12)
    assert gelu[4] == pytest.approx(0.8413447460685429, rel=1e-15)  # Phi(1) from the normal table
    assert silu[5] == 0.0 and gelu[5] == 0.0 and relu[5] == 0.0
    assert silu[6] == pytest.approx(40.0, rel=1e-15) and abs(silu[7]) < 1e-15
    assert list(relu) == [ln3, 0.0, z975, 0.0, 1.0, 0.0, 40.0, 0.0, 2.5, 0.0]
    np.testing.assert_array_equal(oracle.epilogue(v, None, oracle.ACT_NONE), v)


def test_epilogue_odd_part_identities():
    # x sigmoid(x) - (-x) sigmoid(-x) = x and x Phi(x) - (-x) Phi(-x) = x for every x
    v = np.random.default_rng(3).normal(0.0, 3.0, (4, 64))
    for act in (oracle.ACT_SILU, oracle.ACT_GELU):
        d = oracle.epilogue(v, None, act) - oracle.epilogue(-v, None, act)
        np.testing.assert_allclose(d, v, rtol=0, atol=1e-12)


def test_epilogue_bias_is_per_output_column_and_precedes_the_activation():
    # [X, 1] . [W, b]^T = X W^T + b: the library matmul on augmented operands
    X = syn.make_act(5, 256, seed=21)
    W = syn.make_weight(128, 256, seed=22)
    wq = oracle.quantize_w4(W)
    bias = syn.make_act(1, 128, seed=23)[0]
    Y = oracle.epilogue(oracle.w4a16_full(X, wq), bias, oracle.ACT_NONE)
    xa = np.hstack([syn.bf16_bits_to_f32(X).astype(np.float64), np.ones((5, 1))])
    wa = np.hstack([oracle.dequant_w4(wq), syn.bf16_bits_to_f32(bias).astype(np.float64)[:, None]])
    np.testing.assert_allclose(Y, xa @ wa.T, rtol=1e-12, atol=1e-12)
    two = np.array([0x4000], np.uint16)  # BF16 2.0
    assert oracle.epilogue(np.array([[-1.0]]), two, oracle.ACT_RELU)[0, 0] == 1.0  # relu(-1 + 2), not relu(-1) + 2


# ---- MXFP8 (OCP Microscaling v1.0, named in [LP] S10): 32-element blocks, E8M0 scale

def _bf16_bits(vals):
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_mxfp8_shared_exponent_at_closed_form_points():
    K = 32
    rows = np.zeros((5, K), np.float32)
    rows[0, 0] = 1.0          # floor(log2 1) = 0 -> e = -8, code 119; 1.0 / 2^-8 = 256 = E4M3 0x78
    rows[1, 0] = 480.0        # e = 0, code 127; 480 saturates to 448 (0x7E)
    rows[2, 0] = 300.0        # e = 0; 300 lies between 288 and 320 -> 288 (nearest)
    rows[3, :] = 0.0          # all-zero block: e = -127 (code 0), codes 0
    rows[4, 0] = 2.0 ** -126  # e would be -134: clamped to -127 (code 0); 2^-126 / 2^-127 = 2 exactly
    codes, scales = oracle.quant_mxfp8_rows(_bf16_bits(rows))
    assert list(scales[:, 0]) == [119, 127, 127, 0, 0]
    tab = oracle.e4m3_table()
    assert codes[0, 0] == 0x78 and tab[codes[0, 0]] == 256.0
    assert codes[1, 0] == 0x7E and tab[codes[1, 0]] == 448.0
    assert tab[codes[2, 0]] == 288.0
    assert not codes[3].any()
    assert tab[codes[4, 0]] == 2.0
    deq = oracle.mx_dequant(codes, scales)
    assert deq[0, 0] == 1.0 and deq[1, 0] == 448.0 and deq[4, 0] == 2.0 ** -126


def test_mxfp8_round_trip_error_bound():
    rng = np.random.default_rng(11)
    X = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-20, 20, (16, 1)))).astype(np.float32)
    Xb = _bf16_bits(X)
    v = syn.bf16_bits_to_f32(Xb).astype(np.float64)
    codes, scales = oracle.quant_mxfp8_rows(Xb)
    deq = oracle.mx_dequant(codes, scales)
    step = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)  # X = 2^e of each element
    sat = np.abs(v) >= 448.0 * step
    # E4M3 keeps 3 mantissa bits: half an ulp is 2^-4 relative; below its normal range the step is 2^-9 X
    ok = np.abs(v - deq) <= 2.0 ** -4 * np.abs(v) + 2.0 ** -10 * step
    assert ok[~sat].all()
    assert (np.abs(deq[sat]) == 448.0 * step[sat]).all()   # only the top of each block's range saturates
    assert (np.abs(v[sat]) < 512.0 * step[sat]).all()


def test_mxfp8_product_applies_each_block_scale_to_its_own_block():
    rng = np.random.default_rng(12)
    X = (rng.standard_normal((6, 128)) * np.exp2(rng.integers(-6, 6, (6, 4)).repeat(32, axis=1))).astype(np.float32)
    W = (rng.standard_normal((8, 128)) * np.exp2(rng.integers(-6, 6, (8, 4)).repeat(32, axis=1))).astype(np.float32)
    Xq, xs = oracle.quant_mxfp8_rows(_bf16_bits(X))
    Wq, ws = oracle.quant_mxfp8_rows(_bf16_bits(W))
    ms, ns = np.repeat(np.arange(6), 8), np.tile(np.arange(8), 6)
    got = oracle.w8a8_mx_at(Xq, xs, Wq, ws, ms, ns)
    want = (oracle.mx_dequant(Xq, xs) @ oracle.mx_dequant(Wq, ws).T)[ms, ns]  # dense product of the dequantised operands
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)


def test_mx_scale_atoms_feed_each_row_its_own_scales():
    """The atom layout, read back the way the tensor cores take it: the 512-byte
    atom as 32 rows of four 32-bit words, copied to lane r (of every lane
    quadrant); row m of the operand reads lane m % 32, word m // 32, byte kk."""
    R, K = 200, 256                                          # a partial second row atom, two column atoms
    rng = np.random.default_rng(21)
    scales = rng.integers(1, 255, (R, K // 32)).astype(np.uint8)
    atoms = oracle.mx_scales_atoms(scales)
    assert atoms.size == 2 * 2 * 512
    nc = K // 128
    for m in range(R):
        for c in range(nc):
            atom = atoms[((m // 128) * nc + c) * 512:((m // 128) * nc + c + 1) * 512].reshape(32, 4, 4)
            mm = m % 128
            assert list(atom[mm % 32, mm // 32]) == list(scales[m, 4 * c:4 * c + 4])
    pad = atoms[(1 * nc) * 512:].reshape(nc, 32, 4, 4)        # rows 200..255 of the second row atom are 0
    for c in range(nc):
        for mm in range(R - 128, 128):
            assert not pad[c, mm % 32, mm // 32].any()


def test_mx_full_product_equals_the_per_element_loops():
    rng = np.random.default_rng(22)
    X = (rng.standard_normal((5, 256)) * np.exp2(rng.integers(-5, 5, (5, 8)).repeat(32, axis=1))).astype(np.float32)
    W = (rng.standard_normal((7, 256)) * np.exp2(rng.integers(-5, 5, (7, 8)).repeat(32, axis=1))).astype(np.float32)
    Xq, xs = oracle.quant_mxfp8_rows(_bf16_bits(X))
    Wq, ws = oracle.quant_mxfp8_rows(_bf16_bits(W))
    full = oracle.w8a8_mx_full(Xq, xs, Wq, ws)
    ms, ns = np.repeat(np.arange(5), 7), np.tile(np.arange(7), 5)
    np.testing.assert_allclose(full[ms, ns], oracle.w8a8_mx_at(Xq, xs, Wq, ws, ms, ns), rtol=1e-12, atol=0)


# ---- W4A8 ([LP] S1 precision manifest: INT4 weights, FP8 activations, FP32 accumulate)

def _w4a8_case(M, N, K, seed):
    W = syn.make_weight(N, K, seed=seed)
    X = syn.make_act(M, K, seed=seed + 1, token_outlier_frac=0.2)
    wq = oracle.quantize_w4(W)
    Xq, sx = oracle.quant_fp8_rows(X)
    return wq, Xq, sx


def test_w4a8_full_equals_the_per_element_loops():
    wq, Xq, sx = _w4a8_case(5, 256, 384, 31)
    full = oracle.w4a8_full(Xq, sx, wq)
    ms, ns = np.repeat(np.arange(5), 9), np.tile(np.arange(0, 256, 29), 5)
    np.testing.assert_allclose(full[ms, ns], oracle.w4a8_at(Xq, sx, wq, ms, ns), rtol=1e-12, atol=1e-300)


def test_w4a8_reduces_to_w4a16_on_fp8_exact_activations():
    # activations whose values are E4M3 codes times a unit scale are exact in BF16:
    # the W4A8 product must then be the (pinned) W4A16 product of those values
    rng = np.random.default_rng(32)
    codes = rng.integers(0, 256, (3, 256)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38            # no NaN codes
    vals = oracle.e4m3_table()[codes].astype(np.float32)
    xb = syn.f32_to_bf16_bits(vals)
    assert np.array_equal(syn.bf16_bits_to_f32(xb), vals)
    wq = oracle.quantize_w4(syn.make_weight(128, 256, seed=33))
    sx = np.ones(3, np.float32)
    np.testing.assert_array_equal(oracle.w4a8_full(codes, sx, wq), oracle.w4a16_full(xb, wq))


def test_w4a8_token_scale_enters_its_row_linearly():
    wq, Xq, sx = _w4a8_case(4, 128, 256, 34)
    base = oracle.w4a8_full(Xq, sx, wq)
    sx2 = sx.copy()
    sx2[2] *= 4.0                                    # power of two: exact
    got = oracle.w4a8_full(Xq, sx2, wq)
    np.testing.assert_array_equal(got[2], 4.0 * base[2])
    np.testing.assert_array_equal(np.delete(got, 2, 0), np.delete(base, 2, 0))


def test_w4a8_brute_force_triple_loop():
    wq, Xq, sx = _w4a8_case(2, 128, 128, 35)
    tab = oracle.e4m3_table()
    deq = oracle.dequant_w4(wq)
    want = np.zeros((2, 128))
    for m in range(2):
        for n in range(128):
            acc = 0.0
            for k in range(128):
                acc += float(sx[m]) * tab[Xq[m, k]] * deq[n, k]
            want[m, n] = acc
    np.testing.assert_allclose(oracle.w4a8_full(Xq, sx, wq), want, rtol=1e-12, atol=1e-300)


# ---- per-channel W4 scales ([LP] S4 "per-channel": one scale spanning the row, G = K)

def test_per_channel_equals_per_group_when_every_group_spans_the_row_range():
    # each row repeats one 128-column pattern: every group has the row's min / max,
    # so one group over K and groups of 128 give the same scale, zero-point and codes
    rng = np.random.default_rng(41)
    pat = (rng.standard_normal((128, 128)) * 0.02).astype(np.float32)
    W = syn.f32_to_bf16_bits(np.tile(pat, (1, 8)))          # [128, 1024]
    pc = oracle.quantize_w4(W, G=1024)
    pg = oracle.quantize_w4(W, G=128)
    assert pc.s.shape == (128, 1) and pg.s.shape == (128, 8)
    assert np.array_equal(pc.q, pg.q)
    assert (pg.s == pc.s).all() and (pg.z == pc.z).all()


def test_per_channel_scale_closed_form():
    W = syn.make_weight(256, 2048, seed=42)
    wq = oracle.quantize_w4(W, G=2048)
    w = syn.bf16_bits_to_f32(W)
    lo = np.minimum(w.min(axis=1), 0.0).astype(np.float32)
    hi = np.maximum(w.max(axis=1), 0.0).astype(np.float32)
    s16 = ((hi - lo) / np.float32(15.0)).astype(np.float32).astype(np.float16)   # binary32 divide, RNE to binary16
    assert np.array_equal(wq.s[:, 0], s16.view(np.uint16))
    deq = oracle.dequant_w4(wq)
    sc = s16.astype(np.float64)[:, None]
    assert (np.abs(deq - w) <= sc / 2 * (1 + 2.0 ** -20)).all()   # round-trip bound inside the range
    c, s, z = oracle.pack_tile(wq)
    assert np.array_equal(s.reshape(2, 128), wq.s[:, 0].reshape(2, 128))       # one scale per row, tile order


# ---- FP4 ([LP] S10): E2M1 = 1 sign, 2 exponent and 1 mantissa bit; MXFP4 and NVFP4 blocks

def test_e2m1_values_are_the_ocp_table():
    # the OCP MX specification's E2M1 table: largest normal 6, smallest normal 1, one subnormal 0.5
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    tab = oracle.e2m1_table()
    assert list(tab[:8]) == want
    assert list(-tab[8:]) == want and np.signbit(tab[8:]).all()
    # every E2M1 value is exact in E4M3 (2 exponent bits and 1 mantissa bit fit in 4 and 3)
    e4 = oracle.e4m3_table()
    for v in want:
        assert e4[oracle.f32_to_e4m3(v)] == v


def test_e2m1_rounding_nearest_ties_even_saturating():
    tab = oracle.e2m1_table()
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}   # midpoints: even code
    for x, v in ties.items():
        assert tab[oracle.f32_to_e2m1(x)] == v and tab[oracle.f32_to_e2m1(-x)] == -v
    for x in (6.0, 6.5, 7.99, 1e30, float("inf")):
        assert oracle.f32_to_e2m1(x) == 7 and oracle.f32_to_e2m1(-x) == 15
    assert oracle.f32_to_e2m1(-0.1) == 8 and oracle.f32_to_e2m1(0.0) == 0     # the sign survives a zero result
    rng = np.random.default_rng(31)
    grid = tab[:8]
    for x in rng.uniform(-7.0, 7.0, 5000).astype(np.float32):            # brute force: a nearest value
        q = tab[oracle.f32_to_e2m1(float(x))]
        assert abs(float(x) - q) <= np.abs(abs(float(x)) - grid).min()
        assert q == 0 or np.sign(q) == np.sign(x)


def test_fp4_packing_puts_the_even_column_in_the_low_nibble():
    codes = np.array([[1, 2, 15, 8, 0, 7]], np.uint8)
    packed = oracle.pack_fp4(codes)
    assert list(packed[0]) == [0x21, 0x8F, 0x70]
    assert np.array_equal(oracle.unpack_fp4(packed), codes)


def test_mxfp4_shared_exponent_at_closed_form_points():
    rows = np.zeros((5, 32), np.float32)
    rows[0, 0] = 1.0                      # floor(log2 1) = 0 -> e = -2 (byte 125); 1 / 2^-2 = 4: code 6
    rows[1, :2] = [7.0, 5.0]              # e = 0 (byte 127); 7 saturates to 6 (code 7); 5 is a tie: 4 (code 6)
    rows[3, 0] = 2.0 ** -126              # e would be -128: clamped to -127 (byte 0); 2^-126 / 2^-127 = 2: code 4
    rows[4, :2] = [-3.0, 0.75]            # e = -1 (byte 126); -3 / 0.5 = -6 (code 15); 0.75 / 0.5 = 1.5 (code 3)
    codes, scales = oracle.quant_mxfp4_rows(_bf16_bits(rows))
    assert list(scales[:, 0]) == [125, 127, 0, 0, 126]
    assert codes[0, 0] == 6 and list(codes[1, :2]) == [7, 6] and not codes[2].any()
    assert codes[3, 0] == 4 and list(codes[4, :2]) == [15, 3]
    deq = oracle.mxfp4_dequant(codes, scales)
    assert deq[0, 0] == 1.0 and deq[1, 0] == 6.0 and deq[1, 1] == 4.0 and deq[3, 0] == 2.0 ** -126
    assert deq[4, 0] == -3.0 and deq[4, 1] == 0.75


def test_mxfp4_round_trip_error_bound():
    rng = np.random.default_rng(32)
    X = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-20, 20, (16, 1)))).astype(np.float32)
    Xb = _bf16_bits(X)
    v = syn.bf16_bits_to_f32(Xb).astype(np.float64)
    codes, scales = oracle.quant_mxfp4_rows(Xb)
    deq = oracle.mxfp4_dequant(codes, scales)
    step = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)   # X = 2^e of each element
    sat = np.abs(v) > 6.0 * step
    # one mantissa bit: half a spacing is at most a quarter of the value; below 1 X the spacing is X / 2
    ok = np.abs(v - deq) <= 0.25 * np.abs(v) + 0.25 * step
    assert ok[~sat].all()
    assert (np.abs(deq[sat]) == 6.0 * step[sat]).all() and (np.abs(v[sat]) < 8.0 * step[sat]).all()
    amax = np.abs(v).reshape(16, 8, 32).max(axis=2)                      # every block's amax lands in [4, 8) X
    sc = np.ldexp(1.0, scales.astype(np.int64) - 127)
    assert ((amax >= 4.0 * sc) & (amax < 8.0 * sc)).all()


def test_mxfp4_product_applies_each_block_scale_to_its_own_block():
    rng = np.random.default_rng(33)
    X = (rng.standard_normal((6, 128)) * np.exp2(rng.integers(-6, 6, (6, 4)).repeat(32, axis=1))).astype(np.float32)
    W = (rng.standard_normal((8, 128)) * np.exp2(rng.integers(-6, 6, (8, 4)).repeat(32, axis=1))).astype(np.float32)
    Xq, xs = oracle.quant_mxfp4_rows(_bf16_bits(X))
    Wq, ws = oracle.quant_mxfp4_rows(_bf16_bits(W))
    ms, ns = np.repeat(np.arange(6), 8), np.tile(np.arange(8), 6)
    got = oracle.w4a4_mx_at(Xq, xs, Wq, ws, ms, ns)
    want = (oracle.mxfp4_dequant(Xq, xs) @ oracle.mxfp4_dequant(Wq, ws).T)[ms, ns]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)
    np.testing.assert_allclose(oracle.w4a4_mx_full(Xq, xs, Wq, ws)[ms, ns], got, rtol=1e-12, atol=0)


def test_nvfp4_global_scale():
    X = np.zeros((2, 16), np.float32)
    assert oracle.nvfp4_global_scale(_bf16_bits(X)) == 1.0                 # all zero: 1
    X[1, 3] = -2688.0
    assert oracle.nvfp4_global_scale(_bf16_bits(X)) == 1.0                 # 2688 = 6 * 448
    X[1, 3] = 1.0
    assert oracle.nvfp4_global_scale(_bf16_bits(X)) == float(np.float32(1.0) / np.float32(2688.0))


def test_nvfp4_two_level_scales_at_closed_form_points():
    X = np.zeros((2, 32), np.float32)
    X[0, 0] = 2688.0                      # sg = 1; block 0: sb = 2688 / 6 = 448 (0x7E), 2688 / 448 = 6 (code 7)
    X[0, 16:20] = [6.0, 3.0, -1.5, 0.25]  # block 1: sb = 1 (0x38); codes 7, 5, 11 (-1.5), 0 (0.25: tie -> 0)
    X[1, 0:2] = [1.25, 0.5]               # sb = E4M3(1.25 / 6 = 0.2083) = 0.203125 (0x25): 1.25 / sb = 6.15 -> 6
                                          # (code 7, saturated); 0.5 / sb = 2.46 -> 2 (code 4); block 1 all zero
    Xb = _bf16_bits(X)
    sg = oracle.nvfp4_global_scale(Xb)
    assert sg == 1.0
    codes, scales = oracle.quant_nvfp4_rows(Xb, sg)
    assert scales.tolist() == [[0x7E, 0x38], [0x25, 0x00]]
    assert codes[0, 0] == 7 and list(codes[0, 16:20]) == [7, 5, 11, 0]
    assert list(codes[1, :2]) == [7, 4] and not codes[1, 16:].any()
    deq = oracle.nvfp4_dequant(codes, scales, sg)
    assert deq[0, 0] == 2688.0 and deq[1, 0] == 6 * 0.203125 and deq[1, 1] == 2 * 0.203125
    # a tensor amax of 1: sg = 1/2688 in binary32, the block scale lands on 448 and the element on 6
    Y = np.zeros((1, 16), np.float32)
    Y[0, 0] = 1.0
    sgy = oracle.nvfp4_global_scale(_bf16_bits(Y))
    c, s = oracle.quant_nvfp4_rows(_bf16_bits(Y), sgy)
    assert s[0, 0] == 0x7E and c[0, 0] == 7


def test_nvfp4_round_trip_error_bound():
    rng = np.random.default_rng(34)
    X = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-8, 8, (16, 16)).repeat(16, axis=1))).astype(np.float32)
    Xb = _bf16_bits(X)
    v = syn.bf16_bits_to_f32(Xb).astype(np.float64)
    sg = oracle.nvfp4_global_scale(Xb)
    assert sg == float(np.float32(np.float32(np.abs(v).max()) / np.float32(2688.0)))
    codes, scales = oracle.quant_nvfp4_rows(Xb, sg)
    deq = oracle.nvfp4_dequant(codes, scales, sg)
    e4 = oracle.e4m3_table()
    sb = e4[scales]
    amax = np.abs(v).reshape(16, 16, 16).max(axis=2)
    t = amax / (6.0 * sg)
    normal = t >= 2.0 ** -6                  # E4M3 normal range: the block scale is within 2^-4 of amax / (6 sg)
    assert (np.abs(sb - t)[normal] <= 2.0 ** -4 * t[normal] * (1 + 1e-6)).all()
    step = np.repeat(sb * sg, 16, axis=1)     # the element's unit
    sat = np.abs(v) > 6.0 * step
    ok = np.abs(v - deq) <= 0.25 * np.abs(v) + 0.25 * step + 1e-6 * np.abs(v)   # 1e-6: binary32 v / (sb sg)
    assert ok[~sat].all()
    assert (np.abs(deq[sat]) == 6.0 * step[sat]).all()


def test_nvfp4_product_equals_the_per_block_loops():
    rng = np.random.default_rng(35)
    X = (rng.standard_normal((5, 128)) * np.exp2(rng.integers(-5, 5, (5, 8)).repeat(16, axis=1))).astype(np.float32)
    W = (rng.standard_normal((7, 128)) * np.exp2(rng.integers(-5, 5, (7, 8)).repeat(16, axis=1))).astype(np.float32)
    sgx, sgw = oracle.nvfp4_global_scale(_bf16_bits(X)), oracle.nvfp4_global_scale(_bf16_bits(W))
    Xq, xs = oracle.quant_nvfp4_rows(_bf16_bits(X), sgx)
    Wq, ws = oracle.quant_nvfp4_rows(_bf16_bits(W), sgw)
    ms, ns = np.repeat(np.arange(5), 7), np.tile(np.arange(7), 5)
    got = oracle.w4a4_nv_at(Xq, xs, sgx, Wq, ws, sgw, ms, ns)
    want = (oracle.nvfp4_dequant(Xq, xs, sgx) @ oracle.nvfp4_dequant(Wq, ws, sgw).T)[ms, ns]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=0)
    np.testing.assert_allclose(oracle.w4a4_nv_full(Xq, xs, sgx, Wq, ws, sgw)[ms, ns], got, rtol=1e-12, atol=0)
