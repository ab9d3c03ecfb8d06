"""The C ABI library loads and exports every symbol the header declares, and
argument validation rejects bad calls before touching the GPU (no compute)."""
import ctypes
import os
import re

import pytest

import precision_quantized_linear_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlin.h")


@pytest.fixture(scope="module")
def lib():
    q.build()
    return q.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_\w+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = _declared()
    for n in ("qlin_pack_w4", "qlin_w4a16_gemm", "qlin_quant_act_fp8", "qlin_w8a8_fp8_gemm", "qlin_quant_w_fp8",
              "qlin_get_device_error", "qlin_workspace_size", "qlin_w4_packed_sizes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(q._SIGS), "binding misses a declared call"


def test_status_strings_and_version(lib):
    assert q.qlin_status_string(0) == "QLIN_OK"
    assert q.qlin_status_string(7) == "QLIN_ERR_TIMEOUT"
    assert q.qlin_status_string(99) == "QLIN_ERR_UNKNOWN"
    assert q.qlin_pack_format_version() == q.PACK_FORMAT_VERSION == 2
    assert q.qlin_last_cuda_error() == 0  # nothing has failed on this thread
    assert q.qlin_cuda_error_name(0) == "cudaSuccess"
    assert q.qlin_cuda_error_name(2) == "cudaErrorMemoryAllocation"


def test_packed_sizes_give_4_125_bits(lib):
    c, s, z = q.qlin_w4_packed_sizes(4096, 14336, 128)
    assert 8 * (c + s) / (4096 * 14336) == 4.125
    assert 8 * (c + s + z) / (4096 * 14336) == 4.15625
    for G, bits in ((64, 4.25), (32, 4.5)):  # b + m / G at the other group sizes
        c, s_, z = q.qlin_w4_packed_sizes(4096, 4096, G)
        assert 8 * (c + s_) / (4096 * 4096) == bits and 8 * z / (4096 * 4096) == 4 / G
    for G in (16, 48, 256):
        with pytest.raises(q.QlinError) as e:
            q.qlin_w4_packed_sizes(4096, 4096, G)
        assert e.value.status == 2


# Validation happens before any CUDA call: these return without a device.
def _w4(lib, X=16, codes=16, s=16, z=16, Y=16, M=1, N=128, K=128, G=128, ws=None, wsb=0, path=0):
    return lib.qlin_w4a16_gemm_ex(X, codes, s, z, Y, M, N, K, G, ws, wsb, path, None)


def test_w4a16_rejects_bad_arguments(lib):
    assert _w4(lib, G=48) == 2
    assert _w4(lib, G=256) == 2
    assert _w4(lib, N=100) == 2
    assert _w4(lib, K=192) == 2
    assert _w4(lib, M=-1) == 2
    assert _w4(lib, M=(1 << 24) + 1) == 2
    assert _w4(lib, path=3) == 1
    assert _w4(lib, X=None) == 1
    assert _w4(lib, Y=None) == 1
    assert _w4(lib, codes=24) == 3
    assert _w4(lib, ws=8) == 3
    assert _w4(lib, M=0, X=None) == 0          # empty call: nothing to do


def test_fp8_and_pack_reject_bad_arguments(lib):
    assert lib.qlin_quant_act_fp8(16, 1, 100, 16, 16, None) == 2
    assert lib.qlin_quant_act_fp8(None, 1, 128, 16, 16, None) == 1
    assert lib.qlin_quant_act_fp8(16, 1, 128, 17, 16, None) == 3
    assert lib.qlin_quant_act_fp8(None, 0, 128, None, None, None) == 0
    assert lib.qlin_w8a8_fp8_gemm_ex(16, 16, 16, 16, 16, 1, 96, 128, None, 0, 0, None) == 2
    assert lib.qlin_w8a8_fp8_gemm_ex(16, 18, 16, 16, 16, 1, 128, 128, None, 0, 0, None) == 3
    assert lib.qlin_pack_w4(16, 128, 128, 128, 2, 16, 16, 16, None) == 1
    assert lib.qlin_pack_w4(16, 128, 128, 48, 0, 16, 16, 16, None) == 2
    assert lib.qlin_quant_w_fp8(16, 128, 128, 16, 16, None, 0, None) == 1


def test_fused_calls_reject_bad_epilogue_arguments(lib):
    """Every *_gemm_fused call checks its activation and bias before anything
    else (no device needed); an empty call launches nothing."""
    calls = {
        "qlin_w4a16_gemm_fused": lambda b, a, M=1: lib.qlin_w4a16_gemm_fused(16, 16, 16, 16, 16, M, 128, 128, 128, b, a,
                                                                             None, 0, 0, None),
        "qlin_w8a8_fp8_gemm_fused": lambda b, a, M=1: lib.qlin_w8a8_fp8_gemm_fused(16, 16, 16, 16, 16, M, 128, 128, b,
                                                                                   a, None, 0, 0, None),
        "qlin_w8a8_fp8_block_gemm_fused": lambda b, a, M=1: lib.qlin_w8a8_fp8_block_gemm_fused(
            16, 16, 16, 16, 16, M, 128, 128, b, a, None, 0, None),
        "qlin_w4a8_gemm_fused": lambda b, a, M=1: lib.qlin_w4a8_gemm_fused(16, 16, 16, 16, 16, 16, M, 128, 128, 128, b,
                                                                           a, None, 0, None),
        "qlin_mxfp8_gemm_fused": lambda b, a, M=1: lib.qlin_mxfp8_gemm_fused(16, 16, 16, 16, 16, M, 128, 128, b, a,
                                                                             None, 0, None),
        "qlin_mxfp4_gemm_fused": lambda b, a, M=1: lib.qlin_mxfp4_gemm_fused(16, 16, 16, 16, 16, M, 128, 256, b, a,
                                                                             None, 0, None),
        "qlin_nvfp4_gemm_fused": lambda b, a, M=1: lib.qlin_nvfp4_gemm_fused(16, 16, 16, 16, 16, 16, 16, M, 128, 256,
                                                                             b, a, None, 0, None),
    }
    for name, call in calls.items():
        assert call(None, q.ACT_GELU + 1) == 1, name    # unknown activation
        assert call(None, -1) == 1, name
        assert call(24, q.ACT_SILU) == 3, name          # bias not 16-byte aligned
        assert call(16, q.ACT_RELU, M=0) == 0, name     # empty call


# The dispatch query plans without a device when given an SM count.
def test_plan_query_without_device(lib):
    p = q.qlin_plan_info(q.OP_W4A16_GEMM, 2048, 28672, 4096, 128, q.PATH_TC, 152)
    assert p["kernel"] == q.KERNEL_W4A16_TC and p["tokens_per_tile"] == 256 and p["a_in_tmem"] == 0
    assert p["token_blocks"] == 8 and p["splits"] == 1 and p["ws_bytes"] == 0
    p = q.qlin_plan_info(q.OP_W4A16_GEMM, 128, 14336, 4096, 128, q.PATH_TC, 152)
    assert p["tokens_per_tile"] == 128 and p["a_in_tmem"] == 1
    p = q.qlin_plan_info(q.OP_W8A8_GEMM, 8192, 4096, 14336, 128, q.PATH_AUTO, 152)
    assert p["kernel"] == q.KERNEL_W8A8_TC and p["tokens_per_tile"] == 256
    p = q.qlin_plan_info(q.OP_W8A8_BLOCK_GEMM, 256, 28672, 4096, 128, q.PATH_AUTO, 152)
    assert p["kernel"] == q.KERNEL_W8A8_BLOCK_TC and p["rows_per_tile"] == 256
    # a split K range always has a workspace of counters + FP32 partial sums
    p = q.qlin_plan_info(q.OP_W4A16_GEMM, 64, 4096, 14336, 128, q.PATH_TC, 152)
    tiles = (4096 // 128) * p["token_blocks"]
    assert p["splits"] > 1 and p["ws_bytes"] == (tiles * 4 + 255) // 256 * 256 + 4 * p["splits"] * 64 * 4096
    # the CUDA-core GEMV (K % 256 != 0) keeps its split-K sums in the workspace
    p = q.qlin_plan_info(q.OP_W4A16_GEMM, 4, 6144, 4224, 128, q.PATH_GEMV, 152)
    assert p["kernel"] == q.KERNEL_W4A16_GEMV and p["splits"] > 1 and p["ws_bytes"] > 0


def test_plan_query_rejects_what_the_call_rejects(lib):
    info = (ctypes.c_int64 * 8)()
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 4, 100, 4096, 128, 0, 152, info) == 2     # N % 128
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 4, 128, 4096, 48, 0, 152, info) == 2      # G
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 4, 128, 4096, 128, 5, 152, info) == 1     # path
    assert lib.qlin_plan_info(99, 4, 128, 4096, 128, 0, 152, info) == 1                  # op
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 0, 128, 4096, 128, 0, 152, info) == 2     # empty call
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 4, 128, 4096, 128, 0, 152, None) == 1
    # the CUDA-core GEMVs launch one grid row per 4 tokens: at most 65535 rows
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 4 * 65535, 128, 4224, 128, q.PATH_GEMV, 152, info) == 0
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 4 * 65535 + 1, 128, 4224, 128, q.PATH_GEMV, 152, info) == 2
    assert lib.qlin_plan_info(q.OP_W8A8_GEMM, 4 * 65535 + 1, 128, 4224, 128, q.PATH_GEMV, 152, info) == 2
    # G = 32 / 64 are tensor-core only when K % 256 != 0
    assert lib.qlin_plan_info(q.OP_W4A16_GEMM, 4, 128, 4224, 64, q.PATH_GEMV, 152, info) == 2


def test_fp4_plans_and_size_queries_without_device(lib):
    # FP4 K blocks are 256 columns (128 bytes): the plan of an E4M3 problem of K / 2 columns
    for op, kern in ((q.OP_MXFP4_GEMM, q.KERNEL_MXFP4_TC), (q.OP_NVFP4_GEMM, q.KERNEL_NVFP4_TC)):
        p = q.qlin_plan_info(op, 2048, 28672, 4096, 128, q.PATH_AUTO, 152)
        assert p["kernel"] == kern and p["tokens_per_tile"] == 256 and p["splits"] == 1
        p8 = q.qlin_plan_info(q.OP_MXFP8_GEMM, 8, 4096, 7168, 128, q.PATH_AUTO, 152)
        p4 = q.qlin_plan_info(op, 8, 4096, 14336, 128, q.PATH_AUTO, 152)
        assert (p4["tokens_per_tile"], p4["splits"], p4["ws_bytes"]) == (p8["tokens_per_tile"], p8["splits"],
                                                                          p8["ws_bytes"])
        assert p4["tokens_per_tile"] == 32 and p4["splits"] > 1
        assert q.qlin_plan_info(op, 1, 512, 1024, 128, q.PATH_AUTO, 152)["tokens_per_tile"] == 32
        # no 64-token FP4 tiles: from 33 tokens the tile is 128 or 256, and a 32-token tile is one token block
        for M in (33, 40, 64, 65, 100, 300, 2048):
            for N, K in ((512, 1024), (512, 28672), (4096, 4096), (14336, 8192)):
                assert q.qlin_plan_info(op, M, N, K, 128, q.PATH_AUTO, 152)["tokens_per_tile"] in (128, 256)
    info = (ctypes.c_int64 * 8)()
    assert lib.qlin_plan_info(q.OP_MXFP4_GEMM, 4, 128, 384, 128, 0, 152, info) == 2      # K % 256
    assert lib.qlin_plan_info(q.OP_NVFP4_GEMM, 4, 128, 384, 128, 0, 152, info) == 2
    # scale bytes: MXFP4 shares the MXFP8 atoms (K / 32 scales per row), NVFP4 K / 16 per row
    assert q.qlin_mx_scale_bytes(200, 512) == 256 * 512 // 32
    assert q.qlin_nvfp4_scale_bytes(200, 512) == 256 * 512 // 16
    b = ctypes.c_size_t()
    assert lib.qlin_nvfp4_scale_bytes(1, 384, ctypes.byref(b)) == 2
    # argument checks before any device work
    assert lib.qlin_quant_mxfp4(16, 1, 384, 16, 16, None) == 2
    assert lib.qlin_quant_nvfp4(16, 1, 256, None, 16, 16, None) == 1
    assert lib.qlin_nvfp4_tensor_scale(16, 12, 16, None) == 2
    assert lib.qlin_mxfp4_gemm(16, 16, 16, 16, 16, 1, 128, 384, None, 0, None) == 2
    assert lib.qlin_nvfp4_gemm(16, 16, None, 16, 16, 16, 16, 1, 128, 256, None, 0, None) == 1
