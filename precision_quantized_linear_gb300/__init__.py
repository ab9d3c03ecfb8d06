"""qlin: GB300-native quantized linear layers (W4A16 INT4 and W8A8 FP8-E4M3).

Thin ctypes binding over ``libqlin.so`` (the C ABI declared in
``include/qlin.h``).  The ``qlin_*`` functions take the same arguments as the
C calls, with torch CUDA tensors in place of device pointers, and raise
``QlinError`` on a non-zero status; every step of the computation runs in the
library's CUDA kernels.  PyTorch is only used for device memory and streams.

If the shared library is missing the first call raises: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build_mod

__all__ = [
    "QlinError", "load", "build",
    "qlin_status_string", "qlin_pack_format_version", "qlin_last_cuda_error", "qlin_cuda_error_name",
    "qlin_w4_packed_sizes", "qlin_workspace_size",
    "qlin_pack_w4", "qlin_w4a16_gemm", "qlin_w4a16_gemm_ex", "qlin_quant_act_fp8", "qlin_quant_w_fp8",
    "qlin_w8a8_fp8_gemm", "qlin_w8a8_fp8_gemm_ex", "qlin_get_device_error", "qlin_gemv_max_m",
    "qlin_selftest_wait_timeout", "qlin_w4a16_gemv_noalloc", "qlin_quant_act_fp8_blocks", "qlin_quant_w_fp8_blocks",
    "qlin_w8a8_fp8_block_gemm", "OP_W4A16_GEMM", "OP_W8A8_GEMM", "OP_QUANT_W_FP8", "OP_W8A8_BLOCK_GEMM",
    "PATH_AUTO", "PATH_GEMV", "PATH_TC", "ACT_NONE", "ACT_RELU", "ACT_SILU", "ACT_GELU",
    "qlin_w4a16_gemm_fused", "qlin_w8a8_fp8_gemm_fused",
    "PACK_FORMAT_VERSION", "qlin_plan_info", "PLAN_FIELDS",
    "KERNEL_W4A16_MMA", "KERNEL_W4A16_GEMV", "KERNEL_W4A16_TC", "KERNEL_W8A8_MMA", "KERNEL_W8A8_GEMV",
    "KERNEL_W8A8_TC", "KERNEL_W8A8_BLOCK_TC", "KERNEL_MXFP8_TC", "OP_MXFP8_GEMM",
    "qlin_mx_scale_bytes", "qlin_quant_mxfp8", "qlin_mxfp8_gemm", "qlin_w4a8_gemm", "OP_W4A8_GEMM",
    "KERNEL_W4A8_TC", "OP_MXFP4_GEMM", "OP_NVFP4_GEMM", "KERNEL_MXFP4_TC", "KERNEL_NVFP4_TC",
    "qlin_nvfp4_scale_bytes", "qlin_quant_mxfp4", "qlin_nvfp4_tensor_scale", "qlin_quant_nvfp4", "qlin_mxfp4_gemm",
    "qlin_nvfp4_gemm", "qlin_w4a8_gemm_fused", "qlin_mxfp8_gemm_fused", "qlin_mxfp4_gemm_fused",
    "qlin_nvfp4_gemm_fused", "qlin_w8a8_fp8_block_gemm_fused",
]

OP_W4A16_GEMM, OP_W8A8_GEMM, OP_QUANT_W_FP8, OP_W8A8_BLOCK_GEMM, OP_MXFP8_GEMM, OP_W4A8_GEMM = 1, 2, 3, 4, 5, 6
OP_MXFP4_GEMM, OP_NVFP4_GEMM = 7, 8
PATH_AUTO, PATH_GEMV, PATH_TC = 0, 1, 2
(KERNEL_W4A16_MMA, KERNEL_W4A16_GEMV, KERNEL_W4A16_TC, KERNEL_W8A8_MMA, KERNEL_W8A8_GEMV, KERNEL_W8A8_TC,
 KERNEL_W8A8_BLOCK_TC, KERNEL_MXFP8_TC, KERNEL_W4A8_TC, KERNEL_MXFP4_TC, KERNEL_NVFP4_TC) = range(1, 12)
ACT_NONE, ACT_RELU, ACT_SILU, ACT_GELU = 0, 1, 2, 3
PACK_FORMAT_VERSION = 2

_lock = threading.Lock()
_lib = None
_i64 = ctypes.c_int64
_p = ctypes.c_void_p
_sz = ctypes.c_size_t
_int = ctypes.c_int

# name -> argtypes (restype is int for all but qlin_status_string)
_SIGS = {
    "qlin_status_string": [_int],
    "qlin_pack_format_version": [],
    "qlin_last_cuda_error": [],
    "qlin_cuda_error_name": [_int],
    "qlin_gemv_max_m": [_int],
    "qlin_w4_packed_sizes": [_i64, _i64, _int, ctypes.POINTER(_sz), ctypes.POINTER(_sz), ctypes.POINTER(_sz)],
    "qlin_workspace_size": [_int, _i64, _i64, _i64, _int, ctypes.POINTER(_sz)],
    "qlin_plan_info": [_int, _i64, _i64, _i64, _int, _int, _int, ctypes.POINTER(_i64)],
    "qlin_pack_w4": [_p, _i64, _i64, _int, _int, _p, _p, _p, _p],
    "qlin_w4a16_gemm": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _int, _p, _sz, _p],
    "qlin_w4a16_gemm_ex": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _int, _p, _sz, _int, _p],
    "qlin_quant_act_fp8": [_p, _i64, _i64, _p, _p, _p],
    "qlin_quant_w_fp8": [_p, _i64, _i64, _p, _p, _p, _sz, _p],
    "qlin_w8a8_fp8_gemm": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _sz, _p],
    "qlin_w8a8_fp8_gemm_ex": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _sz, _int, _p],
    "qlin_w4a16_gemm_fused": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _int, _p, _int, _p, _sz, _int, _p],
    "qlin_w8a8_fp8_gemm_fused": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _int, _p, _sz, _int, _p],
    "qlin_get_device_error": [_p],
    "qlin_selftest_wait_timeout": [ctypes.c_uint32, _p],
    "qlin_w4a16_gemv_noalloc": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _int, _p],
    "qlin_quant_act_fp8_blocks": [_p, _i64, _i64, _p, _p, _p],
    "qlin_quant_w_fp8_blocks": [_p, _i64, _i64, _p, _p, _p],
    "qlin_w8a8_fp8_block_gemm": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _sz, _p],
    "qlin_mx_scale_bytes": [_i64, _i64, ctypes.POINTER(_sz)],
    "qlin_w4a8_gemm": [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _int, _p, _sz, _p],
    "qlin_quant_mxfp8": [_p, _i64, _i64, _p, _p, _p],
    "qlin_mxfp8_gemm": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _sz, _p],
    "qlin_nvfp4_scale_bytes": [_i64, _i64, ctypes.POINTER(_sz)],
    "qlin_quant_mxfp4": [_p, _i64, _i64, _p, _p, _p],
    "qlin_nvfp4_tensor_scale": [_p, _i64, _p, _p],
    "qlin_quant_nvfp4": [_p, _i64, _i64, _p, _p, _p, _p],
    "qlin_mxfp4_gemm": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _sz, _p],
    "qlin_nvfp4_gemm": [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _sz, _p],
    "qlin_w4a8_gemm_fused": [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _int, _p, _int, _p, _sz, _p],
    "qlin_mxfp8_gemm_fused": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _int, _p, _sz, _p],
    "qlin_mxfp4_gemm_fused": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _int, _p, _sz, _p],
    "qlin_nvfp4_gemm_fused": [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _int, _p, _sz, _p],
    "qlin_w8a8_fp8_block_gemm_fused": [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _int, _p, _sz, _p],
}


class QlinError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.cuda_error = 0
        msg = "%s failed: %s (%d)" % (where, qlin_status_string(status), status)
        if self.status == 6:  # QLIN_ERR_CUDA: name the CUDA error behind it
            self.cuda_error = qlin_last_cuda_error()
            msg += " [%s]" % qlin_cuda_error_name(self.cuda_error)
        super().__init__(msg)


def build(force: bool = False) -> str:
    return _build_mod.build(force=force)


def lib_path() -> str:
    return _build_mod.LIB


def load():
    """Load libqlin.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build_mod.LIB
        if not os.path.exists(path):
            raise RuntimeError("libqlin.so is not built (%s); run precision_quantized_linear_gb300.build()" % path)
        lib = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name in ("qlin_status_string", "qlin_cuda_error_name") else _int
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str) -> int:
    if st != 0:
        raise QlinError(st, where)
    return st


def qlin_status_string(status: int) -> str:
    return load().qlin_status_string(int(status)).decode()


def qlin_last_cuda_error() -> int:
    return load().qlin_last_cuda_error()


def qlin_cuda_error_name(code: int) -> str:
    return load().qlin_cuda_error_name(int(code)).decode()


def qlin_pack_format_version() -> int:
    return load().qlin_pack_format_version()


def qlin_gemv_max_m(op: int) -> int:
    return load().qlin_gemv_max_m(op)


def qlin_w4_packed_sizes(N: int, K: int, G: int = 128):
    a, b, c = _sz(), _sz(), _sz()
    _check(load().qlin_w4_packed_sizes(N, K, G, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
           "qlin_w4_packed_sizes")
    return a.value, b.value, c.value


def qlin_workspace_size(op: int, M: int, N: int, K: int, G: int = 128) -> int:
    b = _sz()
    _check(load().qlin_workspace_size(op, M, N, K, G, ctypes.byref(b)), "qlin_workspace_size")
    return b.value


PLAN_FIELDS = ("kernel", "tokens_per_tile", "rows_per_tile", "kblocks_per_stage", "splits", "ws_bytes",
               "a_in_tmem", "token_blocks")


def qlin_plan_info(op: int, M: int, N: int, K: int, G: int = 128, path: int = 0, num_sms: int = 0) -> dict:
    """Kernel and tiling a GEMM call would launch (launches nothing): a dict of PLAN_FIELDS."""
    info = (_i64 * 8)()
    _check(load().qlin_plan_info(op, M, N, K, G, path, num_sms, info), "qlin_plan_info")
    return dict(zip(PLAN_FIELDS, (int(v) for v in info)))


def qlin_pack_w4(W, N, K, G, symmetric, codes, scales, zeros, stream=None):
    return _check(load().qlin_pack_w4(_ptr(W), N, K, G, int(symmetric), _ptr(codes), _ptr(scales), _ptr(zeros),
                                      _stream(stream)), "qlin_pack_w4")


def qlin_w4a16_gemm(X, codes, scales, zeros, Y, M, N, K, G, workspace, ws_bytes, stream=None):
    return _check(load().qlin_w4a16_gemm(_ptr(X), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(Y), M, N, K, G,
                                         _ptr(workspace), ws_bytes, _stream(stream)), "qlin_w4a16_gemm")


def qlin_w4a16_gemm_ex(X, codes, scales, zeros, Y, M, N, K, G, workspace, ws_bytes, path, stream=None):
    return _check(load().qlin_w4a16_gemm_ex(_ptr(X), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(Y), M, N, K, G,
                                            _ptr(workspace), ws_bytes, path, _stream(stream)), "qlin_w4a16_gemm_ex")


def qlin_w4a16_gemm_fused(X, codes, scales, zeros, Y, M, N, K, G, bias, act, workspace, ws_bytes, path,
                          stream=None):
    return _check(load().qlin_w4a16_gemm_fused(_ptr(X), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(Y), M, N, K,
                                               G, _ptr(bias), act, _ptr(workspace), ws_bytes, path,
                                               _stream(stream)), "qlin_w4a16_gemm_fused")


def qlin_quant_act_fp8(X, M, K, Xq, sx, stream=None):
    return _check(load().qlin_quant_act_fp8(_ptr(X), M, K, _ptr(Xq), _ptr(sx), _stream(stream)),
                  "qlin_quant_act_fp8")


def qlin_quant_w_fp8(W, N, K, Wq, sw, workspace, ws_bytes, stream=None):
    return _check(load().qlin_quant_w_fp8(_ptr(W), N, K, _ptr(Wq), _ptr(sw), _ptr(workspace), ws_bytes,
                                          _stream(stream)), "qlin_quant_w_fp8")


def qlin_w8a8_fp8_gemm(Xq, sx, Wq, sw, Y, M, N, K, workspace, ws_bytes, stream=None):
    return _check(load().qlin_w8a8_fp8_gemm(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(Y), M, N, K,
                                            _ptr(workspace), ws_bytes, _stream(stream)), "qlin_w8a8_fp8_gemm")


def qlin_w8a8_fp8_gemm_ex(Xq, sx, Wq, sw, Y, M, N, K, workspace, ws_bytes, path, stream=None):
    return _check(load().qlin_w8a8_fp8_gemm_ex(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(Y), M, N, K,
                                               _ptr(workspace), ws_bytes, path, _stream(stream)),
                  "qlin_w8a8_fp8_gemm_ex")


def qlin_w8a8_fp8_gemm_fused(Xq, sx, Wq, sw, Y, M, N, K, bias, act, workspace, ws_bytes, path, stream=None):
    return _check(load().qlin_w8a8_fp8_gemm_fused(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(Y), M, N, K,
                                                  _ptr(bias), act, _ptr(workspace), ws_bytes, path,
                                                  _stream(stream)), "qlin_w8a8_fp8_gemm_fused")


def qlin_quant_act_fp8_blocks(X, M, K, Xq, sx, stream=None):
    return _check(load().qlin_quant_act_fp8_blocks(_ptr(X), M, K, _ptr(Xq), _ptr(sx), _stream(stream)),
                  "qlin_quant_act_fp8_blocks")


def qlin_quant_w_fp8_blocks(W, N, K, Wq, sw, stream=None):
    return _check(load().qlin_quant_w_fp8_blocks(_ptr(W), N, K, _ptr(Wq), _ptr(sw), _stream(stream)),
                  "qlin_quant_w_fp8_blocks")


def qlin_w8a8_fp8_block_gemm(Xq, sx, Wq, sw, Y, M, N, K, workspace, ws_bytes, stream=None):
    return _check(load().qlin_w8a8_fp8_block_gemm(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(Y), M, N, K,
                                                  _ptr(workspace), ws_bytes, _stream(stream)),
                  "qlin_w8a8_fp8_block_gemm")


def qlin_w4a8_gemm(Xq, sx, codes, scales, zeros, Y, M, N, K, G, workspace, ws_bytes, stream=None):
    return _check(load().qlin_w4a8_gemm(_ptr(Xq), _ptr(sx), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(Y), M, N,
                                        K, G, _ptr(workspace), ws_bytes, _stream(stream)), "qlin_w4a8_gemm")


def qlin_mx_scale_bytes(R: int, K: int) -> int:
    b = _sz()
    _check(load().qlin_mx_scale_bytes(R, K, ctypes.byref(b)), "qlin_mx_scale_bytes")
    return b.value


def qlin_quant_mxfp8(X, R, K, codes, scales, stream=None):
    return _check(load().qlin_quant_mxfp8(_ptr(X), R, K, _ptr(codes), _ptr(scales), _stream(stream)),
                  "qlin_quant_mxfp8")


def qlin_mxfp8_gemm(Xq, xs, Wq, ws_sf, Y, M, N, K, workspace, ws_bytes, stream=None):
    return _check(load().qlin_mxfp8_gemm(_ptr(Xq), _ptr(xs), _ptr(Wq), _ptr(ws_sf), _ptr(Y), M, N, K,
                                         _ptr(workspace), ws_bytes, _stream(stream)), "qlin_mxfp8_gemm")


def qlin_nvfp4_scale_bytes(R: int, K: int) -> int:
    b = _sz()
    _check(load().qlin_nvfp4_scale_bytes(R, K, ctypes.byref(b)), "qlin_nvfp4_scale_bytes")
    return b.value


def qlin_quant_mxfp4(X, R, K, codes, scales, stream=None):
    return _check(load().qlin_quant_mxfp4(_ptr(X), R, K, _ptr(codes), _ptr(scales), _stream(stream)),
                  "qlin_quant_mxfp4")


def qlin_nvfp4_tensor_scale(X, n, sg, stream=None):
    return _check(load().qlin_nvfp4_tensor_scale(_ptr(X), n, _ptr(sg), _stream(stream)), "qlin_nvfp4_tensor_scale")


def qlin_quant_nvfp4(X, R, K, sg, codes, scales, stream=None):
    return _check(load().qlin_quant_nvfp4(_ptr(X), R, K, _ptr(sg), _ptr(codes), _ptr(scales), _stream(stream)),
                  "qlin_quant_nvfp4")


def qlin_mxfp4_gemm(Xq, xs, Wq, ws_sf, Y, M, N, K, workspace, ws_bytes, stream=None):
    return _check(load().qlin_mxfp4_gemm(_ptr(Xq), _ptr(xs), _ptr(Wq), _ptr(ws_sf), _ptr(Y), M, N, K,
                                         _ptr(workspace), ws_bytes, _stream(stream)), "qlin_mxfp4_gemm")


def qlin_nvfp4_gemm(Xq, xs, sgx, Wq, ws_sf, sgw, Y, M, N, K, workspace, ws_bytes, stream=None):
    return _check(load().qlin_nvfp4_gemm(_ptr(Xq), _ptr(xs), _ptr(sgx), _ptr(Wq), _ptr(ws_sf), _ptr(sgw), _ptr(Y),
                                         M, N, K, _ptr(workspace), ws_bytes, _stream(stream)), "qlin_nvfp4_gemm")


def qlin_w4a8_gemm_fused(Xq, sx, codes, scales, zeros, Y, M, N, K, G, bias, act, workspace, ws_bytes, stream=None):
    return _check(load().qlin_w4a8_gemm_fused(_ptr(Xq), _ptr(sx), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(Y),
                                              M, N, K, G, _ptr(bias), act, _ptr(workspace), ws_bytes,
                                              _stream(stream)), "qlin_w4a8_gemm_fused")


def qlin_mxfp8_gemm_fused(Xq, xs, Wq, ws_sf, Y, M, N, K, bias, act, workspace, ws_bytes, stream=None):
    return _check(load().qlin_mxfp8_gemm_fused(_ptr(Xq), _ptr(xs), _ptr(Wq), _ptr(ws_sf), _ptr(Y), M, N, K,
                                               _ptr(bias), act, _ptr(workspace), ws_bytes, _stream(stream)),
                  "qlin_mxfp8_gemm_fused")


def qlin_mxfp4_gemm_fused(Xq, xs, Wq, ws_sf, Y, M, N, K, bias, act, workspace, ws_bytes, stream=None):
    return _check(load().qlin_mxfp4_gemm_fused(_ptr(Xq), _ptr(xs), _ptr(Wq), _ptr(ws_sf), _ptr(Y), M, N, K,
                                               _ptr(bias), act, _ptr(workspace), ws_bytes, _stream(stream)),
                  "qlin_mxfp4_gemm_fused")


def qlin_nvfp4_gemm_fused(Xq, xs, sgx, Wq, ws_sf, sgw, Y, M, N, K, bias, act, workspace, ws_bytes, stream=None):
    return _check(load().qlin_nvfp4_gemm_fused(_ptr(Xq), _ptr(xs), _ptr(sgx), _ptr(Wq), _ptr(ws_sf), _ptr(sgw),
                                               _ptr(Y), M, N, K, _ptr(bias), act, _ptr(workspace), ws_bytes,
                                               _stream(stream)), "qlin_nvfp4_gemm_fused")


def qlin_get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return load().qlin_get_device_error(_stream(stream))


def qlin_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    """Launch the bounded-wait self-test kernel (see include/qlin.h)."""
    return _check(load().qlin_selftest_wait_timeout(int(limit_us), _stream(stream)), "qlin_selftest_wait_timeout")


def qlin_w4a16_gemv_noalloc(X, codes, scales, zeros, Y, M, N, K, G, stream=None):
    """W4A16 GEMV whose scratch is a fixed array inside the library (no workspace
    argument, nothing allocated): for callers that cannot allocate device memory."""
    return _check(load().qlin_w4a16_gemv_noalloc(_ptr(X), _ptr(codes), _ptr(scales), _ptr(zeros), _ptr(Y), M, N, K,
                                                 G, _stream(stream)), "qlin_w4a16_gemv_noalloc")


def qlin_w8a8_fp8_block_gemm_fused(Xq, sx, Wq, sw, Y, M, N, K, bias, act, workspace, ws_bytes, stream=None):
    return _check(load().qlin_w8a8_fp8_block_gemm_fused(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(Y), M, N, K,
                                                        _ptr(bias), act, _ptr(workspace), ws_bytes,
                                                        _stream(stream)), "qlin_w8a8_fp8_block_gemm_fused")
