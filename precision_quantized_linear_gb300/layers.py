"""Layer objects that own the packed weights and the split-K workspace.

``W4A16Linear`` packs BF16 weights once at construction ([LP] S18 "pack once,
reuse") and runs ``qlin_w4a16_gemm`` per call; ``W8A8Linear`` quantises the
weights to E4M3 once and runs the fused per-token activation quantiser plus
``qlin_w8a8_fp8_gemm`` per call.  A layer built with a bias, or called with an
activation, runs the ``*_gemm_fused`` calls instead: bias and activation are
applied where the kernel writes Y (every layer here takes them).  Device
memory comes from torch; every computation is a libqlin kernel.
"""
from __future__ import annotations

import torch

from . import (ACT_NONE, OP_MXFP4_GEMM, OP_MXFP8_GEMM, OP_NVFP4_GEMM, OP_QUANT_W_FP8, OP_W4A8_GEMM, OP_W4A16_GEMM,
               OP_W8A8_BLOCK_GEMM, OP_W8A8_GEMM, PATH_AUTO, qlin_mx_scale_bytes, qlin_mxfp4_gemm, qlin_mxfp8_gemm,
               qlin_nvfp4_gemm, qlin_nvfp4_scale_bytes, qlin_nvfp4_tensor_scale, qlin_pack_w4, qlin_quant_mxfp4,
               qlin_quant_mxfp8, qlin_quant_nvfp4, qlin_w4a8_gemm, qlin_w4a8_gemm_fused, qlin_mxfp8_gemm_fused,
               qlin_mxfp4_gemm_fused, qlin_nvfp4_gemm_fused, qlin_w8a8_fp8_block_gemm_fused,
               qlin_quant_act_fp8, qlin_quant_act_fp8_blocks, qlin_quant_w_fp8, qlin_quant_w_fp8_blocks,
               qlin_w4_packed_sizes, qlin_w4a16_gemm_ex, qlin_w4a16_gemm_fused, qlin_w8a8_fp8_block_gemm,
               qlin_w8a8_fp8_gemm_ex, qlin_w8a8_fp8_gemm_fused, qlin_workspace_size)


def _as_u16(t: torch.Tensor) -> torch.Tensor:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    assert t.dtype in (torch.int16, torch.uint16)
    return t


class Workspace:
    """Zero-filled split-K scratch, grown on demand (the library leaves it zeroed)."""

    def __init__(self, device):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        if nbytes == 0:
            return None, 0
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf, self.buf.numel()


def _bias_bf16(bias, N):
    if bias is None:
        return None
    assert bias.shape == (N,) and bias.dtype == torch.bfloat16
    return bias.contiguous()


class W4A16Linear:
    def __init__(self, W_bf16: torch.Tensor, G: int = 128, symmetric: bool = False, stream=None, bias=None):
        N, K = W_bf16.shape
        self.N, self.K, self.G = N, K, G
        self.bias = _bias_bf16(bias, N)
        dev = W_bf16.device
        nc, ns, nz = qlin_w4_packed_sizes(N, K, G)
        self.codes = torch.empty(nc, dtype=torch.uint8, device=dev)
        self.scales = torch.empty(ns // 2, dtype=torch.int16, device=dev)
        self.zeros = torch.empty(nz, dtype=torch.uint8, device=dev)
        qlin_pack_w4(_as_u16(W_bf16.contiguous()), N, K, G, symmetric, self.codes, self.scales, self.zeros,
                     stream)
        self.ws = Workspace(dev)

    def packed_bytes(self) -> int:
        return self.codes.numel() + 2 * self.scales.numel() + self.zeros.numel()

    def __call__(self, X_bf16: torch.Tensor, Y: torch.Tensor = None, path: int = PATH_AUTO, stream=None,
                 act: int = ACT_NONE):
        M = X_bf16.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.bfloat16, device=X_bf16.device)
        buf, nb = self.ws.get(qlin_workspace_size(OP_W4A16_GEMM, M, self.N, self.K, self.G))
        if self.bias is None and act == ACT_NONE:
            qlin_w4a16_gemm_ex(_as_u16(X_bf16), self.codes, self.scales, self.zeros, Y.view(torch.int16), M, self.N,
                               self.K, self.G, buf, nb, path, stream)
        else:
            qlin_w4a16_gemm_fused(_as_u16(X_bf16), self.codes, self.scales, self.zeros, Y.view(torch.int16), M,
                                  self.N, self.K, self.G, self.bias, act, buf, nb, path, stream)
        return Y


class W4A8Linear(W4A16Linear):
    """W4A8: the packed INT4 weights of W4A16Linear (G = 128) times per-token E4M3
    activations from the fused amax quantiser."""

    def __init__(self, W_bf16: torch.Tensor, symmetric: bool = False, stream=None, bias=None):
        super().__init__(W_bf16, G=128, symmetric=symmetric, stream=stream, bias=bias)

    def quant_act(self, X_bf16: torch.Tensor, Xq=None, sx=None, stream=None):
        M, K = X_bf16.shape
        if Xq is None:
            Xq = torch.empty((M, K), dtype=torch.uint8, device=X_bf16.device)
        if sx is None:
            sx = torch.empty(max(M, 1), dtype=torch.float32, device=X_bf16.device)
        qlin_quant_act_fp8(_as_u16(X_bf16), M, K, Xq, sx, stream)
        return Xq, sx

    def gemm(self, Xq, sx, Y=None, stream=None, act: int = ACT_NONE):
        M = Xq.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.bfloat16, device=Xq.device)
        buf, nb = self.ws.get(qlin_workspace_size(OP_W4A8_GEMM, M, self.N, self.K, 128))
        if self.bias is None and act == ACT_NONE:
            qlin_w4a8_gemm(Xq, sx, self.codes, self.scales, self.zeros, Y.view(torch.int16), M, self.N, self.K, 128,
                           buf, nb, stream)
        else:
            qlin_w4a8_gemm_fused(Xq, sx, self.codes, self.scales, self.zeros, Y.view(torch.int16), M, self.N, self.K,
                                 128, self.bias, act, buf, nb, stream)
        return Y

    def __call__(self, X_bf16, Y=None, stream=None, act: int = ACT_NONE):
        Xq, sx = self.quant_act(X_bf16, stream=stream)
        return self.gemm(Xq, sx, Y, stream, act)


class W8A8Linear:
    def __init__(self, W_bf16: torch.Tensor, stream=None, bias=None):
        N, K = W_bf16.shape
        self.N, self.K = N, K
        self.bias = _bias_bf16(bias, N)
        dev = W_bf16.device
        self.Wq = torch.empty((N, K), dtype=torch.uint8, device=dev)
        self.sw = torch.empty(1, dtype=torch.float32, device=dev)
        ws = torch.zeros(qlin_workspace_size(OP_QUANT_W_FP8, 1, N, K), dtype=torch.uint8, device=dev)
        qlin_quant_w_fp8(_as_u16(W_bf16.contiguous()), N, K, self.Wq, self.sw, ws, ws.numel(), stream)
        self.ws = Workspace(dev)
        self._amax_ws = ws

    def quant_act(self, X_bf16: torch.Tensor, Xq=None, sx=None, stream=None):
        M, K = X_bf16.shape
        if Xq is None:
            Xq = torch.empty((M, K), dtype=torch.uint8, device=X_bf16.device)
        if sx is None:
            sx = torch.empty(max(M, 1), dtype=torch.float32, device=X_bf16.device)
        qlin_quant_act_fp8(_as_u16(X_bf16), M, K, Xq, sx, stream)
        return Xq, sx

    def gemm(self, Xq, sx, Y=None, path: int = PATH_AUTO, stream=None, act: int = ACT_NONE):
        M = Xq.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.bfloat16, device=Xq.device)
        buf, nb = self.ws.get(qlin_workspace_size(OP_W8A8_GEMM, M, self.N, self.K))
        if self.bias is None and act == ACT_NONE:
            qlin_w8a8_fp8_gemm_ex(Xq, sx, self.Wq, self.sw, Y.view(torch.int16), M, self.N, self.K, buf, nb, path,
                                  stream)
        else:
            qlin_w8a8_fp8_gemm_fused(Xq, sx, self.Wq, self.sw, Y.view(torch.int16), M, self.N, self.K, self.bias,
                                     act, buf, nb, path, stream)
        return Y

    def __call__(self, X_bf16, Y=None, path: int = PATH_AUTO, stream=None, act: int = ACT_NONE):
        Xq, sx = self.quant_act(X_bf16, stream=stream)
        return self.gemm(Xq, sx, Y, path, stream, act)


class W8A8BlockLinear:
    """FP8 W8A8 with block scaling: 128 x 128 weight blocks, 1 x 128 activation blocks."""

    def __init__(self, W_bf16: torch.Tensor, stream=None, bias=None):
        N, K = W_bf16.shape
        self.N, self.K = N, K
        self.bias = _bias_bf16(bias, N)
        dev = W_bf16.device
        self.Wq = torch.empty((N, K), dtype=torch.uint8, device=dev)
        self.sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
        qlin_quant_w_fp8_blocks(_as_u16(W_bf16.contiguous()), N, K, self.Wq, self.sw, stream)
        self.ws = Workspace(dev)

    def quant_act(self, X_bf16: torch.Tensor, Xq=None, sx=None, stream=None):
        M, K = X_bf16.shape
        if Xq is None:
            Xq = torch.empty((M, K), dtype=torch.uint8, device=X_bf16.device)
        if sx is None:
            sx = torch.empty((K // 128, max(M, 1)), dtype=torch.float32, device=X_bf16.device)
        qlin_quant_act_fp8_blocks(_as_u16(X_bf16), M, K, Xq, sx, stream)
        return Xq, sx

    def gemm(self, Xq, sx, Y=None, stream=None, act: int = ACT_NONE):
        M = Xq.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.bfloat16, device=Xq.device)
        buf, nb = self.ws.get(qlin_workspace_size(OP_W8A8_BLOCK_GEMM, M, self.N, self.K))
        if self.bias is None and act == ACT_NONE:
            qlin_w8a8_fp8_block_gemm(Xq, sx, self.Wq, self.sw, Y.view(torch.int16), M, self.N, self.K, buf, nb, stream)
        else:
            qlin_w8a8_fp8_block_gemm_fused(Xq, sx, self.Wq, self.sw, Y.view(torch.int16), M, self.N, self.K, self.bias,
                                           act, buf, nb, stream)
        return Y

    def __call__(self, X_bf16, Y=None, stream=None, act: int = ACT_NONE):
        Xq, sx = self.quant_act(X_bf16, stream=stream)
        return self.gemm(Xq, sx, Y, stream, act)


class MXFP8Linear:
    """MXFP8 W8A8: E4M3 weights and activations with E8M0 scales per 32 columns,
    both block scales applied by the tensor cores."""

    def __init__(self, W_bf16: torch.Tensor, stream=None, bias=None):
        N, K = W_bf16.shape
        self.N, self.K = N, K
        self.bias = _bias_bf16(bias, N)
        dev = W_bf16.device
        self.Wq = torch.empty((N, K), dtype=torch.uint8, device=dev)
        self.ws_sf = torch.empty(qlin_mx_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        qlin_quant_mxfp8(_as_u16(W_bf16.contiguous()), N, K, self.Wq, self.ws_sf, stream)
        self.ws = Workspace(dev)

    def quant_act(self, X_bf16: torch.Tensor, Xq=None, xs=None, stream=None):
        M, K = X_bf16.shape
        if Xq is None:
            Xq = torch.empty((M, K), dtype=torch.uint8, device=X_bf16.device)
        if xs is None:
            xs = torch.empty(max(qlin_mx_scale_bytes(M, K), 16), dtype=torch.uint8, device=X_bf16.device)
        qlin_quant_mxfp8(_as_u16(X_bf16), M, K, Xq, xs, stream)
        return Xq, xs

    def gemm(self, Xq, xs, Y=None, stream=None, act: int = ACT_NONE):
        M = Xq.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.bfloat16, device=Xq.device)
        buf, nb = self.ws.get(qlin_workspace_size(OP_MXFP8_GEMM, M, self.N, self.K))
        if self.bias is None and act == ACT_NONE:
            qlin_mxfp8_gemm(Xq, xs, self.Wq, self.ws_sf, Y.view(torch.int16), M, self.N, self.K, buf, nb, stream)
        else:
            qlin_mxfp8_gemm_fused(Xq, xs, self.Wq, self.ws_sf, Y.view(torch.int16), M, self.N, self.K, self.bias, act,
                                  buf, nb, stream)
        return Y

    def __call__(self, X_bf16, Y=None, stream=None, act: int = ACT_NONE):
        Xq, xs = self.quant_act(X_bf16, stream=stream)
        return self.gemm(Xq, xs, Y, stream, act)


class MXFP4Linear:
    """MXFP4 W4A4: E2M1 weights and activations (two per byte) with E8M0 scales
    per 32 columns, both block scales applied by the tensor cores."""

    def __init__(self, W_bf16: torch.Tensor, stream=None, bias=None):
        N, K = W_bf16.shape
        self.N, self.K = N, K
        self.bias = _bias_bf16(bias, N)
        dev = W_bf16.device
        self.Wq = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
        self.ws_sf = torch.empty(qlin_mx_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        qlin_quant_mxfp4(_as_u16(W_bf16.contiguous()), N, K, self.Wq, self.ws_sf, stream)
        self.ws = Workspace(dev)

    def quant_act(self, X_bf16: torch.Tensor, Xq=None, xs=None, stream=None):
        M, K = X_bf16.shape
        if Xq is None:
            Xq = torch.empty((M, K // 2), dtype=torch.uint8, device=X_bf16.device)
        if xs is None:
            xs = torch.empty(max(qlin_mx_scale_bytes(M, K), 16), dtype=torch.uint8, device=X_bf16.device)
        qlin_quant_mxfp4(_as_u16(X_bf16), M, K, Xq, xs, stream)
        return Xq, xs

    def gemm(self, Xq, xs, Y=None, stream=None, act: int = ACT_NONE):
        M = Xq.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.bfloat16, device=Xq.device)
        buf, nb = self.ws.get(qlin_workspace_size(OP_MXFP4_GEMM, M, self.N, self.K))
        if self.bias is None and act == ACT_NONE:
            qlin_mxfp4_gemm(Xq, xs, self.Wq, self.ws_sf, Y.view(torch.int16), M, self.N, self.K, buf, nb, stream)
        else:
            qlin_mxfp4_gemm_fused(Xq, xs, self.Wq, self.ws_sf, Y.view(torch.int16), M, self.N, self.K, self.bias, act,
                                  buf, nb, stream)
        return Y

    def __call__(self, X_bf16, Y=None, stream=None, act: int = ACT_NONE):
        Xq, xs = self.quant_act(X_bf16, stream=stream)
        return self.gemm(Xq, xs, Y, stream, act)


class NVFP4Linear:
    """NVFP4 W4A4: E2M1 weights and activations with E4M3 scales per 16 columns
    and one FP32 scale per tensor; the block scales are applied by the tensor
    cores, the two tensor scales in the epilogue.  The activations' tensor scale
    is computed on the device for every call (an amax reduction before the
    quantiser)."""

    def __init__(self, W_bf16: torch.Tensor, stream=None, bias=None):
        N, K = W_bf16.shape
        self.N, self.K = N, K
        self.bias = _bias_bf16(bias, N)
        dev = W_bf16.device
        W = _as_u16(W_bf16.contiguous())
        self.sgw = torch.empty(4, dtype=torch.float32, device=dev)
        qlin_nvfp4_tensor_scale(W, N * K, self.sgw, stream)
        self.Wq = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
        self.ws_sf = torch.empty(qlin_nvfp4_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        qlin_quant_nvfp4(W, N, K, self.sgw, self.Wq, self.ws_sf, stream)
        self.ws = Workspace(dev)

    def quant_act(self, X_bf16: torch.Tensor, Xq=None, xs=None, sgx=None, stream=None):
        M, K = X_bf16.shape
        dev = X_bf16.device
        if Xq is None:
            Xq = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
        if xs is None:
            xs = torch.empty(max(qlin_nvfp4_scale_bytes(M, K), 16), dtype=torch.uint8, device=dev)
        if sgx is None:
            sgx = torch.empty(4, dtype=torch.float32, device=dev)
        X = _as_u16(X_bf16)
        qlin_nvfp4_tensor_scale(X, M * K, sgx, stream)
        qlin_quant_nvfp4(X, M, K, sgx, Xq, xs, stream)
        return Xq, xs, sgx

    def gemm(self, Xq, xs, sgx, Y=None, stream=None, act: int = ACT_NONE):
        M = Xq.shape[0]
        if Y is None:
            Y = torch.empty((M, self.N), dtype=torch.bfloat16, device=Xq.device)
        buf, nb = self.ws.get(qlin_workspace_size(OP_NVFP4_GEMM, M, self.N, self.K))
        if self.bias is None and act == ACT_NONE:
            qlin_nvfp4_gemm(Xq, xs, sgx, self.Wq, self.ws_sf, self.sgw, Y.view(torch.int16), M, self.N, self.K, buf,
                            nb, stream)
        else:
            qlin_nvfp4_gemm_fused(Xq, xs, sgx, self.Wq, self.ws_sf, self.sgw, Y.view(torch.int16), M, self.N, self.K,
                                  self.bias, act, buf, nb, stream)
        return Y

    def __call__(self, X_bf16, Y=None, stream=None, act: int = ACT_NONE):
        Xq, xs, sgx = self.quant_act(X_bf16, stream=stream)
        return self.gemm(Xq, xs, sgx, Y, stream, act)
