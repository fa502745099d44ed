"""ctypes binding of libfp8bs.so -- the same call names as include/fp8bs.h.

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch provides device memory and
streams); outputs not passed in are allocated here with torch.  Importing this
module raises ImportError if the library has not been built
(``python -m fp8_block_scaled_18_b300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libfp8bs.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fp8bs.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m fp8_block_scaled_18_b300.build`")

lib = ctypes.CDLL(LIB_PATH)

_P, _I64, _I32, _SZ, _U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_uint64
_ST = ctypes.c_int

_SIGS = {
    "fp8bs_act_quant": (_ST, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P]),
    "fp8bs_weight_quant": (_ST, [_P, _I64, _I64, _P, _P, _P]),
    "fp8bs_act_quant_pow2": (_ST, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P]),
    "fp8bs_weight_quant_pow2": (_ST, [_P, _I64, _I64, _P, _P, _P]),
    "fp8bs_weight_dequant": (_ST, [_P, _P, _I64, _I64, _P, _P]),
    "fp8bs_gemm": (_ST, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _SZ, _P]),
    "fp8bs_gemm_fused": (_ST, [_P, _P, _I64, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P]),
    "fp8bs_gemm_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "fp8bs_gemm_noalloc": (_ST, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _I64, _P]),
    "fp8bs_grouped_gemm": (_ST, [_P, _P, _I64, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _I64, _P]),
    "fp8bs_grouped_gemm_workspace_size": (_SZ, [_I32, _I64, _I64]),
    "fp8bs_act_quant_cols": (_ST, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P]),
    "fp8bs_gemm_wgrad": (_ST, [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _I64, _P]),
    "fp8bs_grouped_gemm_swiglu": (_ST, [_P, _P, _I64, _P, _P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _I64, _P,
                                        _I64, _P, _I64, _P]),
    "fp8bs_moe_dispatch": (_ST, [_P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P]),
    "fp8bs_moe_combine": (_ST, [_P, _I64, _I64, _P, _P, _I64, _I32, _I64, _P, _I64, _P, _I64, _P]),
    "fp8bs_moe_gate": (_ST, [_P, _I64, _P, _P, _I64, _I64, _I32, _I32, _I32, _I32, ctypes.c_float, _P, _P, _P]),
    "fp8bs_moe_route": (_ST, [_P, _P, _I64, _I32, _I32, _P, _P, _P, _P, _P]),
    "fp8bs_sync_status": (_ST, [_P]),
    "fp8bs_status_string": (ctypes.c_char_p, [_ST]),
    "fp8bs_e4m3_encode_f32": (_ST, [_P, _I64, _P, _P]),
    "fp8bs_debug_wait_timeout": (_ST, [_U64, _P]),
    "fp8bs_version": (ctypes.c_int, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

FP8BS_OK = 0
FP8BS_ERR_INVALID_ARG = 1
FP8BS_ERR_UNSUPPORTED = 2
FP8BS_ERR_MISALIGNED = 3
FP8BS_ERR_CUDA = 4
FP8BS_ERR_TIMEOUT = 5
FP8BS_ERR_INDEX = 6


class Fp8bsError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {fp8bs_status_string(status)}")


def declared_symbols() -> list[str]:
    """Every function name include/fp8bs.h declares."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"\b(fp8bs_[a-z0-9_]+)\s*\(", text)))


def fp8bs_status_string(status: int) -> str:
    return lib.fp8bs_status_string(status).decode()


def fp8bs_version() -> int:
    return lib.fp8bs_version()


def _check(status: int, call: str) -> None:
    if status != FP8BS_OK:
        raise Fp8bsError(status, call)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _rows_stride(t: torch.Tensor, name: str) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")
    return t.stride(0)


# bf16 tensors are passed as their bit patterns; both torch.bfloat16 and
# int16/uint16 views are accepted.
def _bf16_ptr(t: torch.Tensor, name: str) -> int:
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must be bfloat16 (or its 16-bit bit pattern)")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr()


def fp8bs_act_quant(x: torch.Tensor, xq: Optional[torch.Tensor] = None, sx: Optional[torch.Tensor] = None,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """x [M, K] bf16 -> (xq [M, K] uint8 e4m3, sx [M, lds] fp32)."""
    M, K = x.shape
    ldx = _rows_stride(x, "x")
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((M, max(4, ((K // 128) + 3) // 4 * 4)), dtype=torch.float32, device=x.device)
    _check(lib.fp8bs_act_quant(_bf16_ptr(x, "x"), M, K, ldx, _dev(xq, torch.uint8, "xq"),
                               _rows_stride(xq, "xq"), _dev(sx, torch.float32, "sx"),
                               _rows_stride(sx, "sx"), _stream(stream)), "fp8bs_act_quant")
    return xq, sx


def fp8bs_weight_quant(w: torch.Tensor, wq: Optional[torch.Tensor] = None, sw: Optional[torch.Tensor] = None,
                       stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """w [N, K] bf16 (dense) -> (wq [N, K] uint8, sw [ceil(N/128), K/128] fp32)."""
    N, K = w.shape
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if sw is None:
        sw = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=w.device)
    _check(lib.fp8bs_weight_quant(_bf16_ptr(w, "w"), N, K, _dev(wq, torch.uint8, "wq"),
                                  _dev(sw, torch.float32, "sw"), _stream(stream)), "fp8bs_weight_quant")
    return wq, sw


def fp8bs_act_quant_pow2(x: torch.Tensor, xq: Optional[torch.Tensor] = None, sx: Optional[torch.Tensor] = None,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """x [M, K] bf16 -> (xq [M, K] uint8 e4m3, sx [M, lds] fp32)."""
    M, K = x.shape
    ldx = _rows_stride(x, "x")
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((M, max(4, ((K // 128) + 3) // 4 * 4)), dtype=torch.float32, device=x.device)
    _check(lib.fp8bs_act_quant_pow2(_bf16_ptr(x, "x"), M, K, ldx, _dev(xq, torch.uint8, "xq"),
                               _rows_stride(xq, "xq"), _dev(sx, torch.float32, "sx"),
                               _rows_stride(sx, "sx"), _stream(stream)), "fp8bs_act_quant_pow2")
    return xq, sx


def fp8bs_weight_quant_pow2(w: torch.Tensor, wq: Optional[torch.Tensor] = None, sw: Optional[torch.Tensor] = None,
                       stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """w [N, K] bf16 (dense) -> (wq [N, K] uint8, sw [ceil(N/128), K/128] fp32)."""
    N, K = w.shape
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if sw is None:
        sw = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=w.device)
    _check(lib.fp8bs_weight_quant_pow2(_bf16_ptr(w, "w"), N, K, _dev(wq, torch.uint8, "wq"),
                                  _dev(sw, torch.float32, "sw"), _stream(stream)), "fp8bs_weight_quant_pow2")
    return wq, sw


def fp8bs_weight_dequant(wq: torch.Tensor, sw: torch.Tensor, w: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """(wq [N, K] uint8, sw) -> w [N, K] bf16."""
    N, K = wq.shape
    if w is None:
        w = torch.empty((N, K), dtype=torch.bfloat16, device=wq.device)
    _check(lib.fp8bs_weight_dequant(_dev(wq, torch.uint8, "wq"), _dev(sw, torch.float32, "sw"), N, K,
                                    _bf16_ptr(w, "w"), _stream(stream)), "fp8bs_weight_dequant")
    return w


def _out_rows(M: int, N: int, device) -> torch.Tensor:
    """bf16 [M, N] output whose row stride is padded to a multiple of 8."""
    ld = (N + 7) // 8 * 8
    y = torch.empty((M, ld), dtype=torch.bfloat16, device=device)
    return y if ld == N else y[:, :N]


def fp8bs_gemm_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib.fp8bs_gemm_workspace_size(M, N, K))


def fp8bs_gemm(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
               y: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """y [M, N] bf16 = fp8_gemm(xq, sx, wq, sw); workspace: optional uint8 CUDA
    tensor for the split-K plan (see fp8bs_gemm_workspace_size)."""
    M, K = xq.shape
    N = wq.shape[0]
    if y is None:
        y = _out_rows(M, N, xq.device)
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (_dev(workspace, torch.uint8, "workspace"),
                                                            workspace.numel())
    _check(lib.fp8bs_gemm(_dev(xq, torch.uint8, "xq"), _dev(sx, torch.float32, "sx"), _rows_stride(sx, "sx"),
                          _dev(wq, torch.uint8, "wq"), _dev(sw, torch.float32, "sw"), M, N, K,
                          _bf16_ptr(y, "y"), _rows_stride(y, "y"), ws_ptr, ws_bytes, _stream(stream)),
           "fp8bs_gemm")
    return y


def fp8bs_gemm_fused(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
                     bias: Optional[torch.Tensor] = None, want_y: bool = True, want_fp8: bool = False,
                     y: Optional[torch.Tensor] = None, yq: Optional[torch.Tensor] = None,
                     sy: Optional[torch.Tensor] = None, stream=None):
    """fp8_gemm with the fused epilogue: returns (y, yq, sy), y [M, N] bf16 =
    gemm + bias (None unless want_y), and (yq [M, N] uint8 e4m3, sy [M, N/128]
    fp32) = y quantised per row per 128 columns (None unless want_fp8)."""
    M, K = xq.shape
    N = wq.shape[0]
    if bias is not None and (bias.dim() != 1 or bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous 1-D tensor of N elements")
    if want_y and y is None:
        y = _out_rows(M, N, xq.device)
    if want_fp8:
        if yq is None:
            yq = torch.empty((M, (N + 15) // 16 * 16), dtype=torch.uint8, device=xq.device)[:, :N]
        if sy is None:
            sy = torch.empty((M, max(4, (N // 128 + 3) // 4 * 4)), dtype=torch.float32, device=xq.device)
    _check(lib.fp8bs_gemm_fused(_dev(xq, torch.uint8, "xq"), _dev(sx, torch.float32, "sx"), _rows_stride(sx, "sx"),
                                _dev(wq, torch.uint8, "wq"), _dev(sw, torch.float32, "sw"),
                                None if bias is None else _bf16_ptr(bias, "bias"), M, N, K,
                                None if y is None else _bf16_ptr(y, "y"), 0 if y is None else _rows_stride(y, "y"),
                                None if yq is None else _dev(yq, torch.uint8, "yq"),
                                0 if yq is None else _rows_stride(yq, "yq"),
                                None if sy is None else _dev(sy, torch.float32, "sy"),
                                0 if sy is None else _rows_stride(sy, "sy"), _stream(stream)),
           "fp8bs_gemm_fused")
    return y, yq, (None if sy is None else sy[:, :N // 128])


def fp8bs_gemm_noalloc(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
                       y: torch.Tensor, stream=None) -> torch.Tensor:
    """fp8bs_gemm for callers that cannot allocate: the library takes its
    split-K scratch from a fixed device array; y must be supplied."""
    M, K = xq.shape
    N = wq.shape[0]
    _check(lib.fp8bs_gemm_noalloc(_dev(xq, torch.uint8, "xq"), _dev(sx, torch.float32, "sx"),
                                  _rows_stride(sx, "sx"), _dev(wq, torch.uint8, "wq"),
                                  _dev(sw, torch.float32, "sw"), M, N, K, _bf16_ptr(y, "y"),
                                  _rows_stride(y, "y"), _stream(stream)), "fp8bs_gemm_noalloc")
    return y


def fp8bs_act_quant_cols(x: torch.Tensor, xqt: Optional[torch.Tensor] = None, sc: Optional[torch.Tensor] = None,
                         stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """x [M, K] bf16 -> (xqt [K, ldt] e4m3, the codes transposed, ldt = M
    rounded up to 16; sc [ceil(M/128), K] fp32): 128x1 groups along the rows."""
    M, K = x.shape
    if xqt is None:
        xqt = torch.empty((K, (M + 15) // 16 * 16), dtype=torch.uint8, device=x.device)
    if sc is None:
        sc = torch.empty(((M + 127) // 128, K), dtype=torch.float32, device=x.device)
    _check(lib.fp8bs_act_quant_cols(_bf16_ptr(x, "x"), M, K, _rows_stride(x, "x"), _dev(xqt, torch.uint8, "xqt"),
                                    _rows_stride(xqt, "xqt"), _dev(sc, torch.float32, "sc"), _rows_stride(sc, "sc"),
                                    _stream(stream)), "fp8bs_act_quant_cols")
    return xqt, sc


def fp8bs_gemm_wgrad(dyqt: torch.Tensor, sdy: torch.Tensor, xqt: torch.Tensor, sx: torch.Tensor, T: int,
                     dw: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """dW [N, K] fp32 = dY^T X over T tokens from fp8bs_act_quant_cols of dY
    (dyqt [N, >=T], sdy) and of X (xqt [K, >=T], sx)."""
    N, K = dyqt.shape[0], xqt.shape[0]
    if dw is None:
        dw = torch.empty((N, (K + 3) // 4 * 4), dtype=torch.float32, device=dyqt.device)[:, :K]
    _check(lib.fp8bs_gemm_wgrad(_dev(dyqt, torch.uint8, "dyqt"), _rows_stride(dyqt, "dyqt"),
                                _dev(sdy, torch.float32, "sdy"), _rows_stride(sdy, "sdy"),
                                _dev(xqt, torch.uint8, "xqt"), _rows_stride(xqt, "xqt"),
                                _dev(sx, torch.float32, "sx"), _rows_stride(sx, "sx"), T, N, K,
                                _dev(dw, torch.float32, "dw"), _rows_stride(dw, "dw"), _stream(stream)),
           "fp8bs_gemm_wgrad")
    return dw


def fp8bs_grouped_gemm_workspace_size(G: int, N: int, K: int) -> int:
    return lib.fp8bs_grouped_gemm_workspace_size(G, N, K)


def fp8bs_grouped_gemm(xq: torch.Tensor, sx: torch.Tensor, wq: torch.Tensor, sw: torch.Tensor,
                       offsets: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """xq [T, K], wq [G, N, K], sw [G, ceil(N/128), K/128], offsets int32 [G+1]
    on the device -> y [T, N] bf16."""
    T, K = xq.shape
    G, N, _ = wq.shape
    if y is None:
        y = _out_rows(T, N, xq.device)
    _check(lib.fp8bs_grouped_gemm(_dev(xq, torch.uint8, "xq"), _dev(sx, torch.float32, "sx"),
                                  _rows_stride(sx, "sx"), _dev(wq, torch.uint8, "wq"),
                                  _dev(sw, torch.float32, "sw"), _dev(offsets, torch.int32, "offsets"), G, T,
                                  N, K, _bf16_ptr(y, "y"), _rows_stride(y, "y"), _stream(stream)),
           "fp8bs_grouped_gemm")
    return y


def fp8bs_grouped_gemm_swiglu(xq: torch.Tensor, sx: torch.Tensor, w1q: torch.Tensor, sw1: torch.Tensor,
                              w3q: torch.Tensor, sw3: torch.Tensor, offsets: torch.Tensor,
                              h: Optional[torch.Tensor] = None, want_h: bool = True, want_fp8: bool = False,
                              hq: Optional[torch.Tensor] = None, sh: Optional[torch.Tensor] = None, stream=None):
    """h [T, I] bf16 = silu(x w1[g]^T) * (x w3[g]^T) per expert (bf16 steps);
    w1q, w3q: [G, I, K] uint8, sw1, sw3: [G, I/128, K/128] fp32.  Returns h
    (want_h and not want_fp8), else (h or None, hq [T, I] uint8, sh [T, I/128])."""
    T, K = xq.shape
    G, I = w1q.shape[0], w1q.shape[1]
    if w3q.shape != w1q.shape or sw3.shape != sw1.shape:
        raise ValueError("w1 and w3 operands must have the same shapes")
    if offsets.dtype != torch.int32 or offsets.numel() != G + 1 or not offsets.is_cuda:
        raise ValueError("offsets must be a CUDA int32 tensor of G + 1 elements")
    if want_h and h is None:
        h = _out_rows(T, I, xq.device)
    if want_fp8:
        if hq is None:
            hq = torch.empty((T, (I + 15) // 16 * 16), dtype=torch.uint8, device=xq.device)[:, :I]
        if sh is None:
            sh = torch.empty((T, max(4, (I // 128 + 3) // 4 * 4)), dtype=torch.float32, device=xq.device)
    _check(lib.fp8bs_grouped_gemm_swiglu(_dev(xq, torch.uint8, "xq"), _dev(sx, torch.float32, "sx"),
                                         _rows_stride(sx, "sx"), _dev(w1q, torch.uint8, "w1q"),
                                         _dev(sw1, torch.float32, "sw1"), _dev(w3q, torch.uint8, "w3q"),
                                         _dev(sw3, torch.float32, "sw3"), offsets.data_ptr(), G, T, I, K,
                                         None if h is None else _bf16_ptr(h, "h"),
                                         0 if h is None else _rows_stride(h, "h"),
                                         None if hq is None else _dev(hq, torch.uint8, "hq"),
                                         0 if hq is None else _rows_stride(hq, "hq"),
                                         None if sh is None else _dev(sh, torch.float32, "sh"),
                                         0 if sh is None else _rows_stride(sh, "sh"), _stream(stream)),
           "fp8bs_grouped_gemm_swiglu")
    if not want_fp8:
        return h
    return h, hq, sh[:, :I // 128]


def fp8bs_moe_dispatch(xq: torch.Tensor, sx: torch.Tensor, token_of_row: torch.Tensor, K: Optional[int] = None,
                       xq_rows: Optional[torch.Tensor] = None, sx_rows: Optional[torch.Tensor] = None,
                       stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Gather quantised token rows into routed order: xq [tokens, K] uint8,
    sx [tokens, lds] fp32, token_of_row int32 [R] on the device ->
    (xq_rows [R, K] uint8, sx_rows [R, lds'] fp32)."""
    tokens = xq.shape[0]
    K = xq.shape[1] if K is None else K
    if token_of_row.dtype != torch.int32 or token_of_row.dim() != 1 or not token_of_row.is_contiguous():
        raise ValueError("token_of_row must be a contiguous 1-D int32 tensor")
    R = token_of_row.numel()
    if xq_rows is None:
        xq_rows = torch.empty((R, (K + 15) // 16 * 16), dtype=torch.uint8, device=xq.device)[:, :K]
    if sx_rows is None:
        sx_rows = torch.empty((R, max(4, (K // 128 + 3) // 4 * 4)), dtype=torch.float32, device=xq.device)
    _check(lib.fp8bs_moe_dispatch(_dev(xq, torch.uint8, "xq"), _rows_stride(xq, "xq"),
                                  _dev(sx, torch.float32, "sx"), _rows_stride(sx, "sx"), tokens, K,
                                  _dev(token_of_row, torch.int32, "token_of_row"), R,
                                  _dev(xq_rows, torch.uint8, "xq_rows"), _rows_stride(xq_rows, "xq_rows"),
                                  _dev(sx_rows, torch.float32, "sx_rows"), _rows_stride(sx_rows, "sx_rows"),
                                  _stream(stream)), "fp8bs_moe_dispatch")
    return xq_rows, sx_rows


def fp8bs_moe_combine(yk: torch.Tensor, weight_of_row: torch.Tensor, rows_of_token: torch.Tensor,
                      z: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """y [tokens, dim] bf16 = z + sum_k weight_of_row[r_k] * yk[r_k] (fp32,
    k in order), r_k = rows_of_token[t, k]; yk [R, dim] bf16, weight_of_row
    fp32 [R], rows_of_token int32 [tokens, topk], z bf16 [tokens, dim] or
    None.  y may be z itself (in-place add)."""
    R, dim = yk.shape
    if rows_of_token.dtype != torch.int32 or rows_of_token.dim() != 2 or not rows_of_token.is_contiguous():
        raise ValueError("rows_of_token must be a contiguous 2-D int32 tensor")
    if weight_of_row.numel() != R or not weight_of_row.is_contiguous():
        raise ValueError("weight_of_row must be a contiguous tensor of R elements")
    tokens, topk = rows_of_token.shape
    if y is None:
        y = _out_rows(tokens, dim, yk.device)
    _check(lib.fp8bs_moe_combine(_bf16_ptr(yk, "yk"), _rows_stride(yk, "yk"), R,
                                 _dev(weight_of_row, torch.float32, "weight_of_row"),
                                 _dev(rows_of_token, torch.int32, "rows_of_token"), tokens, topk, dim,
                                 None if z is None else _bf16_ptr(z, "z"), 0 if z is None else _rows_stride(z, "z"),
                                 _bf16_ptr(y, "y"), _rows_stride(y, "y"), _stream(stream)), "fp8bs_moe_combine")
    return y


def fp8bs_moe_gate(x: torch.Tensor, wg: torch.Tensor, bias: Optional[torch.Tensor] = None, n_groups: int = 8,
                   topk_groups: int = 4, top_k: int = 8, route_scale: float = 2.5,
                   ids: Optional[torch.Tensor] = None, weights: Optional[torch.Tensor] = None,
                   stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Router: x [T, dim] bf16, wg [E, dim] bf16, bias fp32 [E] or None ->
    (ids int32 [T, top_k], gate values fp32 [T, top_k])."""
    T, dim = x.shape
    E = wg.shape[0]
    if not wg.is_contiguous() or wg.shape[1] != dim:
        raise ValueError("wg must be a contiguous [E, dim] tensor")
    if bias is not None and (bias.numel() != E or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous tensor of E elements")
    if ids is None:
        ids = torch.empty((T, top_k), dtype=torch.int32, device=x.device)
    if weights is None:
        weights = torch.empty((T, top_k), dtype=torch.float32, device=x.device)
    _check(lib.fp8bs_moe_gate(_bf16_ptr(x, "x"), _rows_stride(x, "x"), _bf16_ptr(wg, "wg"),
                              None if bias is None else _dev(bias, torch.float32, "bias"), T, dim, E, n_groups,
                              topk_groups, top_k, route_scale, _dev(ids, torch.int32, "ids"),
                              _dev(weights, torch.float32, "weights"), _stream(stream)), "fp8bs_moe_gate")
    return ids, weights


def fp8bs_moe_route(ids: torch.Tensor, weights: torch.Tensor, n_experts: int,
                    offsets: Optional[torch.Tensor] = None, token_of_row: Optional[torch.Tensor] = None,
                    rows_of_token: Optional[torch.Tensor] = None, weight_of_row: Optional[torch.Tensor] = None,
                    stream=None):
    """Routing tables from ids / weights [T, top_k]: returns (offsets int32
    [E+1], token_of_row int32 [R], rows_of_token int32 [T, top_k],
    weight_of_row fp32 [R]), R = T * top_k."""
    T, k = ids.shape
    if not ids.is_contiguous() or not weights.is_contiguous() or weights.shape != ids.shape:
        raise ValueError("ids and weights must be contiguous [T, top_k] tensors")
    dev_ = ids.device
    if offsets is None:
        offsets = torch.empty(n_experts + 1, dtype=torch.int32, device=dev_)
    if token_of_row is None:
        token_of_row = torch.empty(T * k, dtype=torch.int32, device=dev_)
    if rows_of_token is None:
        rows_of_token = torch.empty((T, k), dtype=torch.int32, device=dev_)
    if weight_of_row is None:
        weight_of_row = torch.empty(T * k, dtype=torch.float32, device=dev_)
    _check(lib.fp8bs_moe_route(_dev(ids, torch.int32, "ids"), _dev(weights, torch.float32, "weights"), T, k,
                               n_experts, _dev(offsets, torch.int32, "offsets"),
                               _dev(token_of_row, torch.int32, "token_of_row"),
                               _dev(rows_of_token, torch.int32, "rows_of_token"),
                               _dev(weight_of_row, torch.float32, "weight_of_row"), _stream(stream)),
           "fp8bs_moe_route")
    return offsets, token_of_row, rows_of_token, weight_of_row


def fp8bs_sync_status(stream=None) -> int:
    """Synchronise and return (not raise) the library status."""
    return lib.fp8bs_sync_status(_stream(stream))


def fp8bs_e4m3_encode_f32(v: torch.Tensor, q: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    if q is None:
        q = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check(lib.fp8bs_e4m3_encode_f32(_dev(v, torch.float32, "v"), v.numel(), _dev(q, torch.uint8, "q"),
                                     _stream(stream)), "fp8bs_e4m3_encode_f32")
    return q


def fp8bs_debug_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(lib.fp8bs_debug_wait_timeout(timeout_ns, _stream(stream)), "fp8bs_debug_wait_timeout")
