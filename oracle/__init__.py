"""CPU oracle for the FP8 (e4m3) block-scaled linear layer.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product package (``fp8_block_scaled_18_b300``) never imports it, and the two
share no code: the oracle is the plain C in ``oracle.c`` (see its header for
the passages each function follows), wrapped here with numpy arrays.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np

from . import build as _build

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_lock = threading.Lock()
_libs: dict[tuple[int, bool], ctypes.CDLL] = {}


def load(mutant: int = 0, omp: bool = False) -> ctypes.CDLL:
    """Build (if needed) and load the oracle library; mutant>0 loads a copy
    with a deliberately planted mistake (used only by the mutant tests);
    omp=True loads the same source built with OpenMP (the GEMM's rows spread
    over the host cores; used by the full-size parity tests)."""
    with _lock:
        if (mutant, omp) in _libs:
            return _libs[(mutant, omp)]
        lib = ctypes.CDLL(_build.build(mutant, omp=omp))
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode_search.restype = ctypes.c_uint8
        lib.orc_e4m3_encode_search.argtypes = [ctypes.c_float]
        lib.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
        lib.orc_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        for name, args in {
            "orc_e4m3_encode_array": [_P, _I64, _P],
            "orc_e4m3_encode_search_array": [_P, _I64, _P],
            "orc_act_quant": [_P, _I64, _I64, _I64, _P, _I64, _P, _I64],
            "orc_weight_quant": [_P, _I64, _I64, _P, _P],
            "orc_weight_dequant": [_P, _P, _I64, _I64, _P],
            "orc_gemm_rows": [_P, _I64, _P, _I64, _P, _P, _I64, _I64, _P, _I64, _P, _P],
            "orc_add_bias_rows": [_P, _I64, _I64, _P],
            "orc_swiglu": [_P, _P, _I64, _P],
            "orc_grouped_gemm_rows": [_P, _I64, _P, _I64, _P, _P, _P, ctypes.c_int32,
                                      _I64, _I64, _P, _I64, _P, _P],
            "orc_moe_dispatch": [_P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P, _P],
            "orc_moe_combine": [_P, _I64, _I64, _P, _P, _I64, ctypes.c_int32, _I64, _P, _I64, _P, _P],
            "orc_moe_gate": [_P, _P, _P, _I64, _I64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                             ctypes.c_int32, ctypes.c_double, _P, _P, _P],
            "orc_moe_route": [_P, _P, _I64, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P],
            "orc_act_quant_cols": [_P, _I64, _I64, _I64, _P, _I64, _P],
            "orc_act_quant_pow2": [_P, _I64, _I64, _I64, _P, _I64, _P, _I64],
            "orc_weight_quant_pow2": [_P, _I64, _I64, _P, _P],
            "orc_gemm_dgrad_rows": [_P, _I64, _P, _I64, _P, _P, _I64, _I64, _P, _I64, _P, _P],
            "orc_gemm_wgrad": [_P, _I64, _P, _P, _I64, _P, _I64, _I64, _I64, _P, _P],
            "orc_gemm_wgrad_rows": [_P, _I64, _P, _P, _I64, _P, _I64, _I64, _I64, _P, _I64, _P, _P],
        }.items():
            fn = getattr(lib, name)
            fn.restype = None
            fn.argtypes = args
        lib.orc_mutant_id.restype = ctypes.c_int
        _libs[(mutant, omp)] = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class Oracle:
    """numpy front end of one oracle build (mutant=0 is the real one)."""

    def __init__(self, mutant: int = 0, threads: bool = False):
        self.lib = load(mutant, omp=threads)
        self.mutant = mutant

    # -- codec -----------------------------------------------------------
    def e4m3_decode(self, codes) -> np.ndarray:
        codes = np.asarray(codes, dtype=np.uint8)
        return np.array([self.lib.orc_e4m3_decode(int(c)) for c in codes.ravel()],
                        dtype=np.float64).reshape(codes.shape)

    def e4m3_encode(self, v) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float32)
        out = np.empty(v.shape, dtype=np.uint8)
        self.lib.orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
        return out

    def e4m3_encode_search(self, v) -> np.ndarray:
        v = np.ascontiguousarray(v, dtype=np.float32)
        out = np.empty(v.shape, dtype=np.uint8)
        self.lib.orc_e4m3_encode_search_array(_ptr(v), v.size, _ptr(out))
        return out

    def bf16_rne(self, v) -> np.ndarray:
        v = np.asarray(v, dtype=np.float32)
        return np.array([self.lib.orc_f32_to_bf16_rne(float(x)) for x in v.ravel()],
                        dtype=np.uint16).reshape(v.shape)

    # -- quantisers --------------------------------------------------------
    def act_quant(self, x_bits: np.ndarray, lds: int | None = None):
        """x_bits: uint16 bf16 bit patterns [M, K].  Returns (xq [M,K] u8,
        sx [M, lds] f32); padding columns of sx (>= K/128) are left 0."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = x_bits.shape
        kb = K // 128
        lds = kb if lds is None else lds
        xq = np.zeros((M, K), dtype=np.uint8)
        sx = np.zeros((M, lds), dtype=np.float32)
        self.lib.orc_act_quant(_ptr(x_bits), M, K, K, _ptr(xq), K, _ptr(sx), lds)
        return xq, sx

    def weight_quant(self, w_bits: np.ndarray):
        w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
        N, K = w_bits.shape
        wq = np.zeros((N, K), dtype=np.uint8)
        sw = np.zeros(((N + 127) // 128, K // 128), dtype=np.float32)
        self.lib.orc_weight_quant(_ptr(w_bits), N, K, _ptr(wq), _ptr(sw))
        return wq, sw

    def weight_dequant(self, wq: np.ndarray, sw: np.ndarray) -> np.ndarray:
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        N, K = wq.shape
        assert sw.shape == ((N + 127) // 128, K // 128)
        w = np.zeros((N, K), dtype=np.uint16)
        self.lib.orc_weight_dequant(_ptr(wq), _ptr(sw), N, K, _ptr(w))
        return w

    # -- gemm --------------------------------------------------------------
    def gemm(self, xq, sx, wq, sw, rows=None, bias=None):
        """Returns (y_ref fp64 [len(rows), N], L fp64 [len(rows), N]); with
        bias (bf16 bits [N]) y_ref includes y += bias."""
        xq = np.ascontiguousarray(xq, dtype=np.uint8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, K = xq.shape
        N = wq.shape[0]
        assert wq.shape[1] == K and sw.shape == ((N + 127) // 128, K // 128)
        assert sx.shape[0] == M and sx.shape[1] >= K // 128
        rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        y = np.zeros((rows.size, N), dtype=np.float64)
        L = np.zeros((rows.size, N), dtype=np.float64)
        self.lib.orc_gemm_rows(_ptr(xq), K, _ptr(sx), sx.shape[1], _ptr(wq), _ptr(sw),
                               N, K, _ptr(rows), rows.size, _ptr(y), _ptr(L))
        if bias is not None:
            b = np.ascontiguousarray(bias, dtype=np.uint16)
            assert b.shape == (N,)
            self.lib.orc_add_bias_rows(_ptr(y), rows.size, N, _ptr(b))
        return y, L

    def swiglu(self, a, b):
        """h = silu(a) * b, elementwise, fp64."""
        return _swiglu(self.lib, a, b)

    def grouped_swiglu(self, xq, sx, w1q, sw1, w3q, sw3, offsets, rows=None):
        """The expert first stage: returns (h, a, b, La, Lb), a and b the
        grouped GEMMs with w1 and w3, h = silu(a) * b (all fp64)."""
        a, La = self.grouped_gemm(xq, sx, w1q, sw1, offsets, rows=rows)
        b, Lb = self.grouped_gemm(xq, sx, w3q, sw3, offsets, rows=rows)
        return self.swiglu(a, b), a, b, La, Lb

    def grouped_gemm(self, xq, sx, wq, sw, offsets, rows=None):
        """wq: [G, N, K] u8, sw: [G, ceil(N/128), K/128], offsets int32 [G+1]."""
        xq = np.ascontiguousarray(xq, dtype=np.uint8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        offsets = np.ascontiguousarray(offsets, dtype=np.int32)
        T, K = xq.shape
        G, N, _ = wq.shape
        assert sw.shape == (G, (N + 127) // 128, K // 128) and offsets.size == G + 1
        rows = np.arange(T, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        y = np.zeros((rows.size, N), dtype=np.float64)
        L = np.zeros((rows.size, N), dtype=np.float64)
        self.lib.orc_grouped_gemm_rows(_ptr(xq), K, _ptr(sx), sx.shape[1], _ptr(wq), _ptr(sw),
                                       _ptr(offsets), G, N, K, _ptr(rows), rows.size,
                                       _ptr(y), _ptr(L))
        return y, L


    def moe_dispatch(self, xq, sx, token_of_row):
        """Gather quantised token rows into routed order: returns
        (xr [R, K] u8, sr [R, K/128] fp32); rows of out-of-range ids are 0."""
        xq = np.ascontiguousarray(xq, dtype=np.uint8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        tor = np.ascontiguousarray(token_of_row, dtype=np.int32)
        tokens, K = xq.shape
        R = tor.size
        xr = np.empty((R, K), dtype=np.uint8)
        sr = np.empty((R, K // 128), dtype=np.float32)
        self.lib.orc_moe_dispatch(_ptr(xq), K, _ptr(sx), sx.shape[1], tokens, K, _ptr(tor), R,
                                  _ptr(xr), _ptr(sr))
        return xr, sr

    def moe_combine(self, yk, weight_of_row, rows_of_token, z=None):
        """y [tokens, dim] = z + sum_k w[r_k] yk[r_k] (fp64) and its magnitude
        sum L; yk [R, dim] (any real dtype, widened to fp64 exactly),
        weight_of_row fp32 [R], rows_of_token int32 [tokens, topk]."""
        yk = np.ascontiguousarray(yk, dtype=np.float64)
        w = np.ascontiguousarray(weight_of_row, dtype=np.float32)
        rt = np.ascontiguousarray(rows_of_token, dtype=np.int32)
        R, dim = yk.shape
        tokens, topk = rt.shape
        assert w.size == R
        y = np.empty((tokens, dim), dtype=np.float64)
        L = np.empty((tokens, dim), dtype=np.float64)
        zp = None
        if z is not None:
            z = np.ascontiguousarray(z, dtype=np.float64)
            assert z.shape == (tokens, dim)
            zp = _ptr(z)
        self.lib.orc_moe_combine(_ptr(yk), dim, R, _ptr(w), _ptr(rt), tokens, topk, dim, zp, dim,
                                 _ptr(y), _ptr(L))
        return y, L


    def moe_gate(self, x_bits, wg_bits, bias, n_groups=8, topk_groups=4, top_k=8, route_scale=2.5,
                 want_scores=False):
        """Router in fp64: returns (ids int32 [T, top_k] in descending biased
        score, gate values fp64 [T, top_k]) and, if asked, the affinities
        [T, E]."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        wg = np.ascontiguousarray(wg_bits, dtype=np.uint16)
        b = np.ascontiguousarray(bias, dtype=np.float32)
        T, dim = x.shape
        E = wg.shape[0]
        assert wg.shape[1] == dim and b.size == E and E % n_groups == 0
        ids = np.empty((T, top_k), dtype=np.int32)
        w = np.empty((T, top_k), dtype=np.float64)
        s = np.empty((T, E), dtype=np.float64) if want_scores else None
        self.lib.orc_moe_gate(_ptr(x), _ptr(wg), _ptr(b), T, dim, E, n_groups, topk_groups, top_k,
                              float(route_scale), _ptr(ids), _ptr(w), None if s is None else _ptr(s))
        return (ids, w, s) if want_scores else (ids, w)

    def moe_route(self, ids, w, n_experts):
        """Stable counting sort of the selections by expert: returns
        (offsets [E+1], token_of_row [R], rows_of_token [T, k], weight_of_row [R])."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        w = np.ascontiguousarray(w, dtype=np.float32)
        T, k = ids.shape
        off = np.empty(n_experts + 1, dtype=np.int32)
        tor = np.empty(T * k, dtype=np.int32)
        rot = np.empty((T, k), dtype=np.int32)
        wor = np.empty(T * k, dtype=np.float32)
        self.lib.orc_moe_route(_ptr(ids), _ptr(w), T, k, n_experts, _ptr(off), _ptr(tor), _ptr(rot), _ptr(wor))
        return off, tor, rot, wor


    def act_quant_pow2(self, x_bits, lds: int | None = None):
        """act_quant with power-of-two (UE8M0-style) scales, rounded up."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = x.shape
        lds = lds or max(1, K // 128)
        xq = np.empty((M, K), dtype=np.uint8)
        sx = np.zeros((M, lds), dtype=np.float32)
        self.lib.orc_act_quant_pow2(_ptr(x), M, K, K, _ptr(xq), K, _ptr(sx), lds)
        return xq, sx

    def weight_quant_pow2(self, w_bits):
        """weight_quant with power-of-two (UE8M0-style) scales, rounded up."""
        w = np.ascontiguousarray(w_bits, dtype=np.uint16)
        N, K = w.shape
        wq = np.zeros((N, K), dtype=np.uint8)
        sw = np.zeros(((N + 127) // 128, K // 128), dtype=np.float32)
        self.lib.orc_weight_quant_pow2(_ptr(w), N, K, _ptr(wq), _ptr(sw))
        return wq, sw

    def act_quant_cols(self, x_bits):
        """x [M, K] bf16 bits -> (xq [M, K] u8, sx [ceil(M/128), K] fp32):
        128x1 groups along the rows (the wgrad operands' quantisation)."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = x.shape
        xq = np.empty((M, K), dtype=np.uint8)
        sx = np.empty(((M + 127) // 128, K), dtype=np.float32)
        self.lib.orc_act_quant_cols(_ptr(x), M, K, K, _ptr(xq), K, _ptr(sx))
        return xq, sx

    def gemm_dgrad(self, dyq, sdy, wq, sw, rows=None):
        """dX = dY W from dyq [M, N] (1x128 groups, sdy [M, >= N/128]) and the
        forward's wq [N, K], sw [ceil(N/128), K/128]: (dx, L) fp64 [rows, K]."""
        dyq = np.ascontiguousarray(dyq, dtype=np.uint8)
        sdy = np.ascontiguousarray(sdy, dtype=np.float32)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, N = dyq.shape
        N2, K = wq.shape
        assert N2 == N and N % 128 == 0 and sw.shape == (N // 128, K // 128)
        rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        dx = np.empty((rows.size, K), dtype=np.float64)
        L = np.empty((rows.size, K), dtype=np.float64)
        self.lib.orc_gemm_dgrad_rows(_ptr(dyq), N, _ptr(sdy), sdy.shape[1], _ptr(wq), _ptr(sw), N, K, _ptr(rows),
                                     rows.size, _ptr(dx), _ptr(L))
        return dx, L

    def gemm_wgrad(self, dyq, sdy, xq, sx, rows=None):
        """dW = dY^T X from 128x1-grouped dyq [M, N] / sdy and xq [M, K] / sx
        (act_quant_cols): (dw, L) fp64 [N, K], or [len(rows), K] for the
        listed rows n of dW."""
        dyq = np.ascontiguousarray(dyq, dtype=np.uint8)
        sdy = np.ascontiguousarray(sdy, dtype=np.float32)
        xq = np.ascontiguousarray(xq, dtype=np.uint8)
        sx = np.ascontiguousarray(sx, dtype=np.float32)
        M, N = dyq.shape
        M2, K = xq.shape
        MB = (M + 127) // 128
        assert M2 == M and sdy.shape == (MB, N) and sx.shape == (MB, K)
        if rows is None:
            dw = np.empty((N, K), dtype=np.float64)
            L = np.empty((N, K), dtype=np.float64)
            self.lib.orc_gemm_wgrad(_ptr(dyq), N, _ptr(sdy), _ptr(xq), K, _ptr(sx), M, N, K, _ptr(dw), _ptr(L))
            return dw, L
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        dw = np.empty((rows.size, K), dtype=np.float64)
        L = np.empty((rows.size, K), dtype=np.float64)
        self.lib.orc_gemm_wgrad_rows(_ptr(dyq), N, _ptr(sdy), _ptr(xq), K, _ptr(sx), M, N, K, _ptr(rows), rows.size,
                                     _ptr(dw), _ptr(L))
        return dw, L


def _swiglu(lib, a, b):
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    h = np.empty_like(a)
    lib.orc_swiglu(_ptr(a), _ptr(b), a.size, _ptr(h))
    return h


def gemm_tolerance(y_ref: np.ndarray, L: np.ndarray) -> np.ndarray:
    """Per-element GEMM acceptance bound: 2^-8 |y_ref| + 1e-4 L."""
    return np.ldexp(np.abs(y_ref), -8) + 1e-4 * L
