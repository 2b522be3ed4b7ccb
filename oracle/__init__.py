"""ctypes wrapper over the plain-C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and the benchmark's CPU-baseline leg
import this module. The CUDA library and its Python binding never do.

Every GEMV here returns ``(y, bound)`` as float64 arrays, where ``bound[i] = sum_k |W[n][k]| * |xhat[k]|``
sets the scale of the comparison tolerance ``|y_gpu - y| <= 1e-3 * bound + 1e-5``.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def _p(a: np.ndarray, ptype):
    return a.ctypes.data_as(ptype)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """One loaded copy of the oracle library (a path lets tests load a deliberately altered build)."""

    def __init__(self, lib_path: str | None = None):
        if lib_path is None:
            if _build.is_stale():
                _build.build()
            lib_path = _build.LIB_PATH
        self.path = lib_path
        L = ctypes.CDLL(lib_path)
        L.oracle_f16_to_f32.restype = ctypes.c_float
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_dequant_q4.argtypes = [_u8p, _u16p, _i64, _i64, _f32p]
        L.oracle_dequant_q4k.argtypes = [_u8p, _i64, _i64, _f32p]
        L.oracle_q4k_scale_min.argtypes = [_u8p, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_int)]
        L.oracle_q4_gemv_batched.argtypes = [_u8p, _u16p, _f32p, _i64, _i64, _i64, _f64p, _f64p]
        L.oracle_rmsnorm.argtypes = [_f32p, _f32p, ctypes.c_float, _i64, _f64p]
        L.oracle_q4k_gemv.argtypes = [_u8p, _f64p, _i64, _i64, _f64p, _f64p]
        L.oracle_fused_rmsnorm_q4k_gemv.argtypes = [_u8p, _f32p, _f32p, ctypes.c_float, _i64, _i64,
                                                    _f64p, _f64p]
        L.oracle_fused_gateup_q4k_gemv.argtypes = [_u8p, _u8p, _f32p, _f32p, ctypes.c_float, _i64, _i64,
                                                   _f64p, _f64p, _f64p, _f64p]
        L.oracle_moe_q4_gemv.argtypes = [_u8p, _u16p, _u8p, _u16p, _f32p, _i32p, _i64, _i64, _i64, _i64,
                                         _i64, _f64p, _f64p, _f64p, _f64p]
        L.oracle_silu.restype = ctypes.c_double
        L.oracle_silu.argtypes = [ctypes.c_double]
        L.oracle_swiglu.argtypes = [_f64p, _f64p, _i64, _f64p]
        L.oracle_topk_softmax_f32.argtypes = [_f32p, _i64, _i64, _i64, ctypes.c_int, _i32p, _f64p]
        L.oracle_moe_router.argtypes = [_u8p, _u16p, _f32p, _i64, _i64, _i64, _i64, ctypes.c_int, _f64p, _f64p,
                                        _i32p, _f64p]
        self.L = L

    # -- element decode ------------------------------------------------------------------------
    def f16_to_f32(self, bits: int) -> float:
        return float(self.L.oracle_f16_to_f32(int(bits) & 0xFFFF))

    def q4k_scale_min(self, s12, j: int):
        s = _c(np.asarray(s12), np.uint8)
        assert s.size == 12
        sc, m = ctypes.c_int(), ctypes.c_int()
        self.L.oracle_q4k_scale_min(_p(s, _u8p), int(j), ctypes.byref(sc), ctypes.byref(m))
        return sc.value, m.value

    def dequant_q4(self, qs, d) -> np.ndarray:
        qs = _c(qs, np.uint8)
        d = _c(np.asarray(d, dtype=np.float16).view(np.uint16), np.uint16)
        N, nblk = d.shape
        K = nblk * 32
        assert qs.size == N * K // 2
        W = np.empty((N, K), np.float32)
        self.L.oracle_dequant_q4(_p(qs, _u8p), _p(d, _u16p), N, K, _p(W, _f32p))
        return W

    def dequant_q4k(self, w) -> np.ndarray:
        w = _c(w, np.uint8)
        N, nsb = w.shape[0], w.shape[1]
        K = nsb * 256
        W = np.empty((N, K), np.float32)
        self.L.oracle_dequant_q4k(_p(w, _u8p), N, K, _p(W, _f32p))
        return W

    # -- GEMVs ---------------------------------------------------------------------------------
    def q4_gemv_batched(self, qs, d, X):
        qs = _c(qs, np.uint8)
        d = _c(np.asarray(d, dtype=np.float16).view(np.uint16), np.uint16)
        X = _c(np.atleast_2d(X), np.float32)
        N, nblk = d.shape
        K = nblk * 32
        M = X.shape[0]
        assert X.shape[1] == K
        Y = np.empty((M, N), np.float64)
        B = np.empty((M, N), np.float64)
        rc = self.L.oracle_q4_gemv_batched(_p(qs, _u8p), _p(d, _u16p), _p(X, _f32p), M, N, K,
                                           _p(Y, _f64p), _p(B, _f64p))
        assert rc == 0
        return Y, B

    def q4_gemv(self, qs, d, x):
        Y, B = self.q4_gemv_batched(qs, d, np.asarray(x).reshape(1, -1))
        return Y[0], B[0]

    def rmsnorm(self, x, gamma, eps) -> np.ndarray:
        x = _c(x, np.float32)
        g = _c(gamma, np.float32)
        out = np.empty(x.size, np.float64)
        self.L.oracle_rmsnorm(_p(x, _f32p), _p(g, _f32p), float(eps), x.size, _p(out, _f64p))
        return out

    def q4k_gemv(self, w, xhat):
        w = _c(w, np.uint8)
        xh = _c(xhat, np.float64)
        N, K = w.shape[0], w.shape[1] * 256
        y = np.empty(N, np.float64)
        b = np.empty(N, np.float64)
        assert self.L.oracle_q4k_gemv(_p(w, _u8p), _p(xh, _f64p), N, K, _p(y, _f64p), _p(b, _f64p)) == 0
        return y, b

    def fused_rmsnorm_q4k_gemv(self, w, x, gamma, eps):
        w = _c(w, np.uint8)
        x = _c(x, np.float32)
        g = _c(gamma, np.float32)
        N, K = w.shape[0], w.shape[1] * 256
        y = np.empty(N, np.float64)
        b = np.empty(N, np.float64)
        rc = self.L.oracle_fused_rmsnorm_q4k_gemv(_p(w, _u8p), _p(x, _f32p), _p(g, _f32p), float(eps), N, K,
                                                  _p(y, _f64p), _p(b, _f64p))
        assert rc == 0
        return y, b

    def fused_gateup_q4k_gemv(self, w_gate, w_up, x, gamma, eps):
        wg = _c(w_gate, np.uint8)
        wu = _c(w_up, np.uint8)
        x = _c(x, np.float32)
        N, K = wg.shape[0], wg.shape[1] * 256
        gp = None
        if gamma is not None:
            g = _c(gamma, np.float32)
            gp = _p(g, _f32p)
        yg = np.empty(N, np.float64)
        yu = np.empty(N, np.float64)
        bg = np.empty(N, np.float64)
        bu = np.empty(N, np.float64)
        rc = self.L.oracle_fused_gateup_q4k_gemv(_p(wg, _u8p), _p(wu, _u8p), _p(x, _f32p), gp, float(eps), N,
                                                 K, _p(yg, _f64p), _p(yu, _f64p), _p(bg, _f64p), _p(bu, _f64p))
        assert rc == 0
        return (yg, bg), (yu, bu)

    def moe_q4_gemv(self, qs_gate, d_gate, qs_up, d_up, x, ids, E):
        qg = _c(qs_gate, np.uint8)
        qu = _c(qs_up, np.uint8)
        dg = _c(np.asarray(d_gate, dtype=np.float16).view(np.uint16), np.uint16)
        du = _c(np.asarray(d_up, dtype=np.float16).view(np.uint16), np.uint16)
        x = _c(np.atleast_2d(x), np.float32)
        ids = _c(np.atleast_2d(ids), np.int32)
        T, topk = ids.shape
        rows, nblk = dg.shape
        K = nblk * 32
        assert rows % E == 0 and x.shape == (T, K)
        N = rows // E
        shape = (T, topk, N)
        yg, yu, bg, bu = (np.empty(shape, np.float64) for _ in range(4))
        rc = self.L.oracle_moe_q4_gemv(_p(qg, _u8p), _p(dg, _u16p), _p(qu, _u8p), _p(du, _u16p), _p(x, _f32p),
                                       _p(ids, _i32p), T, topk, E, N, K, _p(yg, _f64p), _p(yu, _f64p),
                                       _p(bg, _f64p), _p(bu, _f64p))
        assert rc == 0
        return (yg, bg), (yu, bu)


    # -- epilogue and router ---------------------------------------------------------------------
    def silu(self, g: float) -> float:
        return float(self.L.oracle_silu(float(g)))

    def swiglu(self, g, u) -> np.ndarray:
        g = _c(g, np.float64)
        u = _c(u, np.float64)
        assert g.shape == u.shape
        y = np.empty(g.shape, np.float64)
        self.L.oracle_swiglu(_p(g, _f64p), _p(u, _f64p), g.size, _p(y, _f64p))
        return y

    def topk_softmax_f32(self, logits, topk: int, normalize: bool):
        lg = _c(np.atleast_2d(logits), np.float32)
        T, E = lg.shape
        ids = np.empty((T, topk), np.int32)
        w = np.empty((T, topk), np.float64)
        self.L.oracle_topk_softmax_f32(_p(lg, _f32p), T, E, topk, 1 if normalize else 0, _p(ids, _i32p), _p(w, _f64p))
        return ids, w

    def moe_router(self, qs, d, x, topk: int, normalize: bool):
        """(logits [T][E], bounds [T][E], ids [T][topk], weights [T][topk]) for planar-Q4 router rows."""
        qs = _c(qs, np.uint8)
        d = _c(np.asarray(d, dtype=np.float16).view(np.uint16), np.uint16)
        x = _c(np.atleast_2d(x), np.float32)
        E, nblk = d.shape
        K = nblk * 32
        T = x.shape[0]
        assert x.shape == (T, K)
        lg = np.empty((T, E), np.float64)
        bd = np.empty((T, E), np.float64)
        ids = np.empty((T, topk), np.int32)
        w = np.empty((T, topk), np.float64)
        rc = self.L.oracle_moe_router(_p(qs, _u8p), _p(d, _u16p), _p(x, _f32p), T, E, K, topk, 1 if normalize else 0,
                                      _p(lg, _f64p), _p(bd, _f64p), _p(ids, _i32p), _p(w, _f64p))
        assert rc == 0
        return lg, bd, ids, w


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
