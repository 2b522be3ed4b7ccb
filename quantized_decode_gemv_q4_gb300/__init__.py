"""GB300 4-bit decode GEMVs: a thin Python binding over the C ABI in ``include/q4gemv.h``.

Each function has the name of its C entry point and takes CUDA tensors (PyTorch is used only for
device memory and streams). Shapes give the sizes; the call is enqueued on the given stream (default:
the current stream) and returns at once. A refusal or a CUDA failure raises :class:`Q4Error` with the
library's message. There is no CPU path: without the compiled library every call raises.

Layouts (row-major, little-endian):
  * Q4 planar: ``qs`` uint8 ``[N, K/32, 16]`` (or ``[N, K/2]``), ``d`` float16 ``[N, K/32]``.
  * Q4_K: ``w`` uint8 ``[N, K/256, 144]`` (or ``[N, K/256*144]``).
  * inputs and outputs float32.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "Q4Error", "load", "q4_fma_ceiling", "q4_gemv", "q4_gemv_batched", "fused_rmsnorm_q4k_gemv", "fused_gateup_q4k_gemv",
    "moe_q4_gemv", "q4k_gemv_batched", "fused_gateup_swiglu_q4k_gemv", "moe_q4_swiglu_gemv", "moe_router_q4", "q4_pure_read",
    "q4k_pure_read",
    "moe_q4_pure_read", "q4_dequant", "q4k_dequant",
    "q4_device_faults", "q4_set_launch_overlap", "q4_get_launch_overlap", "q4_set_wait_limit", "q4_get_wait_limit",
    "FAULT_BAD_EXPERT", "FAULT_WAIT_TIMEOUT", "FAULT_COPY_LOST", "DEFAULT_WAIT_LIMIT",
]

Q4_OK, Q4_EINVAL, Q4_EALIGN, Q4_ECUDA, Q4_EUNSUPPORTED = 0, -1, -2, -3, -4
FAULT_BAD_EXPERT = 4
FAULT_WAIT_TIMEOUT = 8
FAULT_COPY_LOST = 16
DEFAULT_WAIT_LIMIT = 4_000_000_000
_CODE_NAMES = {Q4_EINVAL: "EINVAL", Q4_EALIGN: "EALIGN", Q4_ECUDA: "ECUDA", Q4_EUNSUPPORTED: "EUNSUPPORTED"}


class Q4Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{_CODE_NAMES.get(code, code)}: {message}")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int

_SIGNATURES = {
    "q4_gemv": [_P, _P, _P, _P, _I, _I, _P],
    "q4_gemv_batched": [_P, _P, _P, _P, _I, _I, _I, _P],
    "fused_rmsnorm_q4k_gemv": [_P, _P, _P, _P, ctypes.c_float, _I, _I, _P],
    "fused_gateup_q4k_gemv": [_P, _P, _P, _P, _P, _P, ctypes.c_float, _I, _I, _P],
    "moe_q4_gemv": [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P],
    "q4_pure_read": [_P, _P, _P, _I, _I, _P],
    "q4k_pure_read": [_P, _P, _I, _I, _P],
    "moe_q4_pure_read": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P],
    "q4_dequant": [_P, _P, _P, _I, _I, _P],
    "q4k_dequant": [_P, _P, _I, _I, _P],
    "fused_gateup_swiglu_q4k_gemv": [_P, _P, _P, _P, _P, ctypes.c_float, _I, _I, _P],
    "moe_q4_swiglu_gemv": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P],
    "moe_router_q4": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P],
    "q4k_gemv_batched": [_P, _P, _P, _I, _I, _I, _P],
    "q4_device_faults": [ctypes.POINTER(ctypes.c_uint)],
    "q4_fma_ceiling": [_P, _I, ctypes.c_longlong, ctypes.c_float, ctypes.c_float, ctypes.POINTER(ctypes.c_longlong),
                       _P],
}


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (once) the compiled library; raise if it was never built."""
    global _lib
    if _lib is None:
        p = path or lib_path()
        if not os.path.exists(p):
            raise RuntimeError(f"libq4gemv is not built ({p} missing): run quantized_decode_gemv_q4_gb300/build.py")
        L = ctypes.CDLL(p)
        for name, args in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.q4_last_error.argtypes = []
        L.q4_last_error.restype = ctypes.c_char_p
        L.q4_set_launch_overlap.argtypes = [ctypes.c_int]
        L.q4_set_launch_overlap.restype = ctypes.c_int
        L.q4_get_launch_overlap.argtypes = []
        L.q4_get_launch_overlap.restype = ctypes.c_int
        L.q4_set_wait_limit.argtypes = [ctypes.c_longlong]
        L.q4_set_wait_limit.restype = ctypes.c_int
        L.q4_get_wait_limit.argtypes = []
        L.q4_get_wait_limit.restype = ctypes.c_longlong
        _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != Q4_OK:
        raise Q4Error(rc, load().q4_last_error().decode())


def _ptr(t: torch.Tensor | None, dtype: torch.dtype, name: str) -> int | None:
    if t is None:
        return None
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _q4_dims(qs: torch.Tensor, d: torch.Tensor):
    N = d.shape[0]
    K = d.numel() // N * 32
    if qs.numel() != N * K // 2:
        raise ValueError(f"qs holds {qs.numel()} bytes, expected N*K/2 = {N * K // 2}")
    return N, K


def _q4k_dims(w: torch.Tensor):
    N = w.shape[0]
    if (w.numel() // N) % 144:
        raise ValueError("Q4_K rows must be a whole number of 144-byte super-blocks")
    return N, w.numel() // N // 144 * 256


def q4_gemv(y, qs, d, x, stream=None) -> None:
    N, K = _q4_dims(qs, d)
    if x.numel() != K or y.numel() != N:
        raise ValueError("x must hold K values and y N values")
    _check(load().q4_gemv(_ptr(y, torch.float32, "y"), _ptr(qs, torch.uint8, "qs"), _ptr(d, torch.float16, "d"),
                          _ptr(x, torch.float32, "x"), N, K, _stream(stream)))


def q4_gemv_batched(Y, qs, d, X, stream=None) -> None:
    N, K = _q4_dims(qs, d)
    M = X.shape[0] if X.dim() == 2 else 1
    if X.numel() != M * K or Y.numel() != M * N:
        raise ValueError("X must be [M, K] and Y [M, N]")
    _check(load().q4_gemv_batched(_ptr(Y, torch.float32, "Y"), _ptr(qs, torch.uint8, "qs"),
                                  _ptr(d, torch.float16, "d"), _ptr(X, torch.float32, "X"), M, N, K,
                                  _stream(stream)))


def fused_rmsnorm_q4k_gemv(y, w, x, gamma, eps: float = 1e-5, stream=None) -> None:
    N, K = _q4k_dims(w)
    if x.numel() != K or gamma.numel() != K or y.numel() != N:
        raise ValueError("x and gamma must hold K values and y N values")
    _check(load().fused_rmsnorm_q4k_gemv(_ptr(y, torch.float32, "y"), _ptr(w, torch.uint8, "w"),
                                         _ptr(x, torch.float32, "x"), _ptr(gamma, torch.float32, "gamma"),
                                         float(eps), N, K, _stream(stream)))


def q4k_gemv_batched(Y, w, X, stream=None) -> None:
    """Y[m] = W X[m] for the M rows of X (Q4_K weights, no normalisation), one weight sweep."""
    N, K = _q4k_dims(w)
    M = X.numel() // K
    if X.numel() != M * K or Y.numel() != M * N:
        raise ValueError("X must be [M, K] and Y [M, N]")
    _check(load().q4k_gemv_batched(_ptr(Y, torch.float32, "Y"), _ptr(w, torch.uint8, "w"), _ptr(X, torch.float32, "X"),
                                   M, N, K, _stream(stream)))


def fused_gateup_q4k_gemv(y_gate, y_up, w_gate, w_up, x, gamma=None, eps: float = 1e-5, stream=None) -> None:
    N, K = _q4k_dims(w_gate)
    if _q4k_dims(w_up) != (N, K) or x.numel() != K or y_gate.numel() != N or y_up.numel() != N:
        raise ValueError("gate and up must be [N, K/256, 144], x K values, outputs N values")
    if gamma is not None and gamma.numel() != K:
        raise ValueError("gamma must hold K values")
    _check(load().fused_gateup_q4k_gemv(_ptr(y_gate, torch.float32, "y_gate"), _ptr(y_up, torch.float32, "y_up"),
                                        _ptr(w_gate, torch.uint8, "w_gate"), _ptr(w_up, torch.uint8, "w_up"),
                                        _ptr(x, torch.float32, "x"), _ptr(gamma, torch.float32, "gamma"),
                                        float(eps), N, K, _stream(stream)))


def _moe_dims(qs_gate, d_gate, expert_ids, E):
    rows, K = _q4_dims(qs_gate, d_gate)
    if rows % E:
        raise ValueError("the expert stores must hold E*N rows")
    T, topk = expert_ids.shape
    return T, topk, rows // E, K


def moe_q4_gemv(y_gate, y_up, qs_gate, d_gate, qs_up, d_up, x, expert_ids, E: int, dev_status=None,
                stream=None) -> None:
    T, topk, N, K = _moe_dims(qs_gate, d_gate, expert_ids, E)
    if x.numel() != T * K or y_gate.numel() != T * topk * N or y_up.numel() != T * topk * N:
        raise ValueError("x must be [T, K] and outputs [T, topk, N]")
    _check(load().moe_q4_gemv(_ptr(y_gate, torch.float32, "y_gate"), _ptr(y_up, torch.float32, "y_up"),
                              _ptr(qs_gate, torch.uint8, "qs_gate"), _ptr(d_gate, torch.float16, "d_gate"),
                              _ptr(qs_up, torch.uint8, "qs_up"), _ptr(d_up, torch.float16, "d_up"),
                              _ptr(x, torch.float32, "x"), _ptr(expert_ids, torch.int32, "expert_ids"),
                              T, topk, E, N, K, _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def fused_gateup_swiglu_q4k_gemv(y, w_gate, w_up, x, gamma=None, eps: float = 1e-5, stream=None) -> None:
    """y = silu(W_gate xhat) * (W_up xhat), one output (xhat as fused_gateup_q4k_gemv)."""
    N, K = _q4k_dims(w_gate)
    if _q4k_dims(w_up) != (N, K) or x.numel() != K or y.numel() != N:
        raise ValueError("w_gate and w_up must be [N, K/256, 144], x [K], y [N]")
    _check(load().fused_gateup_swiglu_q4k_gemv(_ptr(y, torch.float32, "y"), _ptr(w_gate, torch.uint8, "w_gate"),
                                               _ptr(w_up, torch.uint8, "w_up"), _ptr(x, torch.float32, "x"),
                                               _ptr(gamma, torch.float32, "gamma"), float(eps), N, K, _stream(stream)))


def moe_q4_swiglu_gemv(y, qs_gate, d_gate, qs_up, d_up, x, expert_ids, E: int, dev_status=None, stream=None) -> None:
    """y[t, s] = silu(gate) * up for every routed row (routing as moe_q4_gemv)."""
    T, topk, N, K = _moe_dims(qs_gate, d_gate, expert_ids, E)
    if x.numel() != T * K or y.numel() != T * topk * N:
        raise ValueError("x must be [T, K] and y [T, topk, N]")
    _check(load().moe_q4_swiglu_gemv(_ptr(y, torch.float32, "y"), _ptr(qs_gate, torch.uint8, "qs_gate"),
                                     _ptr(d_gate, torch.float16, "d_gate"), _ptr(qs_up, torch.uint8, "qs_up"),
                                     _ptr(d_up, torch.float16, "d_up"), _ptr(x, torch.float32, "x"),
                                     _ptr(expert_ids, torch.int32, "expert_ids"), T, topk, E, N, K,
                                     _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def moe_router_q4(expert_ids, expert_weights, qs, d, x, topk: int, normalize: bool = True, logits=None,
                  stream=None) -> None:
    """Router logits of E planar-Q4 rows for T tokens, then the top-K experts and their softmax weights."""
    E, K = _q4_dims(qs, d)
    T = x.numel() // K
    if x.numel() != T * K or expert_ids.numel() != T * topk or expert_weights.numel() != T * topk:
        raise ValueError("x must be [T, K], expert_ids and expert_weights [T, topk]")
    if logits is not None and logits.numel() != T * E:
        raise ValueError("logits must be [T, E]")
    _check(load().moe_router_q4(_ptr(expert_ids, torch.int32, "expert_ids"),
                                _ptr(expert_weights, torch.float32, "expert_weights"),
                                _ptr(logits, torch.float32, "logits"), _ptr(qs, torch.uint8, "qs"),
                                _ptr(d, torch.float16, "d"), _ptr(x, torch.float32, "x"), T, E, K, topk,
                                1 if normalize else 0, _stream(stream)))


def q4_pure_read(sink, qs, d, stream=None) -> None:
    N, K = _q4_dims(qs, d)
    _check(load().q4_pure_read(_ptr(sink, torch.float32, "sink"), _ptr(qs, torch.uint8, "qs"),
                               _ptr(d, torch.float16, "d"), N, K, _stream(stream)))


def q4_fma_ceiling(sink, fmas: int, mul: float = 1.0 - 2.0 ** -20, add: float = 2.0 ** -20, stream=None) -> int:
    """Run at least `fmas` fp32 FMAs with no loads (the FMA-ceiling instrument); returns the count run."""
    done = ctypes.c_longlong(0)
    _check(load().q4_fma_ceiling(_ptr(sink, torch.float32, "sink"), sink.numel(), int(fmas), float(mul), float(add),
                                 ctypes.byref(done), _stream(stream)))
    return done.value


def q4k_pure_read(sink, w, stream=None) -> None:
    N, K = _q4k_dims(w)
    _check(load().q4k_pure_read(_ptr(sink, torch.float32, "sink"), _ptr(w, torch.uint8, "w"), N, K,
                                _stream(stream)))


def moe_q4_pure_read(sink_gate, sink_up, qs_gate, d_gate, qs_up, d_up, expert_ids, E: int, dev_status=None,
                     stream=None) -> None:
    T, topk, N, K = _moe_dims(qs_gate, d_gate, expert_ids, E)
    _check(load().moe_q4_pure_read(_ptr(sink_gate, torch.float32, "sink_gate"), _ptr(sink_up, torch.float32, "sink_up"),
                                   _ptr(qs_gate, torch.uint8, "qs_gate"), _ptr(d_gate, torch.float16, "d_gate"),
                                   _ptr(qs_up, torch.uint8, "qs_up"), _ptr(d_up, torch.float16, "d_up"),
                                   _ptr(expert_ids, torch.int32, "expert_ids"), T, topk, E, N, K,
                                   _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def q4_dequant(W, qs, d, stream=None) -> None:
    N, K = _q4_dims(qs, d)
    if W.numel() != N * K:
        raise ValueError("W must be [N, K]")
    _check(load().q4_dequant(_ptr(W, torch.float32, "W"), _ptr(qs, torch.uint8, "qs"), _ptr(d, torch.float16, "d"),
                             N, K, _stream(stream)))


def q4k_dequant(W, w, stream=None) -> None:
    N, K = _q4k_dims(w)
    if W.numel() != N * K:
        raise ValueError("W must be [N, K]")
    _check(load().q4k_dequant(_ptr(W, torch.float32, "W"), _ptr(w, torch.uint8, "w"), N, K, _stream(stream)))


def q4_set_launch_overlap(enable: bool) -> None:
    """Turn launch overlap (programmatic dependent launch) on or off for every later GEMV/MoE launch.

    While on, the kernel that runs directly before a call in the same stream must not write that call's
    weights; inputs and outputs may depend on it freely (each kernel waits for it before touching them).
    """
    _check(load().q4_set_launch_overlap(1 if enable else 0))


def q4_get_launch_overlap() -> bool:
    return bool(load().q4_get_launch_overlap())


def q4_set_wait_limit(cycles: int) -> None:
    """Set the limit, in SM cycles, of each kernel wait for a weight stage (default DEFAULT_WAIT_LIMIT). A wait
    that runs out makes its warp store NaN rows and record FAULT_WAIT_TIMEOUT; 0 makes every such wait give up at
    once, which exercises that path."""
    _check(load().q4_set_wait_limit(int(cycles)))


def q4_get_wait_limit() -> int:
    return int(load().q4_get_wait_limit())


def q4_device_faults() -> int:
    """Synchronise the device and return (and clear) the fault bits the kernels recorded."""
    out = ctypes.c_uint(0)
    _check(load().q4_device_faults(ctypes.byref(out)))
    return out.value
