"""The C ABI library without a GPU: it builds, loads, exports every declared symbol, and refuses bad
arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

import quantized_decode_gemv_q4_gb300 as q4
from quantized_decode_gemv_q4_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4gemv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    if lib_build.is_stale():
        lib_build.build()
    return q4.load()


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for n in ("q4_gemv", "q4_gemv_batched", "fused_rmsnorm_q4k_gemv", "fused_gateup_q4k_gemv", "moe_q4_gemv",
              "q4_pure_read", "q4k_pure_read", "moe_q4_pure_read", "q4_dequant", "q4k_dequant", "q4_last_error",
              "q4_device_faults"):
        assert n in names, n


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in q4gemv.h but not exported"


def test_binding_names_match_the_header():
    for name in declared_functions():
        if name != "q4_last_error":
            assert hasattr(q4, name), name


ALIGNED = 1 << 20  # a fake, 16-byte aligned address; refusals happen before any dereference


def test_refusals_need_no_gpu(lib):
    P = ctypes.c_void_p
    # null output
    assert lib.q4_gemv(None, P(ALIGNED), P(ALIGNED), P(ALIGNED), 4, 64, None) == q4.Q4_EINVAL
    assert b"null output" in lib.q4_last_error()
    # K not a multiple of 32
    assert lib.q4_gemv(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), 4, 48, None) == q4.Q4_EINVAL
    # N <= 0
    assert lib.q4_gemv(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), 0, 64, None) == q4.Q4_EINVAL
    # misaligned quants and input
    assert lib.q4_gemv(P(ALIGNED), P(ALIGNED + 4), P(ALIGNED), P(ALIGNED), 4, 64, None) == q4.Q4_EALIGN
    assert lib.q4_gemv(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED + 8), 4, 64, None) == q4.Q4_EALIGN
    # batched M outside 1..16 is refused, not clamped
    for M in (0, 17, -1):
        assert lib.q4_gemv_batched(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), M, 4, 64, None) == q4.Q4_EINVAL
    assert b"M=17 outside 1..16" in (lib.q4_gemv_batched(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), 17, 4, 64, None)
                                   and lib.q4_last_error())
    # Q4_K: K must be a multiple of 256, eps finite and >= 0
    assert lib.fused_rmsnorm_q4k_gemv(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), ctypes.c_float(1e-5), 4, 128,
                                      None) == q4.Q4_EINVAL
    assert lib.fused_rmsnorm_q4k_gemv(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), ctypes.c_float(-1.0), 4, 256,
                                      None) == q4.Q4_EINVAL
    assert lib.fused_rmsnorm_q4k_gemv(P(ALIGNED), P(ALIGNED), P(ALIGNED), None, ctypes.c_float(1e-5), 4, 256,
                                      None) == q4.Q4_EINVAL
    assert lib.fused_gateup_q4k_gemv(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED + 16 + 8), P(ALIGNED), None,
                                     ctypes.c_float(1e-5), 4, 256, None) == q4.Q4_EALIGN
    # MoE: topk > E, T*topk > 512, null ids
    args = [P(ALIGNED)] * 6 + [P(ALIGNED), P(ALIGNED)]
    assert lib.moe_q4_gemv(*args, 2, 9, 8, 16, 64, None, None) == q4.Q4_EINVAL
    assert lib.moe_q4_gemv(*args, 65, 8, 8, 16, 64, None, None) == q4.Q4_EINVAL
    assert lib.moe_q4_gemv(*([P(ALIGNED)] * 7), None, 2, 2, 8, 16, 64, None, None) == q4.Q4_EINVAL
    # dequant output must be 16-byte aligned
    assert lib.q4_dequant(P(ALIGNED + 4), P(ALIGNED), P(ALIGNED), 4, 64, None) == q4.Q4_EALIGN
    assert lib.q4_device_faults(None) == q4.Q4_EINVAL
