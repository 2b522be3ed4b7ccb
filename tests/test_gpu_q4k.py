"""Fused RMSNorm + Q4_K GEMV, fused gate+up Q4_K GEMV, the Q4_K pure-read instrument and dequant dump on
the GPU, through the C ABI, against the fp64 oracle on the same seeded inputs."""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, assert_close, cu
from oracle_pins import q4k_block

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def run_fused(w, x, gamma, eps=1e-5):
    y = Guarded(w.shape[0])
    q4.fused_rmsnorm_q4k_gemv(y.t, cu(w), cu(x), cu(gamma), eps)
    return y.result()


def run_gateup(wg, wu, x, gamma, eps=1e-5):
    N = wg.shape[0]
    yg, yu = Guarded(N), Guarded(N)
    q4.fused_gateup_q4k_gemv(yg.t, yu.t, cu(wg), cu(wu), cu(x), None if gamma is None else cu(gamma), eps)
    return yg.result(), yu.result()


@pytest.mark.parametrize("N,K", [(3584, 3584), (1, 256), (7, 512), (100, 768), (5001, 3584), (257, 4096)])
def test_fused_rmsnorm_q4k_gemv(N, K, oracle_lib):
    f = synth.make_fused_rmsnorm(seed=N + K, N=N, K=K)
    ref, bound = oracle_lib.fused_rmsnorm_q4k_gemv(f["w"], f["x"], f["gamma"], f["eps"])
    assert_close(run_fused(f["w"], f["x"], f["gamma"]), ref, bound, f"fused {N}x{K}")


@pytest.mark.parametrize("N,K,with_gamma", [(18944, 3584, True), (18944, 3584, False), (33, 1024, True),
                                            (1, 256, False), (999, 1280, True)])
def test_fused_gateup_q4k_gemv(N, K, with_gamma, oracle_lib):
    g = synth.make_gateup(seed=N + K, N=N, K=K, with_gamma=with_gamma)
    (rg, bg), (ru, bu) = oracle_lib.fused_gateup_q4k_gemv(g["w_gate"], g["w_up"], g["x"], g["gamma"], g["eps"])
    yg, yu = run_gateup(g["w_gate"], g["w_up"], g["x"], g["gamma"])
    assert_close(yg, rg, bg, "gate")
    assert_close(yu, ru, bu, "up")


def test_q4k_degenerate_blocks(oracle_lib):
    rng = np.random.default_rng(3)
    K, N = 1024, 48
    x = rng.standard_normal(K).astype(np.float32)
    gamma = rng.normal(1, 0.1, K).astype(np.float32)
    cases = {
        "scale 0 (min term only)": lambda: q4k_block(rng.uniform(1e-3, 1e-2), rng.uniform(1e-3, 1e-2), [0] * 8,
                                                     rng.integers(0, 64, 8), rng.integers(0, 256, 128)),
        "min 0 (scale term only)": lambda: q4k_block(rng.uniform(1e-3, 1e-2), rng.uniform(1e-3, 1e-2),
                                                     rng.integers(0, 64, 8), [0] * 8, rng.integers(0, 256, 128)),
        "codes 0": lambda: q4k_block(rng.uniform(1e-3, 1e-2), rng.uniform(1e-3, 1e-2), rng.integers(0, 64, 8),
                                     rng.integers(0, 64, 8), np.zeros(128, np.uint8)),
        "all max": lambda: q4k_block(0.01, 0.01, [63] * 8, [63] * 8, np.full(128, 255, np.uint8)),
    }
    for name, mk in cases.items():
        w = np.stack([np.stack([mk() for _ in range(K // 256)]) for _ in range(N)])
        ref, bound = oracle_lib.fused_rmsnorm_q4k_gemv(w, x, gamma, 1e-5)
        assert_close(run_fused(w, x, gamma), ref, bound, name)
    # gamma = 0 gives exactly zero
    w = synth.q4k_weights(rng, N, K)
    assert np.all(run_fused(w, x, np.zeros(K, np.float32)) == 0.0)
    # constant input: the normalised input is c / sqrt(c^2 + eps) everywhere
    for c in (3.0, 1e-4):
        xc = np.full(K, c, np.float32)
        ref, bound = oracle_lib.fused_rmsnorm_q4k_gemv(w, xc, gamma, 1e-5)
        assert_close(run_fused(w, xc, gamma), ref, bound, f"constant {c}")


def test_gateup_unnormed_extreme_inputs(oracle_lib):
    rng = np.random.default_rng(4)
    N, K = 64, 768
    wg, wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    for scale in (1e20, 1e-30):
        x = (rng.standard_normal(K) * scale).astype(np.float32)
        (rg, bg), (ru, bu) = oracle_lib.fused_gateup_q4k_gemv(wg, wu, x, None, 1e-5)
        yg, yu = run_gateup(wg, wu, x, None)
        assert_close(yg / scale, rg / scale, bg / scale, f"gate x*{scale}")
        assert_close(yu / scale, ru / scale, bu / scale, f"up x*{scale}")


def test_eps_is_honoured(oracle_lib):
    f = synth.make_fused_rmsnorm(seed=9, N=64, K=512)
    x = (f["x"] * 1e-3).astype(np.float32)  # mean square comparable to eps
    for eps in (0.0, 1e-6, 1e-2):
        ref, bound = oracle_lib.fused_rmsnorm_q4k_gemv(f["w"], x, f["gamma"], eps)
        assert_close(run_fused(f["w"], x, f["gamma"], eps), ref, bound, f"eps={eps}")


def test_q4k_pure_read_touches_exactly_the_weight_bytes():
    for N, K in ((3584, 3584), (13, 256), (18944, 3584)):
        w = synth.q4k_weights(np.random.default_rng(N), N, K)
        sink = Guarded(N)
        q4.q4k_pure_read(sink.t, cu(w))
        got = sink.result().view(np.uint32)
        expect = np.bitwise_xor.reduce(w.reshape(N, -1).view("<u4"), axis=1)
        assert np.array_equal(got, expect)


@pytest.mark.parametrize("N,K", [(3584, 3584), (9, 256), (77, 1280)])
def test_q4k_dequant_is_bit_exact(N, K, oracle_lib):
    w = synth.q4k_weights(np.random.default_rng(K + N), N, K)
    W = Guarded(N, K)
    q4.q4k_dequant(W.t, cu(w))
    assert np.array_equal(W.result().view(np.uint32), oracle_lib.dequant_q4k(w).view(np.uint32))


def test_no_fault_bits_after_the_suite():
    assert q4.q4_device_faults() == 0
