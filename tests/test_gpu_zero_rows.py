"""Rows whose weights are all zero, with large inputs, through every GEMV family, against the fp64 oracle
under the undivided tolerance |y - y_ref| <= 1e-3 * sum_k |w_k||x_k| + 1e-5.

For a zero-weight row the oracle's value and bound are both exactly 0, so the limit is the absolute 1e-5
alone, whatever the input's magnitude. The kernels fold each block's offset terms so that such rows come out
exactly 0: planar Q4 blocks of code 8 (w = (q - 8) * d), and Q4_K sub-blocks whose d*sc*q equals dmin*m
(sc = m = 0, or a constant code of 1 or 2 with d = dmin and m = sc*q). Zero rows sit between rows of random
weights, and the inputs are N(0, sigma^2) with sigma = 100 and 10^4.
"""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, assert_close, cu
from oracle_pins import q4k_block

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402

SIGMAS = [100.0, 1e4]


def big_x(seed, M, K, sigma):
    return (np.random.default_rng(seed).standard_normal((M, K)) * sigma).astype(np.float32)


def q4_with_zero_rows(seed, rows, K, every=3):
    """Planar Q4 weights with every `every`-th row all code 8 (zero weights); returns (qs, d, zero-row mask)."""
    qs, d = synth.q4_weights(np.random.default_rng(seed), rows, K)
    zero = np.zeros(rows, bool)
    zero[::every] = True
    qs[zero] = 0x88
    return qs, d, zero


def q4k_with_zero_rows(seed, N, K):
    """Q4_K weights where rows r % 4 == 0 are zero weights by d = dmin, sc = m and codes 1; r % 4 == 1 by
    sc = m = 0 (random codes); r % 4 == 2 by d = dmin, m = 2 sc and codes 2; rows r % 4 == 3 are random."""
    rng = np.random.default_rng(seed)
    w = synth.q4k_weights(rng, N, K)
    nsb = K // 256
    for r in range(N):
        kind = r % 4
        if kind == 3:
            continue
        for sb in range(nsb):
            d = np.float16(rng.uniform(1e-3, 1e-2))
            if kind == 0:
                sc = rng.integers(0, 64, 8)
                w[r, sb] = q4k_block(d, d, sc, sc, np.full(128, 0x11, np.uint8))
            elif kind == 1:
                w[r, sb] = q4k_block(d, np.float16(rng.uniform(1e-3, 1e-2)), np.zeros(8, np.int64), np.zeros(8, np.int64),
                                     rng.integers(0, 256, 128).astype(np.uint8))
            else:
                sc = rng.integers(0, 32, 8)
                w[r, sb] = q4k_block(d, d, sc, 2 * sc, np.full(128, 0x22, np.uint8))
    return w, (np.arange(N) % 4) != 3


@pytest.mark.parametrize("sigma", SIGMAS)
@pytest.mark.parametrize("N,K", [
    (600, 4096),   # the register-input kernel, whole 128-block rows
    (300, 1024),
    (200, 2816),   # 88 blocks: a short last unit round
    (150, 96),     # scales loaded by lanes (K % 256 != 0)
    (90, 8192),    # rows streamed in chunks
])
def test_q4_gemv_zero_rows(N, K, sigma, oracle_lib):
    qs, d, zero = q4_with_zero_rows(N + K, N, K)
    x = big_x(1, 1, K, sigma)
    ref, bound = oracle_lib.q4_gemv(qs, d, x[0])
    y = Guarded(N)
    q4.q4_gemv(y.t, cu(qs), cu(d), cu(x[0]))
    out = y.result()
    assert_close(out, ref, bound, f"q4_gemv {N}x{K} sigma={sigma}")
    assert np.all(out[zero] == 0.0)


@pytest.mark.parametrize("sigma", SIGMAS)
@pytest.mark.parametrize("M", [2, 8, 12])
def test_q4_gemv_batched_zero_rows(M, sigma, oracle_lib):
    N, K = 333, 2048
    qs, d, zero = q4_with_zero_rows(M, N, K)
    X = big_x(2 + M, M, K, sigma)
    ref, bound = oracle_lib.q4_gemv_batched(qs, d, X)
    Y = Guarded(M, N)
    q4.q4_gemv_batched(Y.t, cu(qs), cu(d), cu(X))
    out = Y.result()
    assert_close(out, ref, bound, f"q4_gemv_batched M={M} sigma={sigma}")
    assert np.all(out[:, zero] == 0.0)


@pytest.mark.parametrize("sigma", SIGMAS)
def test_moe_zero_rows(sigma, oracle_lib):
    E, N, K, T, topk = 8, 130, 2048, 5, 4
    qg, dg, zero = q4_with_zero_rows(11, E * N, K, every=4)
    qu, du, _ = q4_with_zero_rows(12, E * N, K, every=4)
    qg[2 * N:3 * N] = 0x88  # every row of expert 2 (gate) is zero
    x = big_x(3, T, K, sigma)
    ids = synth.expert_ids(np.random.default_rng(4), T, topk, E)
    ids[0, 0] = 2
    (rg, bg), (ru, bu) = oracle_lib.moe_q4_gemv(qg, dg, qu, du, x, ids, E)
    yg, yu = Guarded(T, topk, N), Guarded(T, topk, N)
    q4.moe_q4_gemv(yg.t, yu.t, cu(qg), cu(dg), cu(qu), cu(du), cu(x), cu(ids), E)
    og, ou = yg.result(), yu.result()
    assert_close(og, rg, bg, f"moe gate sigma={sigma}")
    assert_close(ou, ru, bu, f"moe up sigma={sigma}")
    assert np.all(og[0, 0] == 0.0)
    assert np.all(og[rg == 0.0] == 0.0) and np.all(ou[ru == 0.0] == 0.0)


@pytest.mark.parametrize("sigma", SIGMAS)
def test_router_zero_rows(sigma, oracle_lib):
    E, K, T, topk = 24, 2048, 3, 6
    rq, rd, zero = q4_with_zero_rows(21, E, K, every=4)
    x = big_x(5, T, K, sigma)
    lg_ref, lg_bound, _, _ = oracle_lib.moe_router(rq, rd, x, topk, True)
    ids = torch.empty(T, topk, dtype=torch.int32, device="cuda")
    wts = torch.empty(T, topk, device="cuda")
    lg = Guarded(T, E)
    q4.moe_router_q4(ids, wts, cu(rq), cu(rd), cu(x), topk, True, logits=lg.t)
    out = lg.result()
    assert_close(out, lg_ref, lg_bound, f"router logits sigma={sigma}")
    assert np.all(out[:, zero] == 0.0)


@pytest.mark.parametrize("sigma", SIGMAS)
def test_gateup_q4k_zero_rows_without_norm(sigma, oracle_lib):
    N, K = 260, 3584
    wg, zero = q4k_with_zero_rows(31, N, K)
    wu, _ = q4k_with_zero_rows(32, N, K)
    x = big_x(6, 1, K, sigma)[0]
    (rg, bg), (ru, bu) = oracle_lib.fused_gateup_q4k_gemv(wg, wu, x, None, 1e-5)
    yg, yu = Guarded(N), Guarded(N)
    q4.fused_gateup_q4k_gemv(yg.t, yu.t, cu(wg), cu(wu), cu(x), None, 1e-5)
    og, ou = yg.result(), yu.result()
    assert_close(og, rg, bg, f"gate sigma={sigma}")
    assert_close(ou, ru, bu, f"up sigma={sigma}")
    assert np.all(og[zero] == 0.0) and np.all(ou[zero] == 0.0)


def test_rmsnorm_q4k_zero_rows(oracle_lib):
    N, K = 200, 2048
    w, zero = q4k_with_zero_rows(41, N, K)
    x = big_x(7, 1, K, 1e4)[0]
    g = synth.gamma(np.random.default_rng(8), K)
    ref, bound = oracle_lib.fused_rmsnorm_q4k_gemv(w, x, g, 1e-5)
    y = Guarded(N)
    q4.fused_rmsnorm_q4k_gemv(y.t, cu(w), cu(x), cu(g), 1e-5)
    out = y.result()
    assert_close(out, ref, bound, "rmsnorm q4k")
    assert np.all(out[zero] == 0.0)


@pytest.mark.parametrize("sigma", SIGMAS)
@pytest.mark.parametrize("M", [1, 3, 8])
def test_q4k_gemv_batched_zero_rows(M, sigma, oracle_lib):
    N, K = 150, 2048
    w, zero = q4k_with_zero_rows(50 + M, N, K)
    X = big_x(9 + M, M, K, sigma)
    Y = Guarded(M, N)
    q4.q4k_gemv_batched(Y.t, cu(w), cu(X))
    out = Y.result()
    for m in range(M):
        ref, bound = oracle_lib.q4k_gemv(w, X[m].astype(np.float64))
        assert_close(out[m], ref, bound, f"q4k_gemv_batched M={M} row {m} sigma={sigma}")
    assert np.all(out[:, zero] == 0.0)
