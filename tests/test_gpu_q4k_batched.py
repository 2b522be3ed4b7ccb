"""Batched (unfused) Q4_K GEMV on the GPU, through the C ABI, against the fp64 oracle (one Q4_K GEMV per input
row, no normalisation)."""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, assert_close, cu

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def oracle_rows(oracle_lib, w, X):
    outs = [oracle_lib.q4k_gemv(w, X[m].astype(np.float64)) for m in range(X.shape[0])]
    return np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs])


@pytest.mark.parametrize("N,K,M", [(3584, 3584, 1), (3584, 3584, 8), (18944, 3584, 4), (300, 256, 3), (1001, 4096, 8),
                                   (17, 512, 2), (5000, 1280, 5), (777, 2048, 6), (1500, 3584, 7)])
def test_q4k_batched_matches_oracle(N, K, M, oracle_lib):
    rng = np.random.default_rng(N + K + M)
    w = synth.q4k_weights(rng, N, K)
    X = synth.activations(rng, M, K)
    ref, bound = oracle_rows(oracle_lib, w, X)
    Y = Guarded(M, N)
    q4.q4k_gemv_batched(Y.t, cu(w), cu(X))
    assert_close(Y.result(), ref, bound, f"q4k batched {N}x{K} M={M}")


def test_q4k_batched_single_row_equals_fused_without_norm_scale(oracle_lib):
    """M = 1 against the fused gate+up kernel run with gamma = NULL on the same matrix: both are W x."""
    rng = np.random.default_rng(3)
    N, K = 2048, 3584
    w = synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, 1, K)
    y = torch.empty(1, N, device="cuda")
    q4.q4k_gemv_batched(y, cu(w), cu(x))
    g, u = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    q4.fused_gateup_q4k_gemv(g, u, cu(w), cu(w), cu(x[0]), None, 1e-5)
    ref, bound = oracle_lib.q4k_gemv(w, x[0].astype(np.float64))
    assert_close(y.cpu().numpy()[0], ref, bound, "batched M=1")
    assert_close(g.cpu().numpy(), ref, bound, "gate+up without norm")


def test_q4k_batched_extreme_and_degenerate_rows(oracle_lib):
    rng = np.random.default_rng(4)
    N, K = 64, 1024
    w = synth.q4k_weights(rng, N, K)
    X = synth.activations(rng, 4, K)
    X[1] *= 1e20
    X[2] *= 1e-30
    X[3] = 0.0
    ref, bound = oracle_rows(oracle_lib, w, X)
    Y = Guarded(4, N)
    q4.q4k_gemv_batched(Y.t, cu(w), cu(X))
    got = Y.result()
    for m, sc in enumerate((1.0, 1e20, 1e-30, 1.0)):
        assert_close(got[m] / sc, ref[m] / sc, bound[m] / sc, f"row {m} scaled {sc}")


def test_q4k_batched_refusals():
    w = synth.q4k_weights(np.random.default_rng(1), 8, 256)
    X = torch.zeros(9, 256, device="cuda")
    Y = torch.empty(9, 8, device="cuda")
    with pytest.raises(q4.Q4Error, match="outside 1..8"):
        q4.q4k_gemv_batched(Y, cu(w), X)
    X = torch.zeros(8, 18944, device="cuda")
    Y = torch.empty(8, 8, device="cuda")
    w = synth.q4k_weights(np.random.default_rng(1), 8, 18944)
    with pytest.raises(q4.Q4Error, match="EUNSUPPORTED"):
        q4.q4k_gemv_batched(Y, cu(w), X)
