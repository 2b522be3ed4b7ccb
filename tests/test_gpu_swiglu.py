"""SwiGLU epilogue variants on the GPU, through the C ABI, against the oracle's silu(g) * u of its fp64 gate and
up outputs.

Tolerance. The two-output kernels hold |g_gpu - g| <= tau_g and |u_gpu - u| <= tau_u with
tau = 1e-3 * sum|w||x| + 1e-5 (the library's stated bound). silu is Lipschitz with constant max|silu'| < 1.1, so
|silu(g_gpu) u_gpu - silu(g) u| <= 1.1 tau_g (|u| + tau_u) + |silu(g)| tau_u; the fp32 exponential and division
add a few ulps of |y|, covered by 1e-6 |y| + 1e-7."""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, cu

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def swiglu_close(y, g, bg, u, bu, oracle_lib, what):
    ref = oracle_lib.swiglu(g, u)
    tg = 1e-3 * bg + 1e-5
    tu = 1e-3 * bu + 1e-5
    lim = 1.1 * tg * (np.abs(u) + tu) + np.abs(oracle_lib.swiglu(g, np.ones_like(g))) * tu + 1e-6 * np.abs(ref) + 1e-7
    y = np.asarray(y, np.float64)
    assert y.shape == ref.shape
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    bad = np.abs(y - ref) > lim
    if np.any(bad):
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} out of tolerance; first {i}: got {y.flat[i]!r}, "
                             f"oracle {ref.flat[i]!r}, limit {lim.flat[i]:.3e}")


@pytest.mark.parametrize("N,K,with_gamma", [(18944, 3584, True), (300, 256, True), (1000, 2048, False),
                                            (17, 512, True)])
def test_gateup_swiglu_matches_oracle(N, K, with_gamma, oracle_lib):
    inp = synth.make_gateup(seed=N + K, N=N, K=K, with_gamma=with_gamma)
    gamma = inp["gamma"] if with_gamma else None
    (g, bg), (u, bu) = oracle_lib.fused_gateup_q4k_gemv(inp["w_gate"], inp["w_up"], inp["x"], gamma, inp["eps"])
    y = Guarded(N)
    q4.fused_gateup_swiglu_q4k_gemv(y.t, cu(inp["w_gate"]), cu(inp["w_up"]), cu(inp["x"]),
                                    cu(gamma) if with_gamma else None, inp["eps"])
    swiglu_close(y.result(), g, bg, u, bu, oracle_lib, f"gate+up swiglu {N}x{K}")


def test_gateup_swiglu_equals_silu_of_the_two_outputs():
    """The fused epilogue applies silu(g)*u to the kernel's own two results (same kernel, same order)."""
    inp = synth.make_gateup(seed=3, N=2048, K=3584)
    args = (cu(inp["w_gate"]), cu(inp["w_up"]), cu(inp["x"]), cu(inp["gamma"]), inp["eps"])
    g, u = torch.empty(2048, device="cuda"), torch.empty(2048, device="cuda")
    q4.fused_gateup_q4k_gemv(g, u, *args)
    y = torch.empty(2048, device="cuda")
    q4.fused_gateup_swiglu_q4k_gemv(y, *args)
    ref = (g / (1 + torch.exp(-g))) * u
    assert torch.allclose(y, ref, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("E,N,K,T,topk", [(64, 1408, 2048, 8, 8), (6, 40, 256, 3, 4), (16, 300, 1024, 8, 2)])
def test_moe_swiglu_matches_oracle(E, N, K, T, topk, oracle_lib):
    m = synth.make_moe(seed=E + N, E=E, N=N, K=K, T=T, topk=topk)
    (g, bg), (u, bu) = oracle_lib.moe_q4_gemv(m["qs_gate"], m["d_gate"], m["qs_up"], m["d_up"], m["x"], m["ids"], E)
    y = Guarded(T, topk, N)
    q4.moe_q4_swiglu_gemv(y.t, cu(m["qs_gate"]), cu(m["d_gate"]), cu(m["qs_up"]), cu(m["d_up"]), cu(m["x"]),
                          cu(m["ids"]), E)
    swiglu_close(y.result(), g, bg, u, bu, oracle_lib, f"moe swiglu E{E} {N}x{K} t{T}k{topk}")


def test_moe_swiglu_one_expert_for_all_tokens_and_invalid_id(oracle_lib):
    """Eight tokens on one expert (two 4-slot groups) plus one invalid id: NaN row and status bit."""
    E, N, K, T, topk = 4, 200, 512, 8, 2
    m = synth.make_moe(seed=5, E=E, N=N, K=K, T=T, topk=topk)
    ids = np.stack([[0, 1 + (t % 3)] for t in range(T)]).astype(np.int32)
    ids[5, 1] = E + 3
    (g, bg), (u, bu) = oracle_lib.moe_q4_gemv(m["qs_gate"], m["d_gate"], m["qs_up"], m["d_up"], m["x"], ids, E)
    y = Guarded(T, topk, N)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q4.moe_q4_swiglu_gemv(y.t, cu(m["qs_gate"]), cu(m["d_gate"]), cu(m["qs_up"]), cu(m["d_up"]), cu(m["x"]),
                          cu(ids), E, dev_status=status)
    out = y.result()
    assert int(status.item()) == q4.FAULT_BAD_EXPERT
    assert q4.q4_device_faults() == q4.FAULT_BAD_EXPERT
    assert np.all(np.isnan(out[5, 1]))
    keep = np.ones((T, topk), bool)
    keep[5, 1] = False
    swiglu_close(out[keep], g[keep], bg[keep], u[keep], bu[keep], oracle_lib, "moe swiglu, valid slots")


def test_no_fault_bits_after_the_suite():
    assert q4.q4_device_faults() == 0
