"""The bounded stage wait's timeout path, run on copies that do land: with the wait limit set to 0 every wait
for a weight stage gives up at once, so each kernel that streams through mbarrier-completed copies must store
NaN rows, record FAULT_WAIT_TIMEOUT (and not FAULT_COPY_LOST: the copies it had issued still land and are
waited for before the CTA exits), and leave the context usable: the next call with the default limit is exact
and records no fault. Kernels that stream with cp.async groups (rows longer than one chunk) have no such wait
and stay exact."""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, assert_close, cu

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def with_zero_limit(fn):
    """Run fn() with every stage wait giving up at once; return its result and the fault bits it recorded."""
    assert q4.q4_device_faults() == 0
    q4.q4_set_wait_limit(0)
    try:
        out = fn()
        faults = q4.q4_device_faults()
    finally:
        q4.q4_set_wait_limit(q4.DEFAULT_WAIT_LIMIT)
    assert q4.q4_get_wait_limit() == q4.DEFAULT_WAIT_LIMIT
    return out, faults


def check_timed_out(faults, *outs):
    assert faults & q4.FAULT_WAIT_TIMEOUT, f"faults={faults}"
    assert not faults & q4.FAULT_COPY_LOST, f"faults={faults}"
    for o in outs:
        assert np.all(np.isnan(o)), "every row must be NaN after every wait gave up"


@pytest.mark.parametrize("N,K", [(1000, 4096), (77, 1024)])
def test_q4_gemv_timeout_then_exact(N, K, oracle_lib):
    inp = synth.make_q4_gemv(seed=N, N=N, K=K)
    qs, d, x = cu(inp["qs"]), cu(inp["d"]), cu(inp["x"][0])

    def call():
        y = Guarded(N)
        q4.q4_gemv(y.t, qs, d, x)
        return y.result()

    out, faults = with_zero_limit(call)
    check_timed_out(faults, out)
    ref, bound = oracle_lib.q4_gemv(inp["qs"], inp["d"], inp["x"][0])
    assert_close(call(), ref, bound, "q4_gemv after the timeout test")
    assert q4.q4_device_faults() == 0


def test_q4_gemv_batched_timeout_then_exact(oracle_lib):
    M, N, K = 4, 500, 2048
    inp = synth.make_q4_gemv(seed=5, N=N, K=K, M=M)
    qs, d, X = cu(inp["qs"]), cu(inp["d"]), cu(inp["x"])

    def call():
        Y = Guarded(M, N)
        q4.q4_gemv_batched(Y.t, qs, d, X)
        return Y.result()

    out, faults = with_zero_limit(call)
    check_timed_out(faults, out)
    ref, bound = oracle_lib.q4_gemv_batched(inp["qs"], inp["d"], inp["x"])
    assert_close(call(), ref, bound, "batched after the timeout test")
    assert q4.q4_device_faults() == 0


def test_chunked_rows_have_no_stage_wait(oracle_lib):
    # rows longer than 128 blocks stream in cp.async chunks: nothing to time out
    N, K = 120, 8192
    inp = synth.make_q4_gemv(seed=6, N=N, K=K)

    def call():
        y = Guarded(N)
        q4.q4_gemv(y.t, cu(inp["qs"]), cu(inp["d"]), cu(inp["x"][0]))
        return y.result()

    out, faults = with_zero_limit(call)
    assert faults == 0
    ref, bound = oracle_lib.q4_gemv(inp["qs"], inp["d"], inp["x"][0])
    assert_close(out, ref, bound, "chunked rows under a zero wait limit")


@pytest.mark.parametrize("gamma", [True, False])
def test_gateup_q4k_timeout_then_exact(gamma, oracle_lib):
    N, K = 700, 3584
    g = synth.make_gateup(seed=7, N=N, K=K, with_gamma=gamma)
    args = (cu(g["w_gate"]), cu(g["w_up"]), cu(g["x"]), cu(g["gamma"]) if gamma else None, float(g["eps"]))

    def call():
        yg, yu = Guarded(N), Guarded(N)
        q4.fused_gateup_q4k_gemv(yg.t, yu.t, *args)
        return yg.result(), yu.result()

    (og, ou), faults = with_zero_limit(call)
    check_timed_out(faults, og, ou)
    (rg, bg), (ru, bu) = oracle_lib.fused_gateup_q4k_gemv(g["w_gate"], g["w_up"], g["x"], g["gamma"], g["eps"])
    og, ou = call()
    assert_close(og, rg, bg, "gate after the timeout test")
    assert_close(ou, ru, bu, "up after the timeout test")
    assert q4.q4_device_faults() == 0


def test_moe_timeout_then_exact(oracle_lib):
    E, N, K, T, topk = 16, 256, 2048, 4, 4
    m = synth.make_moe(seed=8, E=E, N=N, K=K, T=T, topk=topk)
    args = [cu(m[k]) for k in ("qs_gate", "d_gate", "qs_up", "d_up", "x", "ids")]

    def call():
        yg, yu = Guarded(T, topk, N), Guarded(T, topk, N)
        q4.moe_q4_gemv(yg.t, yu.t, *args, E)
        return yg.result(), yu.result()

    (og, ou), faults = with_zero_limit(call)
    check_timed_out(faults, og, ou)
    (rg, bg), (ru, bu) = oracle_lib.moe_q4_gemv(m["qs_gate"], m["d_gate"], m["qs_up"], m["d_up"], m["x"], m["ids"], E)
    og, ou = call()
    assert_close(og, rg, bg, "moe gate after the timeout test")
    assert_close(ou, ru, bu, "moe up after the timeout test")
    assert q4.q4_device_faults() == 0


def test_pure_reads_time_out_too():
    inp = synth.make_q4_gemv(seed=9, N=640, K=4096)
    w = synth.q4k_weights(np.random.default_rng(10), 320, 2048)

    def call():
        s1, s2 = Guarded(640), Guarded(320)
        q4.q4_pure_read(s1.t, cu(inp["qs"]), cu(inp["d"]))
        q4.q4k_pure_read(s2.t, cu(w))
        return s1.result(), s2.result()

    (a, b), faults = with_zero_limit(call)
    check_timed_out(faults, a, b)
    # the sinks hold raw XOR bits (which may spell a NaN), so the normal call is checked bit for bit
    a, b = call()
    qs32 = inp["qs"].reshape(640, -1).view("<u4")
    expect_a = np.bitwise_xor.reduce(qs32, axis=1) ^ np.bitwise_xor.reduce(
        inp["d"].view(np.uint16).astype(np.uint32), axis=1)
    expect_b = np.bitwise_xor.reduce(w.reshape(320, -1).view("<u4"), axis=1)
    assert np.array_equal(a.view(np.uint32), expect_a) and np.array_equal(b.view(np.uint32), expect_b)
    assert q4.q4_device_faults() == 0


def test_wait_limit_refuses_negative():
    with pytest.raises(q4.Q4Error):
        q4.q4_set_wait_limit(-1)
    assert q4.q4_get_wait_limit() == q4.DEFAULT_WAIT_LIMIT
