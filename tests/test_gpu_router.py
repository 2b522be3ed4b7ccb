"""MoE router (gate GEMV + top-K softmax) on the GPU, through the C ABI, against the oracle.

What is compared, and why: the logits are a GEMV, held to the library's tolerance against the oracle's fp64
logits. The expert choice is an integer decided by floating point, so it is checked at the kernel's own
precision: the oracle's top-K selection applied to the kernel's fp32 logits must give exactly the kernel's ids,
and the weights must match the oracle's softmax of those same logits. Where the fp64 logits leave a margin
wider than the tolerance around the K-th place, the ids must also equal the fp64 oracle's."""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, assert_close, cu

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def run_router(qs, d, x, topk, normalize):
    T = x.shape[0]
    E = d.shape[0]
    ids = torch.empty(T, topk, dtype=torch.int32, device="cuda")
    w = Guarded(T, topk)
    lg = Guarded(T, E)
    q4.moe_router_q4(ids, w.t, cu(qs), cu(d), cu(x), topk, normalize, logits=lg.t)
    return ids.cpu().numpy(), w.result(), lg.result()


@pytest.mark.parametrize("E,K,T,topk", [(64, 2048, 8, 8), (16, 256, 3, 4), (128, 4096, 1, 2), (7, 96, 5, 7),
                                        (300, 1024, 2, 33), (1, 256, 2, 1), (4096, 512, 2, 8)])
@pytest.mark.parametrize("normalize", [True, False])
def test_router_matches_oracle(E, K, T, topk, normalize, oracle_lib):
    rng = np.random.default_rng(E * 1000 + K + T)
    qs, d = synth.q4_weights(rng, E, K)
    x = synth.activations(rng, T, K)
    ids, w, lg = run_router(qs, d, x, topk, normalize)
    ref_lg, bound, ref_ids, ref_w = oracle_lib.moe_router(qs, d, x, topk, normalize)
    assert_close(lg, ref_lg, bound, f"router logits E{E} K{K}")
    own_ids, own_w = oracle_lib.topk_softmax_f32(lg, topk, normalize)
    assert np.array_equal(ids, own_ids), "ids differ from the top-K of the kernel's own logits"
    assert np.allclose(w, own_w, rtol=2e-5, atol=1e-7), "weights differ from the softmax of the kernel's logits"
    tol = 1e-3 * bound + 1e-5
    for t in range(T):
        srt = np.sort(ref_lg[t])[::-1]
        if topk < E and srt[topk - 1] - srt[topk] > 2 * tol[t].max():
            assert set(ids[t].tolist()) == set(ref_ids[t].tolist())


def test_router_ties_go_to_the_lower_index(oracle_lib):
    rng = np.random.default_rng(9)
    E, K, T, topk = 12, 512, 4, 5
    qs, d = synth.q4_weights(rng, E, K)
    for a, b in ((2, 9), (4, 5), (0, 11)):  # identical rows give bit-identical logits
        qs[b], d[b] = qs[a], d[a]
    x = synth.activations(rng, T, K)
    ids, w, lg = run_router(qs, d, x, topk, True)
    for a, b in ((2, 9), (4, 5), (0, 11)):
        assert np.array_equal(lg[:, a].view(np.uint32), lg[:, b].view(np.uint32))
    own_ids, _ = oracle_lib.topk_softmax_f32(lg, topk, True)
    assert np.array_equal(ids, own_ids)
    for t in range(T):
        for a, b in ((2, 9), (4, 5), (0, 11)):
            if b in ids[t]:
                assert a in ids[t] and list(ids[t]).index(a) < list(ids[t]).index(b)


def test_router_feeds_moe(oracle_lib):
    """The router's ids drive moe_q4_gemv directly on the device (no host round trip)."""
    rng = np.random.default_rng(11)
    E, N, K, T, topk = 16, 200, 1024, 8, 4
    rq, rd = synth.q4_weights(rng, E, K)
    m = synth.make_moe(seed=12, E=E, N=N, K=K, T=T, topk=topk)
    x = cu(m["x"])
    ids = torch.empty(T, topk, dtype=torch.int32, device="cuda")
    w = torch.empty(T, topk, device="cuda")
    q4.moe_router_q4(ids, w, cu(rq), cu(rd), x, topk, True)
    yg, yu = Guarded(T, topk, N), Guarded(T, topk, N)
    q4.moe_q4_gemv(yg.t, yu.t, cu(m["qs_gate"]), cu(m["d_gate"]), cu(m["qs_up"]), cu(m["d_up"]), x, ids, E)
    idn = ids.cpu().numpy()
    (rg, bg), (ru, bu) = oracle_lib.moe_q4_gemv(m["qs_gate"], m["d_gate"], m["qs_up"], m["d_up"], m["x"], idn, E)
    assert_close(yg.result(), rg, bg, "moe gate after router")
    assert_close(yu.result(), ru, bu, "moe up after router")
    assert np.allclose(w.cpu().numpy().sum(axis=1), 1.0, rtol=1e-5)


def test_router_refusals():
    rng = np.random.default_rng(1)
    qs, d = synth.q4_weights(rng, 8, 64)
    x = torch.zeros(2, 64, device="cuda")
    ids = torch.empty(2, 9, dtype=torch.int32, device="cuda")
    w = torch.empty(2, 9, device="cuda")
    with pytest.raises(q4.Q4Error, match="topk"):
        q4.moe_router_q4(ids, w, cu(qs), cu(d), x, 9, True)


def test_router_nan_input_ranks_every_expert_equal_and_last(oracle_lib):
    # a NaN in token 0's x makes all its logits NaN: NaNs tie to the lower index (ids 0..topk-1) and every
    # weight is NaN; token 1 is unaffected
    E, K, T, topk = 32, 512, 2, 5
    rng = np.random.default_rng(77)
    qs, d = synth.q4_weights(rng, E, K)
    x = synth.activations(rng, T, K)
    x[0, 100] = np.nan
    ids, w, lg = run_router(qs, d, x, topk, True)
    assert np.all(np.isnan(lg[0])) and np.all(np.isfinite(lg[1]))
    assert ids[0].tolist() == list(range(topk))
    assert np.all(np.isnan(w[0]))
    own_ids, own_w = oracle_lib.topk_softmax_f32(lg, topk, True)
    assert np.array_equal(ids, own_ids)
    assert np.allclose(w[1], own_w[1], rtol=2e-5, atol=1e-7)


@pytest.mark.parametrize("E", [6, 40, 100])
def test_router_nan_logit_comes_last_with_topk_all(E, oracle_lib):
    # one expert's row has a NaN scale, so its logit is NaN; with topk = E it must be the last pick
    K, T = 256, 3
    rng = np.random.default_rng(E)
    qs, d = synth.q4_weights(rng, E, K)
    bad = E // 3
    d[bad, 2] = np.float16(np.nan)
    x = synth.activations(rng, T, K)
    ids, w, lg = run_router(qs, d, x, E, False)
    assert np.all(np.isnan(lg[:, bad]))
    assert np.all(ids[:, -1] == bad)
    own_ids, _ = oracle_lib.topk_softmax_f32(lg, E, False)
    assert np.array_equal(ids, own_ids)
    assert np.all(np.isnan(w)), "a NaN logit makes the softmax NaN"
    for t in range(T):
        assert sorted(ids[t].tolist()) == list(range(E))
