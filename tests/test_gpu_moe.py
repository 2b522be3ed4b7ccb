"""Expert-gathered MoE gate+up Q4 GEMV and its pure-read instrument on the GPU, through the C ABI,
against the fp64 oracle on the same seeded inputs."""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, assert_close, cu

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def run_moe(m, ids, E, status=None):
    T, topk = ids.shape
    N = m["d_gate"].shape[0] // E
    yg, yu = Guarded(T, topk, N), Guarded(T, topk, N)
    q4.moe_q4_gemv(yg.t, yu.t, cu(m["qs_gate"]), cu(m["d_gate"]), cu(m["qs_up"]), cu(m["d_up"]), cu(m["x"]),
                   cu(ids), E, dev_status=status)
    return yg.result(), yu.result()


def check(m, ids, E, oracle_lib, what=""):
    (rg, bg), (ru, bu) = oracle_lib.moe_q4_gemv(m["qs_gate"], m["d_gate"], m["qs_up"], m["d_up"], m["x"], ids, E)
    yg, yu = run_moe(m, ids, E)
    assert_close(yg, rg, bg, what + " gate")
    assert_close(yu, ru, bu, what + " up")
    return yg, yu


def test_moe_full_size_64_experts(oracle_lib):
    m = synth.make_moe(seed=0, E=64, N=1408, K=2048, T=8, topk=8)
    check(m, m["ids"], 64, oracle_lib, "64x1408x2048 t8k8")


@pytest.mark.parametrize("E,N,K,T,topk", [(8, 40, 512, 3, 4), (5, 7, 96, 2, 5), (16, 130, 1024, 1, 2),
                                          (64, 33, 256, 64, 8), (5000, 7, 96, 3, 5), (20000, 7, 96, 3, 5)])
def test_moe_shapes(E, N, K, T, topk, oracle_lib):
    m = synth.make_moe(seed=E + N + K, E=E, N=N, K=K, T=T, topk=topk)
    check(m, m["ids"], E, oracle_lib, f"E{E} N{N} K{K} T{T} k{topk}")


def test_moe_one_expert_for_every_token(oracle_lib):
    """More routed slots than one weight sweep serves: the expert is swept once per group."""
    m = synth.make_moe(seed=1, E=6, N=50, K=512, T=11, topk=1)
    ids = np.full((11, 1), 3, np.int32)
    check(m, ids, 6, oracle_lib, "all on expert 3")


def test_moe_two_experts_over_all_64_slots(oracle_lib):
    """64 routed slots on two experts, each with slots in both halves of the 64 (42 and 22 slots: many groups)."""
    m = synth.make_moe(seed=5, E=64, N=72, K=512, T=8, topk=8)
    ids = np.where(np.arange(64) % 3 == 0, 60, 3).astype(np.int32).reshape(8, 8)
    check(m, ids, 64, oracle_lib, "two experts")


def test_moe_duplicate_expert_within_a_token(oracle_lib):
    m = synth.make_moe(seed=2, E=6, N=24, K=256, T=2, topk=3)
    ids = np.array([[1, 1, 4], [4, 0, 4]], np.int32)
    yg, yu = check(m, ids, 6, oracle_lib, "duplicates")
    assert np.array_equal(yg[0, 0], yg[0, 1]) and np.array_equal(yu[1, 0], yu[1, 2])


def test_moe_invalid_expert_gives_nan_and_status(oracle_lib):
    m = synth.make_moe(seed=3, E=6, N=24, K=256, T=2, topk=3)
    ids = np.array([[1, 6, 4], [-1, 0, 2]], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    T, topk, N = 2, 3, 24
    yg, yu = Guarded(T, topk, N), Guarded(T, topk, N)
    q4.moe_q4_gemv(yg.t, yu.t, cu(m["qs_gate"]), cu(m["d_gate"]), cu(m["qs_up"]), cu(m["d_up"]), cu(m["x"]),
                   cu(ids), 6, dev_status=status)
    yg, yu = yg.result(), yu.result()
    assert int(status.item()) == q4.FAULT_BAD_EXPERT
    assert q4.q4_device_faults() == q4.FAULT_BAD_EXPERT
    bad = np.zeros((T, topk), bool)
    bad[0, 1] = bad[1, 0] = True
    assert np.all(np.isnan(yg[bad])) and np.all(np.isnan(yu[bad]))
    (rg, bg), (ru, bu) = oracle_lib.moe_q4_gemv(m["qs_gate"], m["d_gate"], m["qs_up"], m["d_up"], m["x"], ids, 6)
    assert_close(yg[~bad], rg[~bad], bg[~bad], "valid slots gate")
    assert_close(yu[~bad], ru[~bad], bu[~bad], "valid slots up")


def test_moe_pure_read_touches_the_selected_experts():
    m = synth.make_moe(seed=4, E=64, N=1408, K=2048, T=8, topk=8)
    E, N = 64, 1408
    ids = m["ids"]
    T, topk = ids.shape
    sg, su = Guarded(T, topk, N), Guarded(T, topk, N)
    q4.moe_q4_pure_read(sg.t, su.t, cu(m["qs_gate"]), cu(m["d_gate"]), cu(m["qs_up"]), cu(m["d_up"]), cu(ids), E)
    got_g, got_u = sg.result().view(np.uint32), su.result().view(np.uint32)
    for qs, d, got in ((m["qs_gate"], m["d_gate"], got_g), (m["qs_up"], m["d_up"], got_u)):
        words = np.bitwise_xor.reduce(qs.reshape(E * N, -1).view("<u4"), axis=1)
        scales = np.bitwise_xor.reduce(d.view(np.uint16).astype(np.uint32), axis=1)
        per_row = (words ^ scales).reshape(E, N)
        assert np.array_equal(got, per_row[ids])


def test_no_fault_bits_after_the_suite():
    assert q4.q4_device_faults() == 0


def test_moe_unaligned_scales_give_identical_rows():
    """Scales only 2-byte aligned take the plain-load path into the slot; outputs equal the aligned call's."""
    m = synth.make_moe(seed=21, E=16, N=200, K=2048, T=4, topk=4)
    E, (T, topk), N = 16, m["ids"].shape, 200

    def shifted(a):
        flat = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).ravel()).to("cuda")
        buf = torch.zeros(flat.numel() + 8, dtype=torch.int16, device="cuda")
        buf[1:1 + flat.numel()] = flat
        return buf[1:1 + flat.numel()].view(torch.float16).view(a.shape)

    outs = []
    for dg, du in ((cu(m["d_gate"]), cu(m["d_up"])), (shifted(m["d_gate"]), shifted(m["d_up"]))):
        yg, yu = Guarded(T, topk, N), Guarded(T, topk, N)
        q4.moe_q4_gemv(yg.t, yu.t, cu(m["qs_gate"]), dg, cu(m["qs_up"]), du, cu(m["x"]), cu(m["ids"]), E)
        outs.append((yg.result(), yu.result()))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
