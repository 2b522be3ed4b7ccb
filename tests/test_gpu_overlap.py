"""Launch overlap (programmatic dependent launch) keeps a dependent chain exact.

A chain through all five kernel families, each call reading an earlier call's output, runs several times
with a fresh input vector each time: eagerly with overlap off (the reference), eagerly with overlap on, and
captured once in a CUDA graph with overlap on and replayed. The kernels are deterministic, so every output
must match the reference bit for bit; a kernel that read its input or wrote its output before the previous
kernel finished would show up as a difference.
"""

import numpy as np
import pytest
import torch

import synth
from gpu_util import cu

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


class Chain:
    def __init__(self, seed=0):
        rng = np.random.default_rng(seed)
        K = 4096
        self.w1 = [cu(a) for a in synth.q4_weights(rng, 4096, K)]          # q4_gemv: x0 -> buf[0]
        self.w2 = cu(synth.q4k_weights(rng, 4096, K))                        # fused rmsnorm: buf[0] -> buf[1]
        self.g2 = cu(synth.gamma(rng, K))
        self.w3 = [cu(a) for a in synth.q4_weights(rng, 2048, K)]          # batched M=8: buf -> Y3 [8][2048]
        self.moe = [cu(a) for a in synth.q4_weights(rng, 8 * 4096, 2048)]  # MoE gate: 8 experts x 4096 x 2048
        self.moe_up = [cu(a) for a in synth.q4_weights(rng, 8 * 4096, 2048)]
        self.ids = cu(synth.expert_ids(rng, 8, 2, 8))
        self.wg = cu(synth.q4k_weights(rng, 1024, 4096))                     # gate+up: yg[0, 0] -> out
        self.wu = cu(synth.q4k_weights(rng, 1024, 4096))
        self.gg = cu(synth.gamma(rng, 4096))
        self.inputs = [cu(synth.activations(rng, 1, K)[0]) for _ in range(3)]
        rest = cu(synth.activations(rng, 8, K))
        self.x0 = torch.empty(K, device="cuda")
        self.buf = rest.clone()
        self.y3 = torch.empty(8, 2048, device="cuda")
        self.yg = torch.empty(8, 2, 4096, device="cuda")
        self.yu = torch.empty(8, 2, 4096, device="cuda")
        self.og = torch.empty(1024, device="cuda")
        self.ou = torch.empty(1024, device="cuda")

    def step(self, i):
        self.x0.copy_(self.inputs[i])
        q4.q4_gemv(self.buf[0], *self.w1, self.x0)
        q4.fused_rmsnorm_q4k_gemv(self.buf[1], self.w2, self.buf[0], self.g2, 1e-5)
        q4.q4_gemv_batched(self.y3, *self.w3, self.buf)
        q4.moe_q4_gemv(self.yg, self.yu, *self.moe, *self.moe_up, self.y3, self.ids, 8)
        q4.fused_gateup_q4k_gemv(self.og, self.ou, self.wg, self.wu, self.yg[0, 0], self.gg, 1e-5)

    def outputs(self):
        return [t.detach().cpu().numpy().copy() for t in (self.buf, self.y3, self.yg, self.yu, self.og, self.ou)]


def run(chain, overlap, graph):
    q4.q4_set_launch_overlap(overlap)
    try:
        outs = []
        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            gs = []
            with torch.cuda.stream(s):
                chain.step(0)  # warm-up outside capture (lazy module and attribute set-up)
            torch.cuda.synchronize()
            for i in range(3):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    chain.step(i)
                gs.append(g)
            for g in gs:
                g.replay()
                torch.cuda.synchronize()
                outs.append(chain.outputs())
        else:
            for i in range(3):
                chain.step(i)
                torch.cuda.synchronize()
                outs.append(chain.outputs())
        return outs
    finally:
        q4.q4_set_launch_overlap(False)


def test_overlap_setting_round_trips():
    assert q4.q4_get_launch_overlap() is False
    q4.q4_set_launch_overlap(True)
    assert q4.q4_get_launch_overlap() is True
    q4.q4_set_launch_overlap(False)
    assert q4.q4_get_launch_overlap() is False


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_dependent_chain_is_exact_with_overlap(graph):
    chain = Chain()
    ref = run(chain, overlap=False, graph=False)
    got = run(chain, overlap=True, graph=graph)
    for i, (a, b) in enumerate(zip(ref, got)):
        for j, (ra, gb) in enumerate(zip(a, b)):
            assert np.all(np.isfinite(ra)), (i, j)
            assert np.array_equal(ra.view(np.uint32), gb.view(np.uint32)), f"step {i}, output {j}"
    # successive steps saw different inputs, so the chain really depends on x0
    assert not np.array_equal(ref[0][0], ref[1][0])
    assert q4.q4_device_faults() == 0
