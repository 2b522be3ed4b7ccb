"""Seeded synthetic inputs for the 4-bit decode GEMVs.

This module draws random bytes and floats and places them at the byte positions of the two
packed weight formats. It holds none of the method's arithmetic: no nibble decode, no scale
unpack, no dot product. Both the CUDA-path tests and the oracle tests take their inputs from
here, so the two sides see the same bytes.

Formats (as the pages define them):

* Q4, planar (inferencelayer ``kernel_lab.rs``, the ``GEMV_F16S`` shader's bindings):
  ``qs`` is ``uint8[N][K/32][16]`` (16 packed bytes per 32-weight block) and ``d`` is
  ``float16[N][K/32]`` (one scale per block).
* Q4_K (trueno-gpu ``fused.rs``, ``FusedRmsNormQ4KGemvKernel`` phase 3): ``uint8[N][K/256][144]``
  super-blocks: f16 ``d`` at byte 0, f16 ``dmin`` at byte 2, 12 packed scale bytes at 4..15 and
  128 quant bytes at 16..143.

Distributions follow the five workloads: scales f16(U[1e-3, 1e-2]); quant bytes uniform on 0..255,
so every 4-bit code is uniform on 0..15; x ~ N(0, 1) in fp32; gamma ~ N(1, 0.1) in fp32; MoE
routing picks ``topk`` distinct experts per token uniformly at random. The 12 Q4_K scale bytes are
drawn uniformly, which makes every 6-bit sub-block scale and min uniform on 0..63 (the 12 bytes hold
exactly the 8 scales and 8 mins, 96 bits, with no spare bit). Draw order within a workload is fixed:
scales, quants, x, gamma, expert ids.
"""

from __future__ import annotations

import numpy as np

SCALE_LO = 1e-3
SCALE_HI = 1e-2


def rng_for(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed)


def q4_weights(rng: np.random.Generator, N: int, K: int, scale_lo: float = SCALE_LO,
               scale_hi: float = SCALE_HI):
    """Planar Q4 weights: (qs uint8[N][K/32][16], d float16[N][K/32])."""
    assert K % 32 == 0
    nblk = K // 32
    d = rng.uniform(scale_lo, scale_hi, size=(N, nblk)).astype(np.float16)
    qs = rng.integers(0, 256, size=(N, nblk, 16), dtype=np.uint8)
    return qs, d


def q4k_weights(rng: np.random.Generator, N: int, K: int, scale_lo: float = SCALE_LO,
                scale_hi: float = SCALE_HI):
    """Q4_K super-blocks: uint8[N][K/256][144]."""
    assert K % 256 == 0
    nsb = K // 256
    d = rng.uniform(scale_lo, scale_hi, size=(N, nsb)).astype(np.float16)
    dmin = rng.uniform(scale_lo, scale_hi, size=(N, nsb)).astype(np.float16)
    scale_bytes = rng.integers(0, 256, size=(N, nsb, 12), dtype=np.uint8)
    qs = rng.integers(0, 256, size=(N, nsb, 128), dtype=np.uint8)
    w = np.empty((N, nsb, 144), dtype=np.uint8)
    w[..., 0:2] = d.astype("<f2").view(np.uint8).reshape(N, nsb, 2)
    w[..., 2:4] = dmin.astype("<f2").view(np.uint8).reshape(N, nsb, 2)
    w[..., 4:16] = scale_bytes
    w[..., 16:144] = qs
    return w


def activations(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    return rng.standard_normal(size=(M, K)).astype(np.float32)


def gamma(rng: np.random.Generator, K: int) -> np.ndarray:
    return rng.normal(1.0, 0.1, size=K).astype(np.float32)


def expert_ids(rng: np.random.Generator, T: int, topk: int, E: int) -> np.ndarray:
    """int32[T][topk]: each token picks topk distinct experts uniformly at random."""
    return np.stack([rng.choice(E, size=topk, replace=False) for _ in range(T)]).astype(np.int32)


# ---------------------------------------------------------------------------------------------
# The five workloads, by name. Sizes are the ones the decode GEMVs are measured on.
# ---------------------------------------------------------------------------------------------

WORKLOADS = {
    "q4_gemv_256x1024": dict(kind="q4_gemv", N=256, K=1024),
    "rmsnorm_q4k_gemv_3584x3584": dict(kind="fused_rmsnorm_q4k_gemv", N=3584, K=3584, eps=1e-5),
    "gateup_q4k_gemv_2x18944x3584": dict(kind="fused_gateup_q4k_gemv", N=18944, K=3584, eps=1e-5),
    "batched_q4_gemv_14336x4096": dict(kind="q4_gemv_batched", N=14336, K=4096, Ms=(1, 2, 4, 8)),
    "moe_q4_gemv_e64_1408x2048_t8k8": dict(kind="moe_q4_gemv", E=64, N=1408, K=2048, T=8, topk=8),
}


def make_q4_gemv(seed: int, N: int, K: int, M: int = 1):
    rng = rng_for(seed)
    qs, d = q4_weights(rng, N, K)
    x = activations(rng, M, K)
    return dict(qs=qs, d=d, x=x)


def make_fused_rmsnorm(seed: int, N: int, K: int, eps: float = 1e-5):
    rng = rng_for(seed)
    w = q4k_weights(rng, N, K)
    x = activations(rng, 1, K)[0]
    g = gamma(rng, K)
    return dict(w=w, x=x, gamma=g, eps=np.float32(eps))


def make_gateup(seed: int, N: int, K: int, eps: float = 1e-5, with_gamma: bool = True):
    rng = rng_for(seed)
    w_gate = q4k_weights(rng, N, K)
    w_up = q4k_weights(rng, N, K)
    x = activations(rng, 1, K)[0]
    g = gamma(rng, K) if with_gamma else None
    return dict(w_gate=w_gate, w_up=w_up, x=x, gamma=g, eps=np.float32(eps))


def make_moe(seed: int, E: int, N: int, K: int, T: int, topk: int):
    rng = rng_for(seed)
    qs_g, d_g = q4_weights(rng, E * N, K)
    qs_u, d_u = q4_weights(rng, E * N, K)
    x = activations(rng, T, K)
    ids = expert_ids(rng, T, topk, E)
    return dict(qs_gate=qs_g, d_gate=d_g, qs_up=qs_u, d_up=d_u, x=x, ids=ids)
