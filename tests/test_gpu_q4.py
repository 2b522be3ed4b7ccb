"""Planar Q4 GEMV (single and batched), its pure-read instrument and dequant dump on the GPU, through the
C ABI, against the fp64 oracle on the same seeded inputs."""

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, assert_close, cu

pytestmark = pytest.mark.gpu

import quantized_decode_gemv_q4_gb300 as q4  # noqa: E402


def run_q4(inp, M=None):
    qs, d = cu(inp["qs"]), cu(inp["d"])
    N = inp["d"].shape[0]
    X = inp["x"]
    if M is None:
        y = Guarded(N)
        q4.q4_gemv(y.t, qs, d, cu(X[0]))
        return y.result()
    Y = Guarded(M, N)
    q4.q4_gemv_batched(Y.t, qs, d, cu(X[:M]))
    return Y.result()


@pytest.mark.parametrize("N,K", [
    (256, 1024),   # the 256x1024 workload
    (1, 32),       # one row, one block
    (7, 96),       # scales not 16-byte groupable (K % 256 != 0): plain scale loads
    (13, 288),
    (1000, 4128),  # 129 blocks: a ragged lane iteration, N % 4 != 0
    (333, 8192),   # several chunks per row
    (4099, 2048),
])
def test_q4_gemv_matches_oracle(N, K, oracle_lib):
    inp = synth.make_q4_gemv(seed=N + K, N=N, K=K)
    ref, bound = oracle_lib.q4_gemv(inp["qs"], inp["d"], inp["x"][0])
    assert_close(run_q4(inp), ref, bound, f"q4_gemv {N}x{K}")


def test_q4_gemv_full_size_14336x4096(oracle_lib):
    inp = synth.make_q4_gemv(seed=0, N=14336, K=4096, M=8)
    ref, bound = oracle_lib.q4_gemv_batched(inp["qs"], inp["d"], inp["x"])
    assert_close(run_q4(inp), ref[0], bound[0], "q4_gemv 14336x4096")
    for M in (1, 2, 4, 8):
        assert_close(run_q4(inp, M), ref[:M], bound[:M], f"q4_gemv_batched M={M}")


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_q4_gemv_batched_every_M(M, oracle_lib):
    inp = synth.make_q4_gemv(seed=100 + M, N=517, K=2048, M=M)
    ref, bound = oracle_lib.q4_gemv_batched(inp["qs"], inp["d"], inp["x"])
    assert_close(run_q4(inp, M), ref, bound, f"batched M={M}")


@pytest.mark.parametrize("M", [9, 12, 16])
def test_q4_gemv_batched_wide_M(M, oracle_lib):
    """Batches of 9..16 vectors (staged input up to 16 x 2048 fp32), ragged N, and bit-identity of every row
    with the single-vector call."""
    inp = synth.make_q4_gemv(seed=200 + M, N=3003, K=2048, M=M)
    ref, bound = oracle_lib.q4_gemv_batched(inp["qs"], inp["d"], inp["x"])
    Y = run_q4(inp, M)
    assert_close(Y, ref, bound, f"batched M={M}")
    for t in (0, M // 2, M - 1):
        one = dict(inp, x=inp["x"][t:t + 1])
        assert np.array_equal(run_q4(one).view(np.uint32), Y[t].view(np.uint32)), f"row {t}"


def test_q4_gemv_batched_wide_M_too_large_is_refused():
    qs, d = synth.q4_weights(np.random.default_rng(2), 64, 4096)
    X = torch.zeros(16, 4096, device="cuda")
    Y = torch.empty(16, 64, device="cuda")
    with pytest.raises(q4.Q4Error, match="EUNSUPPORTED"):
        q4.q4_gemv_batched(Y, cu(qs), cu(d), X)


@pytest.mark.parametrize("M", [2, 4, 8])
def test_batched_rows_are_bit_identical_to_single_calls(M):
    """Row t of the batched call equals the single-vector call on x_t, bit for bit: each row keeps its own
    accumulator, summation order and cross-lane reduction tree whatever M is."""
    inp = synth.make_q4_gemv(seed=7, N=14336, K=4096, M=M)
    Y = run_q4(inp, M)
    for t in range(M):
        one = dict(inp, x=inp["x"][t:t + 1])
        assert np.array_equal(run_q4(one).view(np.uint32), Y[t].view(np.uint32)), f"row {t}"


def test_degenerate_blocks(oracle_lib):
    rng = np.random.default_rng(5)
    N, K = 64, 1024
    d = rng.uniform(1e-3, 1e-2, (N, K // 32)).astype(np.float16)
    x = rng.standard_normal((1, K)).astype(np.float32)
    # every code 8: every weight is zero, so the reference is exactly zero with a zero bound; the kernel sums
    # q * x and subtracts 8 * sum(x) per block, so it must land within the absolute part of the tolerance
    inp = dict(qs=np.full((N, K // 32, 16), 0x88, np.uint8), d=d, x=x)
    ref, bound = oracle_lib.q4_gemv(inp["qs"], d, x[0])
    assert np.all(ref == 0.0) and np.all(bound == 0.0)
    assert_close(run_q4(inp), ref, bound, "all codes 8")
    # every code 0: -8 * sum_b d_b * S_b
    inp = dict(qs=np.zeros((N, K // 32, 16), np.uint8), d=d, x=x)
    ref, bound = oracle_lib.q4_gemv(inp["qs"], d, x[0])
    assert_close(run_q4(inp), ref, bound, "all codes 0")
    # large and tiny inputs keep relative accuracy (the staged input is pre-scaled by up to 2^23)
    for scale in (1e20, 1e-30):
        inp = dict(qs=rng.integers(0, 256, (N, K // 32, 16), dtype=np.uint8), d=d, x=(x * scale).astype(np.float32))
        ref, bound = oracle_lib.q4_gemv(inp["qs"], d, inp["x"][0])
        assert_close(run_q4(inp) / scale, ref / scale, bound / scale, f"x scaled by {scale}")
    # blocks of very different magnitude in one vector, and all-zero blocks: each block is staged with its
    # own exponent bound
    xm = x.copy().reshape(K // 32, 32)
    xm[0::4] *= 1e25
    xm[1::4] *= 1e-25
    xm[2::8] = 0.0
    inp = dict(qs=rng.integers(0, 256, (N, K // 32, 16), dtype=np.uint8), d=d, x=xm.reshape(1, K))
    ref, bound = oracle_lib.q4_gemv(inp["qs"], d, inp["x"][0])
    assert_close(run_q4(inp), ref, bound, "mixed block magnitudes")


def test_pure_read_touches_exactly_the_weight_bytes():
    for N, K in ((256, 1024), (14336, 4096), (19, 96)):
        qs, d = synth.q4_weights(np.random.default_rng(N), N, K)
        sink = Guarded(N)
        q4.q4_pure_read(sink.t, cu(qs), cu(d))
        got = sink.result().view(np.uint32)
        words = np.bitwise_xor.reduce(qs.reshape(N, -1).view("<u4"), axis=1)
        scales = np.bitwise_xor.reduce(d.view(np.uint16).astype(np.uint32), axis=1)
        assert np.array_equal(got, words ^ scales)


@pytest.mark.parametrize("N,K", [(256, 1024), (37, 96), (3000, 4096)])
def test_q4_dequant_is_bit_exact(N, K, oracle_lib):
    qs, d = synth.q4_weights(np.random.default_rng(K), N, K)
    W = Guarded(N, K)
    q4.q4_dequant(W.t, cu(qs), cu(d))
    assert np.array_equal(W.result().view(np.uint32), oracle_lib.dequant_q4(qs, d).view(np.uint32))


def test_refusals_on_device():
    qs, d = synth.q4_weights(np.random.default_rng(1), 8, 64)
    X = torch.zeros(17, 64, device="cuda")
    Y = torch.empty(17, 8, device="cuda")
    with pytest.raises(q4.Q4Error, match="outside 1..16"):
        q4.q4_gemv_batched(Y, cu(qs), cu(d), X)


def test_no_fault_bits_after_the_suite():
    assert q4.q4_device_faults() == 0


def _offset_copy(a):
    """The same values in device memory at a 2-byte offset from a 16-byte boundary (a view into a larger
    buffer), so the scales cannot move by 16-byte copies."""
    flat = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).ravel()).to("cuda")
    buf = torch.zeros(flat.numel() + 8, dtype=torch.int16, device="cuda")
    buf[1:1 + flat.numel()] = flat
    return buf[1:1 + flat.numel()].view(torch.float16).view(a.shape)


@pytest.mark.parametrize("M", [1, 2, 8])
def test_unaligned_scales_give_identical_rows(M):
    """Scales that are only 2-byte aligned take the plain-load path into the slot; every row must equal, bit for
    bit, the call with 16-byte aligned scales (same values, same summation order)."""
    inp = synth.make_q4_gemv(seed=31 + M, N=1000, K=4096, M=M)
    qs, X = cu(inp["qs"]), cu(inp["x"][:M])
    d_al, d_un = cu(inp["d"]), _offset_copy(inp["d"])
    assert d_un.data_ptr() % 16 == 2
    Ya, Yu = Guarded(M, 1000), Guarded(M, 1000)
    q4.q4_gemv_batched(Ya.t, qs, d_al, X)
    q4.q4_gemv_batched(Yu.t, qs, d_un, X)
    assert np.array_equal(Ya.result().view(np.uint32), Yu.result().view(np.uint32))
