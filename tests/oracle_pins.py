"""Pins of the oracle to facts other than its own code.

Each ``pin_*`` function takes a loaded :class:`oracle.Oracle` and raises ``AssertionError`` when the
oracle disagrees with something the pages or the mathematics fix: hand-worked examples stored under
``tests/golden/`` (each with its source), closed forms on hand-built blocks, exact rational arithmetic,
invariants, and special cases that reduce to a library routine (numpy's binary16 decode, a dense
float64 matmul). ``test_oracle_pins.py`` runs them against the real oracle; ``test_oracle_mutations.py``
runs them against deliberately broken copies of it and checks that every plausible mistake is caught.
"""

from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------------------------
# fixture readers and hand-building helpers (test side; independent of the oracle's code)
# ---------------------------------------------------------------------------------------------

def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line


def read_scale_min_example():
    byts, table = None, {}
    for line in _rows("q4k_scale_min_example.txt"):
        if line.startswith("bytes:"):
            byts = np.array([int(t, 16) for t in line.split(":", 1)[1].split()], np.uint8)
        else:
            j, sc, m = (int(t) for t in line.split())
            table[j] = (sc, m)
    return byts, table


def read_positions(name):
    return [(int(b), h, int(e)) for b, h, e in (line.split() for line in _rows(name))]


def pack_scale_min(sc, m):
    """Pack eight 6-bit (scale, min) pairs into 12 bytes: the inverse of the page's unpack rule.

    Bytes 0-3: low 6 bits = scale 0-3, top 2 bits = scale 4-7 >> 4. Bytes 4-7: low 6 bits = min 0-3,
    top 2 bits = min 4-7 >> 4. Bytes 8-11: low nibble = scale 4-7 & 15, high nibble = min 4-7 & 15.
    """
    s = np.zeros(12, np.int64)
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return s.astype(np.uint8)


def f16_bytes(v):
    return np.array([v], dtype="<f2").view(np.uint8)


def q4k_block(d, dmin, sc, m, qbytes):
    blk = np.zeros(144, np.uint8)
    blk[0:2] = f16_bytes(d)
    blk[2:4] = f16_bytes(dmin)
    blk[4:16] = pack_scale_min(sc, m)
    blk[16:144] = qbytes
    return blk


def tol_ok(y, ref, bound):
    return np.all(np.abs(np.asarray(y, np.float64) - ref) <= 1e-3 * bound + 1e-5)


# ---------------------------------------------------------------------------------------------
# element decode
# ---------------------------------------------------------------------------------------------

def pin_f16_decode(o):
    """All 65536 binary16 codes decode as numpy's IEEE binary16 conversion does."""
    codes = np.arange(65536, dtype=np.uint32)
    ref = codes.astype(np.uint16).view(np.float16).astype(np.float32)
    got = np.array([o.f16_to_f32(int(c)) for c in codes[::1]], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_q4_nibble_positions(o):
    """A lone non-neutral nibble lands on the weight the page's dot pairing gives it."""
    for byte, half, weight in read_positions("q4_nibble_positions.txt"):
        qs = np.full((1, 1, 16), 0x88, np.uint8)  # every code 8 -> weight 0
        qs[0, 0, byte] = (0x8F if half == "lo" else 0xF8)  # code 15 -> 7*d
        d = np.array([[1.0]], np.float16)
        W = o.dequant_q4(qs, d)[0]
        expect = np.zeros(32, np.float32)
        expect[weight] = 7.0
        assert np.array_equal(W, expect), (byte, half, weight, W)


def pin_q4_closed_forms(o):
    """Hand-built Q4 rows: all codes 8 give 0, all codes 0 give -8*sum_b d_b*S_b, one code gives one product."""
    rng = np.random.default_rng(11)
    N, K = 3, 256
    d = rng.uniform(1e-3, 1e-2, size=(N, K // 32)).astype(np.float16)
    x = rng.standard_normal(K).astype(np.float32)

    y, _ = o.q4_gemv(np.full((N, K // 32, 16), 0x88, np.uint8), d, x)
    assert np.all(y == 0.0)

    y, _ = o.q4_gemv(np.zeros((N, K // 32, 16), np.uint8), d, x)
    S = x.astype(np.float64).reshape(-1, 32).sum(axis=1)
    expect = -8.0 * (d.astype(np.float64) * S).sum(axis=1)
    assert np.allclose(y, expect, rtol=1e-12, atol=1e-12)

    # one weight: block 5, byte 9 high nibble -> weight 5*32 + 25, code 3 -> (3-8)*d
    qs = np.full((1, K // 32, 16), 0x88, np.uint8)
    qs[0, 5, 9] = 0x38
    y, _ = o.q4_gemv(qs, d[:1], x)
    assert y[0] == (-5.0 * float(d[0, 5])) * float(x[5 * 32 + 25])


def pin_q4_scale_power_of_two(o):
    """Doubling every f16 scale doubles every weight and every output exactly."""
    rng = np.random.default_rng(12)
    qs, d = synth.q4_weights(rng, 5, 128)
    x = rng.standard_normal(128).astype(np.float32)
    W1, W2 = o.dequant_q4(qs, d), o.dequant_q4(qs, (d.astype(np.float32) * 2).astype(np.float16))
    assert np.array_equal(W2, 2 * W1)
    y1, _ = o.q4_gemv(qs, d, x)
    y2, _ = o.q4_gemv(qs, (d.astype(np.float32) * 2).astype(np.float16), x)
    assert np.array_equal(y2, 2 * y1)


def pin_q4k_scale_min_example(o):
    """The hand-worked 12-byte example decodes to the hand-worked table."""
    byts, table = read_scale_min_example()
    for j in range(8):
        assert o.q4k_scale_min(byts, j) == table[j], (j, o.q4k_scale_min(byts, j), table[j])


def pin_q4k_scale_min_roundtrip(o):
    """Every (scale, min) in 0..63 x 0..63 at every sub-block position survives pack -> unpack."""
    rng = np.random.default_rng(13)
    grid = np.arange(64)
    for j in range(8):
        for sc_v in grid:
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            sc[j] = sc_v
            for m_v in grid[rng.permutation(64)[:8]]:
                m[j] = m_v
                s = pack_scale_min(sc, m)
                for jj in range(8):
                    assert o.q4k_scale_min(s, jj) == (int(sc[jj]), int(m[jj])), (j, jj)
    # and the full grid at one position, exhaustively
    for j in (0, 3, 4, 7):
        for sc_v in grid:
            for m_v in grid:
                sc = np.zeros(8, np.int64)
                m = np.zeros(8, np.int64)
                sc[j], m[j] = sc_v, m_v
                assert o.q4k_scale_min(pack_scale_min(sc, m), j) == (sc_v, m_v)


def pin_q4k_qs_positions(o):
    """With scale 1, min 0, d = 1: a lone nibble of code 9 lands on the page's weight index."""
    for byte, half, weight in read_positions("q4k_qs_positions.txt"):
        q = np.zeros(128, np.uint8)
        q[byte] = 0x09 if half == "lo" else 0x90
        blk = q4k_block(1.0, 1.0, [1] * 8, [0] * 8, q)
        W = o.dequant_q4k(blk.reshape(1, 1, 144))[0]
        expect = np.zeros(256, np.float32)
        expect[weight] = 9.0
        assert np.array_equal(W, expect), (byte, half, weight)


def pin_q4k_closed_forms(o):
    """Scale 1 and min 0 give d*q; codes 0 give -dmin*m per sub-block."""
    rng = np.random.default_rng(14)
    q = rng.integers(0, 256, 128).astype(np.uint8)
    W = o.dequant_q4k(q4k_block(0.5, 0.25, [1] * 8, [0] * 8, q).reshape(1, 1, 144))[0]
    lo, hi = (q & 15).astype(np.float32), (q >> 4).astype(np.float32)
    # weights of chunk c: low nibbles of its 32 bytes, then their high nibbles
    expect = np.concatenate([np.concatenate([lo[32 * c:32 * c + 32], hi[32 * c:32 * c + 32]]) for c in range(4)])
    assert np.array_equal(W, 0.5 * expect)

    m = [0, 1, 7, 63, 31, 32, 5, 60]
    W = o.dequant_q4k(q4k_block(0.5, 0.125, [9] * 8, m, np.zeros(128, np.uint8)).reshape(1, 1, 144))[0]
    assert np.array_equal(W, np.repeat(-0.125 * np.array(m, np.float32), 32))


def _round_f32(exact: Fraction) -> np.float32:
    dbl = float(exact)
    assert Fraction(dbl) == exact  # exact in binary64, so one rounding to binary32 follows
    return np.float32(dbl)


def pin_q4k_dequant_exact_rounding(o):
    """Each weight equals d*sc*q - dmin*m in exact arithmetic, rounded once to fp32."""
    rng = np.random.default_rng(15)
    for _ in range(40):
        d, dmin = (np.float16(rng.uniform(1e-3, 1e-2)) for _ in range(2))
        sc, m = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
        qlo, qhi = rng.integers(0, 16, 4), rng.integers(0, 16, 4)
        qbytes = np.concatenate([np.full(32, (qhi[c] << 4) | qlo[c], np.uint8) for c in range(4)])
        W = o.dequant_q4k(q4k_block(d, dmin, sc, m, qbytes).reshape(1, 1, 144))[0]
        for j in range(8):
            qv = qlo[j // 2] if j % 2 == 0 else qhi[j // 2]
            exact = Fraction(float(d)) * int(sc[j]) * int(qv) - Fraction(float(dmin)) * int(m[j])
            ref = _round_f32(exact)
            assert np.all(W[32 * j:32 * j + 32].view(np.uint32) == ref.view(np.uint32)), (j, W[32 * j], ref)


# ---------------------------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------------------------

def pin_rmsnorm_closed_forms(o):
    """Constant input, unit-RMS input, the K divisor and linearity in gamma."""
    K, eps = 384, 1e-5
    ones = np.ones(K, np.float32)
    for c in (0.5, -3.0, 1e-3):
        xh = o.rmsnorm(np.full(K, c, np.float32), ones, eps)
        expect = float(np.float32(c)) / np.sqrt(float(np.float32(c)) ** 2 + float(np.float32(eps)))
        assert np.allclose(xh, expect, rtol=1e-14, atol=0)

    # mean of squares exactly 1 - eps: output equals input up to fp64 rounding
    e32 = float(np.float32(eps))
    a = np.float32(np.sqrt(1.0 - e32))
    x = np.where(np.arange(K) % 2 == 0, a, -a).astype(np.float32)
    xh = o.rmsnorm(x, ones, eps)
    ms = float(np.mean(np.float64(x) ** 2))
    expect = np.float64(x) / np.sqrt(ms + e32)
    assert np.allclose(xh, expect, rtol=1e-14) and np.allclose(xh, x, rtol=1e-6)

    # the divisor is K: one non-zero entry a among K gives a / sqrt(a^2/K + eps)
    x = np.zeros(K, np.float32)
    x[7] = 2.0
    xh = o.rmsnorm(x, ones, eps)
    assert np.isclose(xh[7], 2.0 / np.sqrt(4.0 / K + e32), rtol=1e-14) and np.all(np.delete(xh, 7) == 0)

    rng = np.random.default_rng(16)
    x = rng.standard_normal(K).astype(np.float32)
    g = rng.normal(1.0, 0.1, K).astype(np.float32)
    assert np.allclose(o.rmsnorm(x, 2 * g, eps), 2 * o.rmsnorm(x, g, eps), rtol=1e-15, atol=0)


# ---------------------------------------------------------------------------------------------
# GEMVs against a dense float64 matmul of the decoded weights
# ---------------------------------------------------------------------------------------------

def pin_q4_gemv_matmul(o):
    rng = np.random.default_rng(17)
    for N, K, M in ((1, 32, 1), (7, 96, 3), (33, 512, 8), (64, 64, 2)):
        qs, d = synth.q4_weights(rng, N, K)
        X = rng.standard_normal((M, K)).astype(np.float32)
        W = o.dequant_q4(qs, d).astype(np.float64)
        Y, B = o.q4_gemv_batched(qs, d, X)
        assert np.allclose(Y, X.astype(np.float64) @ W.T, rtol=1e-12, atol=1e-12)
        assert np.allclose(B, np.abs(X.astype(np.float64)) @ np.abs(W).T, rtol=1e-12)
        for t in range(M):  # batched row t is the single call on x_t, bit for bit
            y, b = o.q4_gemv(qs, d, X[t])
            assert np.array_equal(y, Y[t]) and np.array_equal(b, B[t])


def pin_q4k_gemv_matmul(o):
    rng = np.random.default_rng(18)
    for N, K in ((1, 256), (5, 768), (17, 512)):
        w = synth.q4k_weights(rng, N, K)
        x = rng.standard_normal(K).astype(np.float32)
        g = rng.normal(1.0, 0.1, K).astype(np.float32)
        W = o.dequant_q4k(w).astype(np.float64)
        xh = o.rmsnorm(x, g, 1e-5)
        y, b = o.fused_rmsnorm_q4k_gemv(w, x, g, 1e-5)
        assert np.allclose(y, W @ xh, rtol=1e-12, atol=1e-12)
        assert np.allclose(b, np.abs(W) @ np.abs(xh), rtol=1e-12)


def pin_gateup(o):
    rng = np.random.default_rng(19)
    N, K = 9, 512
    wg, wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x = rng.standard_normal(K).astype(np.float32)
    g = rng.normal(1.0, 0.1, K).astype(np.float32)
    Wg, Wu = o.dequant_q4k(wg).astype(np.float64), o.dequant_q4k(wu).astype(np.float64)
    (yg, _), (yu, _) = o.fused_gateup_q4k_gemv(wg, wu, x, None, 1e-5)
    assert np.allclose(yg, Wg @ x.astype(np.float64), rtol=1e-12, atol=1e-12)
    assert np.allclose(yu, Wu @ x.astype(np.float64), rtol=1e-12, atol=1e-12)
    (yg, _), (yu, _) = o.fused_gateup_q4k_gemv(wg, wu, x, g, 1e-5)
    xh = o.rmsnorm(x, g, 1e-5)
    assert np.allclose(yg, Wg @ xh, rtol=1e-12, atol=1e-12)
    assert np.allclose(yu, Wu @ xh, rtol=1e-12, atol=1e-12)


def pin_moe(o):
    """Each routed slot is its expert's slice times its token; expert relabelling changes nothing."""
    rng = np.random.default_rng(20)
    E, N, K, T, topk = 6, 5, 128, 3, 4
    qg, dg = synth.q4_weights(rng, E * N, K)
    qu, du = synth.q4_weights(rng, E * N, K)
    x = rng.standard_normal((T, K)).astype(np.float32)
    ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(T)]).astype(np.int32)
    Wg = o.dequant_q4(qg, dg).astype(np.float64).reshape(E, N, K)
    Wu = o.dequant_q4(qu, du).astype(np.float64).reshape(E, N, K)
    (yg, bg), (yu, bu) = o.moe_q4_gemv(qg, dg, qu, du, x, ids, E)
    for t in range(T):
        for s in range(topk):
            e = ids[t, s]
            assert np.allclose(yg[t, s], Wg[e] @ x[t], rtol=1e-12, atol=1e-12)
            assert np.allclose(yu[t, s], Wu[e] @ x[t], rtol=1e-12, atol=1e-12)
    perm = rng.permutation(E)  # expert e moves to position perm[e]
    inv = np.argsort(perm)
    rows = lambda a: a.reshape(E, N, *a.shape[1:])[inv].reshape(a.shape)  # noqa: E731
    (yg2, _), (yu2, _) = o.moe_q4_gemv(rows(qg), rows(dg), rows(qu), rows(du), x, perm[ids].astype(np.int32), E)
    assert np.array_equal(yg, yg2) and np.array_equal(yu, yu2)
    bad = ids.copy()
    bad[1, 2] = E
    (yg3, _), (yu3, _) = o.moe_q4_gemv(qg, dg, qu, du, x, bad, E)
    assert np.all(np.isnan(yg3[1, 2])) and np.all(np.isnan(yu3[1, 2]))
    keep = np.ones((T, topk), bool)
    keep[1, 2] = False
    assert np.array_equal(yg3[keep], yg[keep])


def pin_silu(o):
    """silu against the logistic function of a library (scipy.special.expit), its odd-part identity
    silu(x) - silu(-x) = x, its value and slope at 0 and its limits."""
    from scipy.special import expit

    assert o.silu(0.0) == 0.0
    xs = np.concatenate([np.linspace(-30, 30, 241), [1e-8, -1e-8, 0.5, -0.5, 7.25]])
    for x in xs:
        v = o.silu(x)
        assert abs(v - x * float(expit(x))) <= 1e-15 * max(1.0, abs(x)), x
        assert abs((v - o.silu(-x)) - x) <= 4e-16 * max(1.0, abs(x)), x
    h = 1e-6
    assert abs((o.silu(h) - o.silu(-h)) / (2 * h) - 0.5) < 1e-9  # slope 1/2 at 0
    assert o.silu(80.0) == 80.0 and -1e-30 < o.silu(-80.0) < 0.0


def pin_swiglu(o):
    """swiglu(g, u) is silu(g) in the first argument and linear in the second."""
    rng = np.random.default_rng(30)
    g = rng.standard_normal(64) * 4
    u = rng.standard_normal(64)
    y = o.swiglu(g, u)
    assert np.array_equal(o.swiglu(g, np.ones(64)), np.array([o.silu(v) for v in g]))
    assert np.array_equal(o.swiglu(g, 2 * u), 2 * y)
    assert np.array_equal(o.swiglu(g, np.zeros(64)), np.zeros(64))
    assert np.array_equal(o.swiglu(np.zeros(64), u), np.zeros(64))


def pin_topk_softmax(o):
    """Top-K softmax: a hand-worked example with a tie, then random rows against a stable argsort and the
    softmax of a library (scipy.special.softmax), with and without renormalisation."""
    from scipy.special import softmax

    lg = np.array([[0.5, 2.0, -1.0, 2.0, 1.5]], np.float32)
    ids, w = o.topk_softmax_f32(lg, 3, False)
    assert ids.tolist() == [[1, 3, 4]]  # 2.0 (index 1, then index 3), then 1.5
    p = np.exp(lg[0].astype(np.float64) - 2.0)
    p /= p.sum()
    assert np.allclose(w[0], p[[1, 3, 4]], rtol=1e-15, atol=0)
    ids2, w2 = o.topk_softmax_f32(lg, 3, True)
    assert ids2.tolist() == [[1, 3, 4]] and np.allclose(w2[0], p[[1, 3, 4]] / p[[1, 3, 4]].sum(), rtol=1e-15)
    # NaN ranks below every other value (-inf included), two NaNs tie to the lower index, -0 ties with +0, and a
    # NaN anywhere makes every softmax weight NaN (worked by hand)
    nan = np.float32(np.nan)
    ids3, w3 = o.topk_softmax_f32(np.array([[nan, 1.0, -np.inf, 1.0, nan]], np.float32), 5, False)
    assert ids3.tolist() == [[1, 3, 2, 0, 4]] and np.all(np.isnan(w3))
    ids4, _ = o.topk_softmax_f32(np.array([[nan, 2.0, nan, -3.0]], np.float32), 2, True)
    assert ids4.tolist() == [[1, 3]]
    ids5, w5 = o.topk_softmax_f32(np.array([[-0.0, 0.0, -1.0]], np.float32), 2, False)
    assert ids5.tolist() == [[0, 1]] and np.allclose(w5[0], np.exp([0.0, 0.0]) / (2 + np.exp(-1.0)), rtol=1e-15)
    rng = np.random.default_rng(31)
    for E, K in ((64, 8), (16, 2), (7, 7), (128, 1)):
        L = (rng.standard_normal((5, E)) * 3).astype(np.float32)
        L[0, 3] = L[0, 5]  # a tie
        for norm in (False, True):
            ids, w = o.topk_softmax_f32(L, K, norm)
            for t in range(5):
                order = np.argsort(-L[t].astype(np.float64), kind="stable")[:K]
                assert ids[t].tolist() == order.tolist()
                pt = softmax(L[t].astype(np.float64))[order]
                if norm:
                    pt = pt / pt.sum()
                assert np.allclose(w[t], pt, rtol=1e-13, atol=0)


def pin_router(o):
    """Router logits are the dense product of the decoded router rows; ids and weights are the top-K
    softmax of those logits (stable argsort, library softmax)."""
    from scipy.special import softmax

    rng = np.random.default_rng(32)
    E, K, T, topk = 16, 256, 3, 4
    qs, d = synth.q4_weights(rng, E, K)
    x = rng.standard_normal((T, K)).astype(np.float32)
    W = o.dequant_q4(qs, d).astype(np.float64)
    lg, bd, ids, w = o.moe_router(qs, d, x, topk, True)
    assert np.allclose(lg, x.astype(np.float64) @ W.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(bd, np.abs(x.astype(np.float64)) @ np.abs(W).T, rtol=1e-12)
    for t in range(T):
        order = np.argsort(-lg[t], kind="stable")[:topk]
        assert ids[t].tolist() == order.tolist()
        pt = softmax(lg[t])[order]
        assert np.allclose(w[t], pt / pt.sum(), rtol=1e-13)


ALL_PINS = [
    pin_f16_decode,
    pin_q4_nibble_positions,
    pin_q4_closed_forms,
    pin_q4_scale_power_of_two,
    pin_q4k_scale_min_example,
    pin_q4k_scale_min_roundtrip,
    pin_q4k_qs_positions,
    pin_q4k_closed_forms,
    pin_q4k_dequant_exact_rounding,
    pin_rmsnorm_closed_forms,
    pin_q4_gemv_matmul,
    pin_q4k_gemv_matmul,
    pin_gateup,
    pin_moe,
    pin_silu,
    pin_swiglu,
    pin_topk_softmax,
    pin_router,
]
