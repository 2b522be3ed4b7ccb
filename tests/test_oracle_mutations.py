"""Each plausible mistake planted in a copy of the oracle's C source must make some pin fail.

The mutants are compiled on the CPU into a temporary directory; the real oracle is untouched. Every
mutation keeps all memory accesses in bounds, so a mutant can only compute a wrong value.
"""

import os

import pytest

import oracle
from oracle import build as oracle_build
import oracle_pins

# (name, text in oracle.c, replacement)
MUTATIONS = [
    ("silu sign", "return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    ("swiglu uses u twice", "y[i] = oracle_silu(g[i]) * u[i];", "y[i] = oracle_silu(u[i]) * u[i];"),
    ("top-k ties to the higher index", "return isnan(b) || a > b;", "return isnan(b) || a >= b;"),
    ("top-k NaN ranked by plain comparison", "if (best < 0 || ranks_above(lg[e], lg[best])) best = e;",
     "if (best < 0 || lg[e] > lg[best]) best = e;"),
    ("top-k NaN ranked first", "    if (isnan(a)) return 0;", "    if (isnan(a)) return 1;"),
    ("top-k weights not renormalised", "for (int64_t i = 0; i < topk; ++i) weights[i] /= s;",
     "for (int64_t i = 0; i < topk; ++i) weights[i] /= 1.0;"),
    ("softmax over the top-k only", "weights[i] = exp(lg[best] - mx) / z;", "weights[i] = exp(lg[best] - mx);"),
    ("q4 nibble halves swapped", "int q = (j < 16) ? (byte & 0x0F) : (byte >> 4);",
     "int q = (j < 16) ? (byte >> 4) : (byte & 0x0F);"),
    ("q4 sequential byte order", "qs_row[b * 16 + (j % 16)]", "qs_row[b * 16 + (j / 2)]"),
    ("q4 bias dropped", "w[k] = (float)(q - 8) * d;", "w[k] = (float)(q) * d;"),
    ("q4 wrong scale index", "float d = oracle_f16_to_f32(d_row[b]);", "float d = oracle_f16_to_f32(d_row[0]);"),
    ("q4k high-scale bits from s[j]", "*sc = (s[j + 4] & 0x0F) | ((s[j - 4] >> 6) << 4);",
     "*sc = (s[j + 4] & 0x0F) | ((s[j] >> 6) << 4);"),
    ("q4k high-min bits from s[j-4]", "*m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);",
     "*m = (s[j + 4] >> 4) | ((s[j - 4] >> 6) << 4);"),
    ("q4k low min from s[j+8]", "*m = s[j + 4] & 63;", "*m = s[j + 8 - 4 * (j > 3)] & 63;"),
    ("q4k scale nibble high/low swapped", "*sc = (s[j + 4] & 0x0F)", "*sc = (s[j + 4] >> 4)"),
    ("q4k min term dropped", "w[sb * 256 + e] = value - offset;", "w[sb * 256 + e] = value;"),
    ("q4k min term sign", "w[sb * 256 + e] = value - offset;", "w[sb * 256 + e] = value + offset;"),
    ("q4k sequential quant bytes", "uint8_t byte = qs[32 * chunk + e % 32];",
     "uint8_t byte = qs[e / 2]; (void)chunk;"),
    ("q4k nibble halves swapped", "int q = (e % 64 < 32) ? (byte & 0x0F) : (byte >> 4);",
     "int q = (e % 64 < 32) ? (byte >> 4) : (byte & 0x0F);"),
    ("q4k sub-block index by 16", "int j = e / 32;", "int j = (e / 16) % 8;"),
    ("q4k d and dmin swapped", "float d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));",
     "float d = oracle_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));"),
    ("f16 subnormal exponent", "v = ldexp((double)fraction, -24);", "v = ldexp((double)fraction, -25);"),
    ("f16 exponent bias", "exponent - 15 - 10", "exponent - 14 - 10"),
    ("rmsnorm eps outside sqrt", "double r = 1.0 / sqrt(ss / (double)K + (double)eps);",
     "double r = 1.0 / (sqrt(ss / (double)K) + (double)eps);"),
    ("rmsnorm divisor K-1", "double r = 1.0 / sqrt(ss / (double)K + (double)eps);",
     "double r = 1.0 / sqrt(ss / (double)(K - 1) + (double)eps);"),
    ("rmsnorm gamma dropped", "xhat[k] = (double)x[k] * r * (double)gamma[k];", "xhat[k] = (double)x[k] * r;"),
    ("batched output transposed", "dot_f32x(w, X + m * K, K, &Y[m * N + n], &bound[m * N + n]);",
     "dot_f32x(w, X + m * K, K, &Y[n * M + m], &bound[n * M + m]);"),
    ("bound not absolute", "b += fabs((double)w[k]) * fabs((double)x[k]);",
     "b += (double)w[k] * (double)x[k];"),
    ("moe expert rows interleaved", "int64_t row = e * N + r;", "int64_t row = e + r * E;"),
    ("moe wrong token", "dot_f32x(w, x + t * K, K, &y_gate[o], &bound_gate[o]);",
     "dot_f32x(w, x + ((t + 1) % T) * K, K, &y_gate[o], &bound_gate[o]);"),
    ("moe output transposed", "int64_t o = slot * N + r;", "int64_t o = r * (T * topk) + slot;"),
    ("gateup up uses gate weights", "if (rc == 0) rc = oracle_q4k_gemv(w_up, xhat",
     "if (rc == 0) rc = oracle_q4k_gemv(w_gate, xhat"),
    ("gateup gamma ignored", "    if (gamma) {\n        oracle_rmsnorm", "    if (0) {\n        oracle_rmsnorm"),
]


def _first_failing_pin(o):
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            return pin.__name__
    return None


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    with open(oracle_build.SOURCE) as f:
        src = f.read()
    assert old in src, f"mutation target not found: {old!r}"
    mutated = src.replace(old, new)
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle_build.build(source=path, out=os.path.join(tmp_path, "libmutant.so"))
    caught_by = _first_failing_pin(oracle.Oracle(lib))
    assert caught_by is not None, f"no pin catches: {name}"
