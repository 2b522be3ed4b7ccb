/*
 * oracle.c -- plain, slow, single-threaded CPU reference for the 4-bit decode GEMVs.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the package's smoke check and the benchmark's CPU-baseline
 * leg are the only callers. The CUDA library never links, loads or calls anything here, and nothing
 * here shares code with it.
 *
 * What it computes, and where each definition comes from:
 *   - binary16 decode: the IEEE 754 binary16 format (1 sign, 5 exponent bits with bias 15,
 *     10 fraction bits; exponent 0 is subnormal, 31 is inf/NaN).
 *   - Q4 block decode: inferencelayer `kernel_lab.rs`, shader `GEMV_F16S` (helpers q4_lo/q4_hi and the
 *     dot pairing of each packed word with x): a 32-weight block is 16 bytes; byte j carries weight j
 *     in its low nibble and weight j+16 in its high nibble; the value is (q - 8) * d with one f16
 *     scale d per block.
 *   - Q4_K super-block decode: trueno-gpu `fused.rs`, FusedRmsNormQ4KGemvKernel, phase 3: a 144-byte
 *     super-block of 256 weights holds f16 d at byte 0, f16 dmin at byte 2, 12 packed 6-bit
 *     scale/min bytes at 4..15 and 128 quant bytes at 16..143. Weight e lives in 64-weight chunk
 *     e/64, byte 32*(e/64) + e%32 of the quant bytes, low nibble when e%64 < 32, else high nibble;
 *     its sub-block is e/32. The value is d*sc*q - dmin*m computed in fp32 (d*sc, then *q, minus
 *     dmin*m). Both products are exact in fp32, so only the subtraction rounds.
 *   - RMSNorm: the same kernel, phases 1-2: r = 1/sqrt(sum(x^2)/K + eps), xhat = x * r * gamma.
 *     Here it runs in fp64.
 *   - GEMV: y[n] = sum_k W[n][k] * xhat[k] in fp64 over the decoded fp32 weights.
 *   - gate+up: trueno-gpu `fused.rs`, FusedGateUpQ4KGemvKernel: two weight matrices against one input.
 *   - MoE: inferencelayer `kernel_lab.rs`, `moe_lab` and the MoE ceiling shader: expert e's rows are
 *     rows e*N .. e*N+N-1 of one stacked store; slot (t, s) uses expert ids[t*topk+s] on token t and
 *     writes output (t*topk+s)*N + r.
 *
 *   - MoE router: spark_model `gemm_quant.rs`, moe_gate_topk_fused: gate[e] = x . Wgate[e] for every
 *     expert (here Wgate is planar Q4, one row per expert), then the top-K experts and their softmax
 *     weights. Reading: softmax over all E logits (max subtracted), the K largest logits in descending
 *     order with ties to the lower expert index, and with `normalize` the K weights divided by their sum.
 *   - SwiGLU: silu(g) * u with silu(g) = g / (1 + exp(-g)) (the standard gated-linear-unit epilogue; the
 *     pages only show that production MoE keeps one value per routed row).
 *
 * Every GEMV entry also returns bound[i] = sum_k |W[n][k]| * |xhat[k]|, the scale of the tolerance
 * the comparisons use.
 *
 * Known defects in the pages that this code does NOT reproduce: the RMSNorm kernel stores rms_inv over
 * staged x[0]; the gate+up kernel skips the per-sub-block scales, reads the nibbles in sequential order
 * and sums eight identical warp results. This oracle uses the true x[0], the full Q4_K decode for both
 * projections and the plain product.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* Element decode                                                                               */
/* ------------------------------------------------------------------------------------------ */

float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 0x1F;
    int fraction = h & 0x3FF;
    double v;
    if (exponent == 0) {
        v = ldexp((double)fraction, -24); /* subnormal: fraction * 2^-14 * 2^-10 */
    } else if (exponent == 31) {
        v = fraction ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + fraction), exponent - 15 - 10);
    }
    return (float)(sign ? -v : v);
}

/* Q4 planar: one row of K weights from its K/32 blocks. */
void oracle_dequant_q4_row(const uint8_t *qs_row, const uint16_t *d_row, int64_t K, float *w)
{
    for (int64_t k = 0; k < K; ++k) {
        int64_t b = k / 32;
        int64_t j = k % 32;
        uint8_t byte = qs_row[b * 16 + (j % 16)];
        int q = (j < 16) ? (byte & 0x0F) : (byte >> 4);
        float d = oracle_f16_to_f32(d_row[b]);
        w[k] = (float)(q - 8) * d; /* at most 15 significant bits: exact */
    }
}

void oracle_dequant_q4(const uint8_t *qs, const uint16_t *d, int64_t N, int64_t K, float *W)
{
    for (int64_t n = 0; n < N; ++n)
        oracle_dequant_q4_row(qs + n * (K / 2), d + n * (K / 32), K, W + n * K);
}

/* Q4_K: 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes s[0..11]. */
void oracle_q4k_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 0x0F) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* Q4_K: one row of K weights from its K/256 super-blocks of 144 bytes. */
void oracle_dequant_q4k_row(const uint8_t *row, int64_t K, float *w)
{
    for (int64_t sb = 0; sb < K / 256; ++sb) {
        const uint8_t *blk = row + sb * 144;
        float d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
        float dmin = oracle_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
        const uint8_t *s = blk + 4;
        const uint8_t *qs = blk + 16;
        for (int e = 0; e < 256; ++e) {
            int j = e / 32;
            int chunk = e / 64;
            uint8_t byte = qs[32 * chunk + e % 32];
            int q = (e % 64 < 32) ? (byte & 0x0F) : (byte >> 4);
            int sc, m;
            oracle_q4k_scale_min(s, j, &sc, &m);
            float scaled = d * (float)sc;  /* exact */
            float value = scaled * (float)q; /* exact */
            float offset = dmin * (float)m;  /* exact */
            w[sb * 256 + e] = value - offset; /* the one rounding */
        }
    }
}

void oracle_dequant_q4k(const uint8_t *w, int64_t N, int64_t K, float *W)
{
    for (int64_t n = 0; n < N; ++n)
        oracle_dequant_q4k_row(w + n * (K / 256) * 144, K, W + n * K);
}

/* ------------------------------------------------------------------------------------------ */
/* Dot products                                                                                 */
/* ------------------------------------------------------------------------------------------ */

static void dot_f32x(const float *w, const float *x, int64_t K, double *y, double *bound)
{
    double acc = 0.0, b = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        acc += (double)w[k] * (double)x[k];
        b += fabs((double)w[k]) * fabs((double)x[k]);
    }
    *y = acc;
    *bound = b;
}

static void dot_f64x(const float *w, const double *x, int64_t K, double *y, double *bound)
{
    double acc = 0.0, b = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        acc += (double)w[k] * x[k];
        b += fabs((double)w[k]) * fabs(x[k]);
    }
    *y = acc;
    *bound = b;
}

/* Y[m][n] = sum_k W[n][k] * X[m][k] for m < M (M = 1 is the single GEMV). */
int oracle_q4_gemv_batched(const uint8_t *qs, const uint16_t *d, const float *X, int64_t M, int64_t N,
                           int64_t K, double *Y, double *bound)
{
    float *w = (float *)malloc((size_t)K * sizeof(float));
    if (!w) return -1;
    for (int64_t n = 0; n < N; ++n) {
        oracle_dequant_q4_row(qs + n * (K / 2), d + n * (K / 32), K, w);
        for (int64_t m = 0; m < M; ++m)
            dot_f32x(w, X + m * K, K, &Y[m * N + n], &bound[m * N + n]);
    }
    free(w);
    return 0;
}

/* xhat[k] = x[k] * r * gamma[k], r = 1 / sqrt(sum(x^2) / K + eps), all in fp64. */
void oracle_rmsnorm(const float *x, const float *gamma, float eps, int64_t K, double *xhat)
{
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) ss += (double)x[k] * (double)x[k];
    double r = 1.0 / sqrt(ss / (double)K + (double)eps);
    for (int64_t k = 0; k < K; ++k) xhat[k] = (double)x[k] * r * (double)gamma[k];
}

/* y[n] = sum_k W[n][k] * xhat[k] over Q4_K rows, xhat in fp64. */
int oracle_q4k_gemv(const uint8_t *w, const double *xhat, int64_t N, int64_t K, double *y, double *bound)
{
    float *row = (float *)malloc((size_t)K * sizeof(float));
    if (!row) return -1;
    for (int64_t n = 0; n < N; ++n) {
        oracle_dequant_q4k_row(w + n * (K / 256) * 144, K, row);
        dot_f64x(row, xhat, K, &y[n], &bound[n]);
    }
    free(row);
    return 0;
}

int oracle_fused_rmsnorm_q4k_gemv(const uint8_t *w, const float *x, const float *gamma, float eps,
                                  int64_t N, int64_t K, double *y, double *bound)
{
    double *xhat = (double *)malloc((size_t)K * sizeof(double));
    if (!xhat) return -1;
    oracle_rmsnorm(x, gamma, eps, K, xhat);
    int rc = oracle_q4k_gemv(w, xhat, N, K, y, bound);
    free(xhat);
    return rc;
}

/* gamma == NULL: no normalisation, xhat = x. */
int oracle_fused_gateup_q4k_gemv(const uint8_t *w_gate, const uint8_t *w_up, const float *x,
                                 const float *gamma, float eps, int64_t N, int64_t K, double *y_gate,
                                 double *y_up, double *bound_gate, double *bound_up)
{
    double *xhat = (double *)malloc((size_t)K * sizeof(double));
    if (!xhat) return -1;
    if (gamma) {
        oracle_rmsnorm(x, gamma, eps, K, xhat);
    } else {
        for (int64_t k = 0; k < K; ++k) xhat[k] = (double)x[k];
    }
    int rc = oracle_q4k_gemv(w_gate, xhat, N, K, y_gate, bound_gate);
    if (rc == 0) rc = oracle_q4k_gemv(w_up, xhat, N, K, y_up, bound_up);
    free(xhat);
    return rc;
}

/*
 * MoE gate and up: for token t and slot s, expert e = ids[t*topk+s];
 * y_gate[(t*topk+s)*N + r] = sum_k Wgate[e*N + r][k] * x[t][k], likewise for up.
 * A slot whose id is outside [0, E) gets NaN outputs (and NaN bounds).
 */
int oracle_moe_q4_gemv(const uint8_t *qs_gate, const uint16_t *d_gate, const uint8_t *qs_up,
                       const uint16_t *d_up, const float *x, const int32_t *ids, int64_t T, int64_t topk,
                       int64_t E, int64_t N, int64_t K, double *y_gate, double *y_up, double *bound_gate,
                       double *bound_up)
{
    float *w = (float *)malloc((size_t)K * sizeof(float));
    if (!w) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t s = 0; s < topk; ++s) {
            int64_t slot = t * topk + s;
            int64_t e = ids[slot];
            for (int64_t r = 0; r < N; ++r) {
                int64_t o = slot * N + r;
                if (e < 0 || e >= E) {
                    y_gate[o] = y_up[o] = bound_gate[o] = bound_up[o] = NAN;
                    continue;
                }
                int64_t row = e * N + r;
                oracle_dequant_q4_row(qs_gate + row * (K / 2), d_gate + row * (K / 32), K, w);
                dot_f32x(w, x + t * K, K, &y_gate[o], &bound_gate[o]);
                oracle_dequant_q4_row(qs_up + row * (K / 2), d_up + row * (K / 32), K, w);
                dot_f32x(w, x + t * K, K, &y_up[o], &bound_up[o]);
            }
        }
    }
    free(w);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Epilogue and router                                                                          */
/* ------------------------------------------------------------------------------------------ */

double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* y[i] = silu(g[i]) * u[i] in fp64. */
void oracle_swiglu(const double *g, const double *u, int64_t n, double *y)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_silu(g[i]) * u[i];
}

/* Selection order of the top-K: a ranks above b when a > b, and a NaN ranks below every other value. */
static int ranks_above(double a, double b)
{
    if (isnan(a)) return 0;
    return isnan(b) || a > b;
}

/*
 * Top-K softmax of one row of E logits (given as float or double through `get`): ids[0..topk) are the
 * indices of the topk largest logits in descending order (ties, including two NaNs: lower index first; a NaN
 * below every other value); weights[i] is the softmax probability of ids[i] over all E logits (NaN for every
 * pick when any logit is NaN), divided by the sum of the topk probabilities when `normalize` is non-zero.
 * Plain selection: topk passes over the logits.
 */
static void topk_softmax_row(const double *lg, int64_t E, int64_t topk, int normalize, int32_t *ids, double *weights)
{
    double mx = -INFINITY;
    for (int64_t e = 0; e < E; ++e)
        if (lg[e] > mx) mx = lg[e];
    double z = 0.0;
    for (int64_t e = 0; e < E; ++e) z += exp(lg[e] - mx);
    for (int64_t i = 0; i < topk; ++i) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            int taken = 0;
            for (int64_t j = 0; j < i; ++j)
                if (ids[j] == e) taken = 1;
            if (taken) continue;
            if (best < 0 || ranks_above(lg[e], lg[best])) best = e;
        }
        ids[i] = (int32_t)best;
        weights[i] = exp(lg[best] - mx) / z;
    }
    if (normalize) {
        double s = 0.0;
        for (int64_t i = 0; i < topk; ++i) s += weights[i];
        for (int64_t i = 0; i < topk; ++i) weights[i] /= s;
    }
}

/* Top-K softmax over T rows of fp32 logits [T][E] (the selection made on exactly these values). */
void oracle_topk_softmax_f32(const float *logits, int64_t T, int64_t E, int64_t topk, int normalize,
                             int32_t *ids, double *weights)
{
    double *row = (double *)malloc((size_t)E * sizeof(double));
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) row[e] = (double)logits[t * E + e];
        topk_softmax_row(row, E, topk, normalize, ids + t * topk, weights + t * topk);
    }
    free(row);
}

/*
 * MoE router: logits[t][e] = sum_k Wgate[e][k] * x[t][k] (planar Q4, E rows of K), with bounds, then
 * top-K softmax of each token's fp64 logits.
 */
int oracle_moe_router(const uint8_t *qs, const uint16_t *d, const float *x, int64_t T, int64_t E, int64_t K,
                      int64_t topk, int normalize, double *logits, double *bound, int32_t *ids, double *weights)
{
    int rc = oracle_q4_gemv_batched(qs, d, x, T, E, K, logits, bound);
    if (rc) return rc;
    for (int64_t t = 0; t < T; ++t) topk_softmax_row(logits + t * E, E, topk, normalize, ids + t * topk, weights + t * topk);
    return 0;
}
