/*
 * q4gemv.h -- C ABI of a GB300 (sm_103a) library of memory-bound decode GEMVs over 4-bit block-quantized
 * weights.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers are DEVICE pointers owned by the caller; the library never allocates, frees or keeps
 *    them. Outputs must not overlap inputs.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream) and returns
 *    as soon as the work is enqueued. Inputs must stay valid and unmodified until the work completes.
 *  - Return value: Q4_OK (0) when the work was enqueued, otherwise a negative code; nothing is enqueued when
 *    an argument is refused. The library refuses out-of-range arguments instead of clamping them.
 *      Q4_EINVAL       null required pointer, a size <= 0, M outside 1..16, K not a multiple of the block
 *                      size (32 for Q4, 256 for Q4_K), topk > E, eps negative or not finite
 *      Q4_EALIGN       a pointer below the alignment stated for it
 *      Q4_ECUDA        a CUDA call failed (launch error, no device, ...)
 *      Q4_EUNSUPPORTED the current device is not sm_103, or the staged input (M*K*4 bytes, T*K*4 for MoE)
 *                      does not fit in one CTA's shared memory next to the weight rings
 *    q4_last_error() describes the most recent refusal or failure of the calling thread.
 *  - Kernels never trap and contain no unbounded spin: each warp waits only for its own asynchronous copies
 *    (cp.async groups, or an mbarrier that its bulk or tensor copies complete). An mbarrier wait gives up after
 *    q4_set_wait_limit's cycles (default 4e9, about two seconds); the warp whose wait ran out then issues no
 *    further copies, stores NaN for every row it stores from then on (in the Q4_K row kernels, every row its CTA
 *    stores from then on), records Q4_FAULT_WAIT_TIMEOUT, and before exiting waits (bounded by 4e9 cycles) for
 *    the copies it had issued, so none lands in the shared memory of an exited CTA. Rows stored before the
 *    timeout keep their values.
 *  - Inputs are fp32 vectors, outputs fp32. Weights are packed as described per format below; multi-byte
 *    fields are little-endian.
 *
 * Formats
 * -------
 *  Q4 (planar; inferencelayer 0.2.13, src/bin/kernel_lab.rs, shader GEMV_F16S and its bindings
 *  `scales`/`quants`): a row of K weights is K/32 blocks. qs is uint8[N][K/32][16] and d is
 *  binary16[N][K/32] (raw bits in uint16). In block b, byte j holds weight 32b+j in its low nibble and
 *  weight 32b+j+16 in its high nibble; the weight is (q - 8) * d[n][b].
 *
 *  Q4_K (trueno-gpu 0.4.11, src/kernels/quantize/fused.rs, FusedRmsNormQ4KGemvKernel phase 3): a row is
 *  K/256 super-blocks of 144 bytes: binary16 d at byte 0, binary16 dmin at byte 2, 12 bytes of packed
 *  6-bit scales/mins at 4..15 and 128 quant bytes at 16..143. Sub-block j (weights 32j..32j+31) has
 *  scale sc and min m: for j < 4, sc = s[j] & 63 and m = s[j+4] & 63; for j >= 4,
 *  sc = (s[j+4] & 15) | ((s[j-4] >> 6) << 4) and m = (s[j+4] >> 4) | ((s[j] >> 6) << 4). Weight e is in
 *  quant byte 32*(e/64) + e%32, low nibble when e%64 < 32, else high nibble; its value is
 *  d*sc*q - dmin*m.
 *
 * Numerics: products and sums run in fp32 (packed fp32x2 FMAs), so results differ from exact arithmetic by
 * the order of summation; the library's tests hold every output within 1e-3 * sum_k |w_k||x_k| + 1e-5 of
 * an fp64 reference. The dequant entry points are bit-exact. Supported input range: the kernels stage each
 * 32-element block of x (or of the normalised x for Q4_K) scaled by a power of two chosen from its largest
 * magnitude; planar Q4 blocks must stay below 2^105 in magnitude and Q4_K blocks below 2^83, beyond which the
 * affected outputs are non-finite. Small inputs keep their relative accuracy down to the fp32 subnormal range.
 */
#ifndef Q4GEMV_H
#define Q4GEMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *q4_stream_t; /* the same type as cudaStream_t */

enum {
    Q4_OK = 0,
    Q4_EINVAL = -1,
    Q4_EALIGN = -2,
    Q4_ECUDA = -3,
    Q4_EUNSUPPORTED = -4
};

/* Fault bits reported by q4_device_faults. */
enum {
    Q4_FAULT_BAD_EXPERT = 4,   /* moe_q4_gemv or moe_q4_pure_read saw an expert id outside [0, E) */
    Q4_FAULT_WAIT_TIMEOUT = 8, /* a wait for a weight stage ran out of its cycle limit (rows written as NaN) */
    Q4_FAULT_COPY_LOST = 16    /* even the final wait for a warp's issued copies ran out (not seen in practice) */
};

/*
 * y[n] = sum_k W[n][k] * x[k], W in planar Q4 (see Formats).
 * Source: inferencelayer kernel_lab.rs, shader GEMV_F16S (one column of its output).
 *   y   float[N]          output                       (4-byte aligned)
 *   qs  uint8[N][K/32][16] packed codes                (16-byte aligned)
 *   d   uint16[N][K/32]   binary16 block scales        (2-byte aligned; when 16-byte aligned and K % 256 == 0
 *                                                       the scales travel in the same 16-byte async copies
 *                                                       as the codes, otherwise each is read directly)
 *   x   float[K]          input                        (16-byte aligned)
 *   N >= 1; K >= 32 and K % 32 == 0.
 */
int q4_gemv(float *y, const uint8_t *qs, const uint16_t *d, const float *x, int N, int K, q4_stream_t stream);

/*
 * Y[m][n] = sum_k W[n][k] * X[m][k] for m < M, reading every weight byte once for all M rows.
 * Source: spark_model gemm_quant.rs, dense_gemv_batchm (the contract: one weight sweep for all M rows,
 * refusal of any M above the compiled maximum, which the page raises from 8 to 16 with every row bit-identical
 * to a single call); inferencelayer kernel_lab.rs, GEMV_F16S with KC columns per workgroup.
 *   Y float[M][N] (row-major), X float[M][K] (row-major, 16-byte aligned); other arguments as q4_gemv.
 *   1 <= M <= 16. Row m of Y equals q4_gemv on X[m] bit for bit (same per-row summation order and reduction
 *   tree for every M). The M staged input vectors (M*K*4 bytes) must fit in one CTA's shared memory beside the
 *   weight rings: all M <= 8 up to K = 4096 and M = 16 up to K = 2048; larger inputs return Q4_EUNSUPPORTED.
 */
int q4_gemv_batched(float *Y, const uint8_t *qs, const uint16_t *d, const float *X, int M, int N, int K,
                    q4_stream_t stream);

/*
 * y[n] = sum_k W[n][k] * xhat[k], xhat[k] = x[k] * r * gamma[k], r = 1 / sqrt(sum_k x[k]^2 / K + eps).
 * The normalised input stays in shared memory; it is never written to global memory.
 * Source: trueno-gpu fused.rs, FusedRmsNormQ4KGemvKernel (phases 1-3).
 *   y float[N]; w uint8[N][K/256][144] Q4_K (16-byte aligned); x, gamma float[K] (16-byte aligned);
 *   eps >= 0 and finite (1e-5 is the page's default). N >= 1; K >= 256 and K % 256 == 0.
 */
int fused_rmsnorm_q4k_gemv(float *y, const uint8_t *w, const float *x, const float *gamma, float eps, int N,
                           int K, q4_stream_t stream);

/*
 * Unfused Q4_K GEMV for M input rows: Y[m][n] = sum_k W[n][k] * X[m][k] for m < M, reading every weight byte
 * once for all M rows (no normalisation; M = 1 is the plain Q4_K GEMV).
 * Source: trueno-gpu fused.rs (the Q4_K format of FusedRmsNormQ4KGemvKernel phase 3; the page also names an
 * unfused Q4KGemvKernel); the batched contract of spark_model gemm_quant.rs, dense_gemv_batchm.
 *   Y float[M][N] (row-major), X float[M][K] (row-major, 16-byte aligned), w as fused_rmsnorm_q4k_gemv.
 *   1 <= M <= 8; N >= 1; K % 256 == 0. The M staged rows must fit in one CTA's shared memory beside the weight
 *   rings (M*K*4 + M*K/2 bytes: M = 8 up to K = 4096); larger inputs return Q4_EUNSUPPORTED. M = 1 runs the
 *   kernel of fused_rmsnorm_q4k_gemv without the normalisation, so its summation order differs from M >= 2.
 */
int q4k_gemv_batched(float *Y, const uint8_t *w, const float *X, int M, int N, int K, q4_stream_t stream);

/*
 * y_gate[n] = sum_k Wg[n][k] * xhat[k] and y_up[n] = sum_k Wu[n][k] * xhat[k] from one staged input.
 * gamma != NULL: xhat is the RMSNorm of x as in fused_rmsnorm_q4k_gemv; gamma == NULL: xhat = x.
 * Source: trueno-gpu fused.rs, FusedGateUpQ4KGemvKernel (with the full Q4_K decode for both projections).
 *   y_gate, y_up float[N]; w_gate, w_up uint8[N][K/256][144] (16-byte aligned); x float[K] and gamma
 *   float[K] or NULL (16-byte aligned). N >= 1; K >= 256 and K % 256 == 0; eps as above.
 */
int fused_gateup_q4k_gemv(float *y_gate, float *y_up, const uint8_t *w_gate, const uint8_t *w_up,
                          const float *x, const float *gamma, float eps, int N, int K, q4_stream_t stream);

/*
 * Expert-gathered MoE gate and up GEMV over planar Q4 expert stores.
 * For token t < T and slot s < topk with e = expert_ids[t*topk + s]:
 *   y_gate[(t*topk + s)*N + r] = sum_k Wg[e*N + r][k] * x[t][k],  likewise y_up with Wu, for r < N.
 * Each selected expert's rows are streamed once per call and applied to every token routed to it; the
 * routing is read on the device (no host synchronisation).
 * Source: inferencelayer kernel_lab.rs, moe_lab and the MoE ceiling shader (row = eid*MI + r, one output
 * per routed row, gate and up stores).
 *   qs_gate, qs_up uint8[E*N][K/32][16]; d_gate, d_up uint16[E*N][K/32]; x float[T][K] (16-byte aligned);
 *   expert_ids int32[T][topk] (device). 1 <= topk <= E; T*topk <= 512.
 *   A slot whose id is outside [0, E) gets NaN outputs and, when dev_status is not NULL, *dev_status is
 *   set to Q4_FAULT_BAD_EXPERT (dev_status is a device int32 the caller zeroes beforehand).
 */
int moe_q4_gemv(float *y_gate, float *y_up, const uint8_t *qs_gate, const uint16_t *d_gate, const uint8_t *qs_up,
                const uint16_t *d_up, const float *x, const int32_t *expert_ids, int T, int topk, int E, int N,
                int K, int32_t *dev_status, q4_stream_t stream);

/*
 * SwiGLU epilogue variants (one output instead of two):
 *   fused_gateup_swiglu_q4k_gemv: y[n] = silu(g[n]) * u[n] with g, u the two outputs of
 *     fused_gateup_q4k_gemv (same arguments, same RMSNorm rule);
 *   moe_q4_swiglu_gemv: y[(t*topk + s)*N + r] = silu(g) * u with g, u the two outputs of moe_q4_gemv for that
 *     routed row (same arguments, same routing, NaN for an invalid id, same dev_status rule).
 * silu(g) = g / (1 + exp(-g)). The pages show only that production MoE keeps one value per routed row; the
 * gated-linear-unit form is the standard one. Each call reads every weight byte once, as the two-output forms.
 *   y float[N] (gate+up) or float[T][topk][N] (MoE), 4-byte aligned.
 */
int fused_gateup_swiglu_q4k_gemv(float *y, const uint8_t *w_gate, const uint8_t *w_up, const float *x,
                                 const float *gamma, float eps, int N, int K, q4_stream_t stream);
int moe_q4_swiglu_gemv(float *y, const uint8_t *qs_gate, const uint16_t *d_gate, const uint8_t *qs_up,
                       const uint16_t *d_up, const float *x, const int32_t *expert_ids, int T, int topk, int E,
                       int N, int K, int32_t *dev_status, q4_stream_t stream);

/*
 * MoE router: gate GEMV over the experts fused with top-K softmax, for the decode tokens of one step.
 * Source: spark_model gemm_quant.rs, moe_gate_topk_fused (gate[e] = x . Wgate[e] for every expert, then the
 * top-K indices and softmax weights, `normalize` flag). Here the router rows are planar Q4 (the library's
 * format) and the inputs fp32. For token t < T:
 *   logits[t][e] = sum_k Wr[e][k] * x[t][k] for e < E (written when logits != NULL);
 *   expert_ids[t][i], i < topk: the experts of the topk largest logits in descending order, ties to the lower
 *     index (a NaN logit ranks below every other);
 *   expert_weights[t][i] = softmax over all E logits at expert_ids[t][i], divided by the sum over the topk
 *     picks when normalize != 0.
 * The ids can be passed straight to moe_q4_gemv / moe_q4_swiglu_gemv (same [T][topk] layout).
 *   expert_ids int32[T][topk], expert_weights float[T][topk], logits float[T][E] or NULL (4-byte aligned);
 *   qs uint8[E][K/32][16], d uint16[E][K/32] as q4_gemv; x float[T][K] (16-byte aligned).
 *   1 <= E <= 4096; 1 <= topk <= E; T >= 1; K % 32 == 0.
 */
int moe_router_q4(int32_t *expert_ids, float *expert_weights, float *logits, const uint8_t *qs, const uint16_t *d,
                  const float *x, int T, int E, int K, int topk, int normalize, q4_stream_t stream);

/*
 * Pure-read ceiling instruments: the same bytes, the same addressing and the same launch shape as the
 * matching GEMV, but no unpack and no dot products. Each output row receives the XOR of the 32-bit quant
 * words and zero-extended 16-bit scales (Q4) or of the 32-bit words of the super-blocks (Q4_K) of that
 * row, stored as raw bits in a float, so nothing can be optimised away and the result is checkable.
 * Source: inferencelayer kernel_lab.rs, the `pure_read` probe and MOE_PURE_READ ("pureread ~ kernel"
 * means the access pattern is the limit; "pureread >> kernel" means the arithmetic is).
 *   q4_pure_read:  sink float[N]; other arguments as q4_gemv.
 *   q4k_pure_read: sink float[N]; w as fused_rmsnorm_q4k_gemv.
 *   moe_q4_pure_read: sink_gate, sink_up float[T][topk][N]; other arguments as moe_q4_gemv; a slot with
 *   an id outside [0, E) gets NaN.
 */
int q4_pure_read(float *sink, const uint8_t *qs, const uint16_t *d, int N, int K, q4_stream_t stream);
int q4k_pure_read(float *sink, const uint8_t *w, int N, int K, q4_stream_t stream);
int moe_q4_pure_read(float *sink_gate, float *sink_up, const uint8_t *qs_gate, const uint16_t *d_gate,
                     const uint8_t *qs_up, const uint16_t *d_up, const int32_t *expert_ids, int T, int topk,
                     int E, int N, int K, int32_t *dev_status, q4_stream_t stream);

/*
 * FMA-ceiling instrument: at least `fmas` fp32 FMAs (packed fp32x2, a <- a * mul + add in eight independent
 * chains per thread) on one 512-thread CTA per SM, with no memory traffic but one float per CTA written to
 * sink. Its time is the floor for a call's FMA work alone: a batched call at M vectors does M FMAs per weight,
 * and at M = 8 the FMA pipe rather than HBM may bind.
 * Source: no page defines this instrument; it applies the idea of inferencelayer kernel_lab.rs's `pure_read`
 * probe (time one resource alone, here the FMA pipe instead of the weight stream).
 *   sink float[sink_len], sink_len >= the device's SM count; sink[b] = the sum of CTA b's chain ends.
 *   fmas >= 1; the FMAs run are rounded up to a whole number of rounds (SM count * 512 threads * 16), and the
 *   count run is stored in *fmas_done when fmas_done is not NULL (host pointer).
 *   With mul = 1 and add = 0 every chain keeps its start value: thread t's chains j = 0..7 start at
 *   ((t % 7) + j, (t % 5) + j), so sink[b] is the sum of those 8192 small integers (exact).
 */
int q4_fma_ceiling(float *sink, int sink_len, long long fmas, float mul, float add, long long *fmas_done,
                   q4_stream_t stream);

/*
 * Dequant dumps (debug): W[n][k] = the fp32 weight, bit-exact with the format definitions above
 * ((q - 8) * d for Q4; d*sc*q - dmin*m rounded once to fp32 for Q4_K).
 *   W float[N][K] (16-byte aligned); other arguments as q4_gemv / fused_rmsnorm_q4k_gemv.
 */
int q4_dequant(float *W, const uint8_t *qs, const uint16_t *d, int N, int K, q4_stream_t stream);
int q4k_dequant(float *W, const uint8_t *w, int N, int K, q4_stream_t stream);

/* Text of the calling thread's most recent refusal or failure ("" when none). Valid until the next call. */
const char *q4_last_error(void);

/*
 * Launch overlap (programmatic dependent launch; no counterpart in the source pages, which launch each
 * kernel on its own). Off by default. When on, every GEMV, fused and MoE call (not the dequant dumps) is
 * launched so that it may start while the kernel before it in the same stream is still running: the Q4
 * and Q4_K kernels issue their first weight copies at once, then wait for that kernel's completion (and
 * the visibility of its writes) before they read x, gamma or expert ids or write any output; the MoE kernel
 * waits before it reads the expert ids. So a chain of calls where each x is the previous output stays
 * exact, and each call's weight streaming overlaps the previous call's tail.
 * Requirement while it is on: the kernel that runs directly before a call in the same stream must not
 * write that call's weight bytes (qs, d or the Q4_K blocks); weights written earlier in the stream, or on
 * another stream with ordinary event or stream synchronisation, are fine.
 * The setting is process-wide and read at each launch (a CUDA graph keeps the launches it captured).
 * q4_set_launch_overlap returns Q4_OK; q4_get_launch_overlap returns the current setting (0 or 1).
 */
int q4_set_launch_overlap(int enable);
int q4_get_launch_overlap(void);

/*
 * Limit, in SM cycles, of each kernel wait for a weight stage (no counterpart in the source pages). Process-wide,
 * read at each launch (a CUDA graph keeps the value it captured); default 4000000000 (about two seconds). 0 makes
 * every such wait give up at once without looking, which runs the timeout path (NaN rows, Q4_FAULT_WAIT_TIMEOUT)
 * on copies that still land. q4_set_wait_limit returns Q4_OK, or Q4_EINVAL for a negative limit;
 * q4_get_wait_limit returns the current limit.
 */
int q4_set_wait_limit(long long cycles);
long long q4_get_wait_limit(void);

/*
 * Synchronises the current device, then ORs the fault bits every kernel family recorded since the last
 * call into *faults and clears them. Returns Q4_OK or Q4_ECUDA.
 */
int q4_device_faults(unsigned *faults);

#ifdef __cplusplus
}
#endif

#endif /* Q4GEMV_H */
