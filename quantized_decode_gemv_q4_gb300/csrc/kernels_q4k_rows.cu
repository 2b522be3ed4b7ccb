// Row-per-lane Q4_K decode GEMV for sm_103a: fused RMSNorm + GEMV, fused gate+up (two weight streams
// against one staged input, RMSNorm optional, optional SwiGLU epilogue) and the pure-read instrument.
//
// Format (trueno-gpu `fused.rs`, FusedRmsNormQ4KGemvKernel phase 3): a row is K/256 super-blocks of 144
// bytes: f16 d, f16 dmin, 12 bytes of packed 6-bit scales/mins, 128 quant bytes. Chunk c (32 bytes) holds
// sub-block 2c in its low nibbles and sub-block 2c+1 in its high nibbles; weight value d*sc_j*q - dmin*m_j.
//
// Kernel shape (one persistent CTA per SM, nw <= 16 warps, nw <= K/256):
//  * a tile is 32 lane rows: 32 rows of the one matrix, or rows r0..r0+15 of gate (lanes 0-15) and of up
//    (lanes 16-31). CTA b takes tiles b, b + grid, ...; warp w takes super-blocks w, w + nw, ... of every
//    row of the tile, so a stage is one super-block of 32 lane rows (4608 bytes), copied by the warp with
//    coalesced 16-byte cp.async (nine per lane) into its own ring of D slots;
//  * prologue: the first stages are issued, then (after the previous kernel in the stream is done) sum(x^2),
//    r = rsqrt(sum/K + eps), xhat = x * r * gamma staged per 32-element sub-block j, pre-scaled for the
//    bias-free decode with its own exponent bound e_j, next to (S_j, 2^(22+e_j)) where S_j * 2^(-22-e_j) is the
//    sub-block's FMA chain run on codes of 1 (so it matches a sub-block of equal unit codes bit for bit);
//  * lane l decodes the header of its own row's super-block once (eight 6-bit scales and mins), then runs
//    over the four chunks: one shift and eight ANDs per word, packed fp32x2 FMAs against the staged input
//    (every lane reads the same input quads, so each shared load is one broadcast wavefront), one
//    accumulator A_j per sub-block; each sub-block is folded as fl(d*sc_j*2^(22+e_j) * A_j) -
//    fl(dmin*m_j * S_j) with unfused rounded operations, so a sub-block whose weights d*sc_j*q - dmin*m_j are all zero
//    (sc_j = m_j = 0, or a constant power-of-two code with d*sc_j*q = dmin*m_j) contributes exactly zero;
//  * per tile the warps' per-lane partial sums meet in shared memory (double-buffered by tile parity, one
//    CTA barrier per tile) and one warp, rotating with the tile, adds them in warp order and stores the rows.
//  * a stage wait that runs out of its limit makes the warp stop issuing copies and contribute NaN partials, so
//    every row the CTA stores from then on is NaN (kFaultWaitTimeout); before exiting the warp waits, bounded,
//    for the copies it had issued.
// Inputs whose staged value reaches 2^83 in magnitude are outside the supported range (non-finite result).
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include <cuda.h>  // tensor-map types (the encoder is reached through the runtime's driver entry point)

#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

constexpr int kSB = 144;                   // bytes per super-block
constexpr int kPieces = kSB / 16;          // 16-byte copy pieces per super-block
constexpr uint32_t kSlot = 32u * kSB;      // one stage: a super-block of each of the 32 lane rows
constexpr int kMaxWarps = 16;
constexpr int kGroupMax = 4;               // tiles whose partial sums meet at one CTA barrier

struct RowParams {
    CUtensorMap tm0, tm1;  // weight matrices as 2-D byte tensors [N][row bytes], box 144 x rows per stream
    float* y0;
    float* y1;
    const uint8_t* w0;
    const uint8_t* w1;
    const float* x;
    const float* gamma;  // nullptr: no RMSNorm
    float eps;
    int swiglu;          // two streams only: y0 = silu(gate) * up, y1 unused
    int N, K, nsb;
    int tiles;           // ceil(N / rows per tile)
    int nb;              // tiles per reduction group, 1..kGroupMax
    long long wait_cycles;  // limit of one stage wait
    unsigned* fault;        // device fault word
    uint32_t xs_off, ss_off, red_off, bar_off, slots_off;
};


// byte j of w as an exact float (0x4B000000 | b is 2^23 + b)
__device__ __forceinline__ float sbyte(uint32_t w, int j) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + (uint32_t)j)) - 8388608.0f;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
                 : "memory");
}

// 2-D tensor tile (x bytes in, y rows down) into shared memory, completing on the mbarrier's transaction count
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

template <int NS, int D, bool PURE, bool TMA>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) q4k_rows_kernel(const __grid_constant__ RowParams p) {
    constexpr int TR = 32 / NS;  // rows per tile and stream
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = (int)(blockDim.x >> 5);
    const size_t row_bytes = (size_t)p.nsb * kSB;
    const uint32_t ring = smem_addr(smem) + p.slots_off + (uint32_t)(warp * D) * kSlot;
    const uint8_t* const ring_p = smem + p.slots_off + (size_t)(warp * D) * kSlot;
    const uint64_t pol = policy_evict_first();
    const uint32_t bars = smem_addr(smem) + p.bar_off + (uint32_t)(warp * D) * 8u;  // one mbarrier per slot
    // set when a stage wait ran out: the CTA's rows are then stored as NaN
    int& s_err = *reinterpret_cast<int*>(smem + p.bar_off + kMaxWarps * 3 * 8);  // some warp's wait ran out
    if (threadIdx.x == 0) s_err = 0;
    if constexpr (TMA) {
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < D; ++k) mbar_init(bars + 8u * k, 1u);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
    }

    // Copy pieces of this lane: piece j*32 + lane of a stage is bytes [16k, 16k+16) of lane row
    // (j*32 + lane) / 9, which is row rr of stream 0 or 1 of the tile.
    uint32_t soff[kPieces];
    int prow[kPieces];
    uint32_t s1mask = 0u;
#pragma unroll
    for (int j = 0; j < kPieces; ++j) {
        const int pc = j * 32 + lane;
        const int lr = pc / kPieces;
        const int k = pc - lr * kPieces;
        const int rr = lr % TR;
        if (lr >= TR) s1mask |= 1u << j;
        prow[j] = rr;
        soff[j] = (uint32_t)((size_t)rr * row_bytes) + (uint32_t)(16 * k);
    }

    // This warp's stages: for each of the CTA's tiles, super-blocks warp, warp + nw, ...
    const int spb = (p.nsb - warp + nw - 1) / nw;
    const int my_tiles = ((int)blockIdx.x < p.tiles) ? (p.tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = my_tiles * spb;

    int itile = (int)blockIdx.x, ik = 0, islot = 0, iss = 0;
    bool aborted = false;  // a stage wait ran out: no more copies, this warp's partials are NaN
    auto issue = [&]() {
        if (iss < total && !aborted) {
            const int r0 = itile * TR;
            const int nv = p.N - r0;
            const int sb = warp + ik * nw;
            const uint8_t* b0 = p.w0 + (size_t)r0 * row_bytes + (size_t)sb * kSB;
            const uint8_t* b1 = NS == 2 ? p.w1 + (size_t)r0 * row_bytes + (size_t)sb * kSB : b0;
            if constexpr (TMA) {
                // one bulk tensor copy per stream by lane 0 (rows past N arrive zero-filled); this warp's
                // earlier reads of the slot are ordered before the asynchronous write
                if (lane == 0) {
                    const uint32_t bar = bars + 8u * (uint32_t)islot;
                    const uint32_t dst = ring + (uint32_t)islot * kSlot;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(bar, kSlot);
                    tma_load_2d(dst, &p.tm0, sb * kSB, r0, bar, pol);
                    if constexpr (NS == 2) tma_load_2d(dst + (uint32_t)(TR * kSB), &p.tm1, sb * kSB, r0, bar, pol);
                }
                (void)nv;
                (void)b0;
                (void)b1;
            } else {
                const uint32_t dst = ring + (uint32_t)islot * kSlot + (uint32_t)lane * 16u;
#pragma unroll
                for (int j = 0; j < kPieces; ++j)
                    if (prow[j] < nv) cp_async16(dst + (uint32_t)(j * 512), ((s1mask >> j) & 1u ? b1 : b0) + soff[j], pol);
            }
            ++iss;
            if (++ik == spb) {
                ik = 0;
                itile += (int)gridDim.x;
            }
            islot = islot + 1 == D ? 0 : islot + 1;
        }
        if constexpr (!TMA) cp_async_commit();
    };

#pragma unroll
    for (int k = 0; k < D - 1; ++k) issue();

    // The weights are constant; x, gamma and the outputs may belong to the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();

    float* const red = reinterpret_cast<float*>(smem + p.red_off);  // [2][kGroupMax][kMaxWarps][32] + [kMaxWarps]
    if constexpr (!PURE) {
        const int nthreads = (int)blockDim.x;
        float r = 1.0f;
        if (p.gamma) {
            // sum of squares over K: per-thread partials (loads issued ahead), warp shuffles, one value per warp
            const int K4 = p.K >> 2;
            float ss = 0.f;
            for (int base = threadIdx.x; base < K4; base += nthreads * kStageU) {
                float4 xv[kStageU];
#pragma unroll
                for (int j = 0; j < kStageU; ++j) {
                    const int idx = base + j * nthreads;
                    xv[j] = idx < K4 ? __ldg(reinterpret_cast<const float4*>(p.x) + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < kStageU; ++j) {
                    ss = fmaf(xv[j].x, xv[j].x, ss);
                    ss = fmaf(xv[j].y, xv[j].y, ss);
                    ss = fmaf(xv[j].z, xv[j].z, ss);
                    ss = fmaf(xv[j].w, xv[j].w, ss);
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            float* const part = red + 2 * kGroupMax * kMaxWarps * 32;
            if (lane == 0) part[warp] = ss;
            __syncthreads();
            float tot = 0.f;
            for (int w = 0; w < nw; ++w) tot += part[w];
            r = rsqrtf(tot / (float)p.K + p.eps);
        }
        // xhat staged per sub-block j in natural element order, pre-scaled for the code positions of the
        // low (j even) or high (j odd) nibbles: four lanes per sub-block, lane t of the group holding
        // elements 8t .. 8t+7. K/32 is a multiple of 8, so whole warps take part in every group shuffle.
        float4* const xs = reinterpret_cast<float4*>(smem + p.xs_off);
        float2* const ssum = reinterpret_cast<float2*>(smem + p.ss_off);
        const int nsub = p.K / 32;
        const int t4 = lane & 3;
        for (int thr = threadIdx.x; thr < nsub * 4; thr += nthreads) {
            const int js = thr >> 2;
            const float4* src = reinterpret_cast<const float4*>(p.x) + js * 8 + 2 * t4;
            float4 xa = __ldg(src), xb = __ldg(src + 1);
            if (p.gamma) {
                const float4* gsrc = reinterpret_cast<const float4*>(p.gamma) + js * 8 + 2 * t4;
                const float4 ga = __ldg(gsrc), gb = __ldg(gsrc + 1);
                xa = make_float4((xa.x * r) * ga.x, (xa.y * r) * ga.y, (xa.z * r) * ga.z, (xa.w * r) * ga.w);
                xb = make_float4((xb.x * r) * gb.x, (xb.y * r) * gb.y, (xb.z * r) * gb.z, (xb.w * r) * gb.w);
            }
            const Stage4 st = stage_block4(xa, xb, js & 1);
            xs[js * 8 + 2 * t4] = st.a;
            xs[js * 8 + 2 * t4 + 1] = st.b;
            if (t4 == 0) ssum[js] = make_float2(0.f, block_factor(st.e));
        }
        __syncthreads();
        // S_j: the sub-block's chain (quads 0..7, each as its low or high pair) on codes of 1, times 2^(22+e_j)
        const Word8s c1 = decode_word_sub(0x11111111u);
        for (int js = threadIdx.x; js < nsub; js += nthreads) {
            const float2 p01 = (js & 1) ? c1.hi01 : c1.lo01, p23 = (js & 1) ? c1.hi23 : c1.lo23;
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = xs[js * 8 + q];
                a = ffma2(p01, make_float2(v.x, v.y), a);
                a = ffma2(p23, make_float2(v.z, v.w), a);
            }
            ssum[js].x = (a.x + a.y) * ssum[js].y;
        }
    }
    __syncthreads();

    float2 tot2 = make_float2(0.f, 0.f);
    uint32_t fold = 0u;
    int tile = (int)blockIdx.x, k = 0, cslot = 0, tcount = 0;
    uint32_t cphase = 0u;
    int consumed = 0;  // stages whose wait completed (tensor-copy mode)
    for (int g = 0; g < total; ++g) {
        issue();  // stage g + D - 1 into the slot consumed at g - 1
        if constexpr (TMA) {
            // stage g has landed once its slot's mbarrier completes phase cphase; the wait is bounded
            if (!aborted) {
                if (warp_wait_bounded(bars + 8u * (uint32_t)cslot, cphase, p.wait_cycles)) {
                    consumed = g + 1;
                } else {
                    aborted = true;
                    s_err = 1;
                    if (lane == 0) atomicOr(p.fault, kFaultWaitTimeout);
                }
            }
        } else {
            cp_async_wait<D - 1>();  // stage g has landed
        }
        __syncwarp();
        const uint8_t* const sp = ring_p + (size_t)cslot * kSlot + (size_t)lane * kSB;
        const int sb = warp + k * nw;
        const uint4 hdr = *reinterpret_cast<const uint4*>(sp);
        if (aborted) {
            // no compute after a timed-out wait; the tile's rows are stored as NaN
        } else if constexpr (PURE) {
            uint32_t f = hdr.x ^ hdr.y ^ hdr.z ^ hdr.w;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint4 w = *reinterpret_cast<const uint4*>(sp + 16 + 16 * u);
                f ^= w.x ^ w.y ^ w.z ^ w.w;
            }
            fold ^= f;
        } else {
            const float d = f16_bits_to_f32(hdr.x);
            const float dmin = f16_bits_to_f32(hdr.x >> 16);
            // 6-bit scales and mins of sub-blocks 0-3 and 4-7, one per byte
            const uint32_t sc03 = hdr.y & 0x3F3F3F3Fu;
            const uint32_t m03 = hdr.z & 0x3F3F3F3Fu;
            const uint32_t sc47 = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
            const uint32_t m47 = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
            const float4* const xq = reinterpret_cast<const float4*>(smem + p.xs_off) + sb * 64;
            const float4* const sq = reinterpret_cast<const float4*>(smem + p.ss_off) + sb * 4;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 sf = sq[c];  // (S, 2^(22+e)) of sub-blocks 2c and 2c+1
                const uint32_t scw = c < 2 ? sc03 : sc47;
                const uint32_t mw = c < 2 ? m03 : m47;
                // d*sc_j*2^(22+e_j) and -dmin*m_j, both exact (products of at most 17 significant bits)
                const float2 dsc = make_float2((d * sbyte(scw, (2 * c) & 3)) * sf.y, (d * sbyte(scw, (2 * c + 1) & 3)) * sf.w);
                const float2 mn = make_float2(-dmin * sbyte(mw, (2 * c) & 3), -dmin * sbyte(mw, (2 * c + 1) & 3));
                float2 aL = make_float2(0.f, 0.f), aH = make_float2(0.f, 0.f);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 w = *reinterpret_cast<const uint4*>(sp + 16 + 32 * c + 16 * h);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const Word8s d8 = decode_word_sub(i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w);
                        const float4 xl = xq[(2 * c) * 8 + 4 * h + i];
                        const float4 xh = xq[(2 * c + 1) * 8 + 4 * h + i];
                        aL = ffma2(d8.lo01, make_float2(xl.x, xl.y), aL);
                        aL = ffma2(d8.lo23, make_float2(xl.z, xl.w), aL);
                        aH = ffma2(d8.hi01, make_float2(xh.x, xh.y), aH);
                        aH = ffma2(d8.hi23, make_float2(xh.z, xh.w), aH);
                    }
                }
                // fl(dsc * A) - fl(dmin * m * S) per sub-block, then into the running pair; scalar rounded
                // operations, which the compiler never fuses into an FMA (a fused form would leave the
                // product's rounding error instead of an exact zero)
                tot2.x = __fadd_rn(tot2.x, __fadd_rn(__fmul_rn(dsc.x, aL.x + aL.y), __fmul_rn(mn.x, sf.x)));
                tot2.y = __fadd_rn(tot2.y, __fadd_rn(__fmul_rn(dsc.y, aH.x + aH.y), __fmul_rn(mn.y, sf.z)));
            }
        }
        __syncwarp();  // every lane is done with this slot before a later stage reuses it

        if (++k == spb) {
            // tile done: this warp's per-lane partials go to the group buffer (double-buffered by group
            // parity); after the group's last tile a CTA barrier, then for each tile of the group one warp,
            // rotating with the tile, adds the partials in warp order and stores the tile's rows
            const int gi = tcount % p.nb;
            float* const gbuf = red + ((tcount / p.nb) & 1) * (kGroupMax * kMaxWarps * 32);
            gbuf[(gi * kMaxWarps + warp) * 32 + lane] = aborted ? NAN : PURE ? __uint_as_float(fold) : tot2.x + tot2.y;
            tot2 = make_float2(0.f, 0.f);
            fold = 0u;
            if (gi == p.nb - 1 || tcount == my_tiles - 1) {
                __syncthreads();
                for (int i = 0; i <= gi; ++i) {
                    if (warp != (tcount - gi + i) % nw) continue;
                    const float* const buf = gbuf + i * (kMaxWarps * 32);
                    const bool bad = *reinterpret_cast<volatile int*>(&s_err) != 0;
                    const int r0 = (tile - (gi - i) * (int)gridDim.x) * TR;
                    if constexpr (PURE) {
                        uint32_t f = 0u;
                        for (int w = 0; w < nw; ++w) f ^= __float_as_uint(buf[w * 32 + lane]);
                        const int rr = lane % TR;
                        if (r0 + rr < p.N) (NS == 2 && lane >= TR ? p.y1 : p.y0)[r0 + rr] = bad ? NAN : __uint_as_float(f);
                    } else {
                        float v = 0.f;
                        for (int w = 0; w < nw; ++w) v += buf[w * 32 + lane];
                        if (bad) v = NAN;
                        const int rr = lane % TR;
                        if (NS == 2 && p.swiglu) {
                            const float up = __shfl_down_sync(0xffffffffu, v, TR);
                            if (lane < TR && r0 + rr < p.N) p.y0[r0 + rr] = silu(v) * up;
                        } else if (r0 + rr < p.N) {
                            (NS == 2 && lane >= TR ? p.y1 : p.y0)[r0 + rr] = v;
                        }
                    }
                }
            }
            k = 0;
            tile += (int)gridDim.x;
            ++tcount;
        }
        if (++cslot == D) {
            cslot = 0;
            cphase ^= 1u;
        }
    }
    // tensor copies issued but not consumed (only after a wait ran out): let them land before the CTA exits
    if constexpr (TMA)
        for (int st = consumed; st < iss; ++st)
            if (!warp_wait_bounded(bars + 8u * (uint32_t)(st % D), (uint32_t)((st / D) & 1), kDrainCycles) &&
                lane == 0)
                atomicOr(p.fault, kFaultCopyLost);
}

inline uint32_t round_up_u32(uint32_t a, uint32_t b) { return (a + b - 1) / b * b; }

template <int NS, int D, bool PURE, bool TMA>
cudaError_t launch_rows_fixed(const DeviceInfo& di, const RowParams& p, int nw, uint32_t smem, cudaStream_t s) {
    static std::once_flag attr_once[64];
    auto kern = q4k_rows_kernel<NS, D, PURE, TMA>;
    cudaError_t err = cudaSuccess;
    std::call_once(attr_once[di.device & 63], [&] {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (err != cudaSuccess) return err;
    const int grid = std::min(di.sm_count, p.tiles);
    return launch_kernel(kern, grid, nw * 32, smem, s, p);
}

// Tensor map of a Q4_K weight matrix as a 2-D byte tensor [N][K/256*144], box 144 bytes x `rows`, rows past
// N zero-filled. The encoder comes from the driver through the runtime's entry-point query; maps are cached
// per (matrix, N, K, rows) since encoding one costs host time on every call otherwise.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

struct MapEntry {
    const void* w = nullptr;
    int N = 0, K = 0, rows = 0;
    CUtensorMap map;
};

bool weight_map(CUtensorMap* out, const uint8_t* w, int N, int K, int rows) {
    static std::mutex mu;
    static MapEntry cache[16];
    static int next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (const MapEntry& m : cache)
        if (m.w == w && m.N == N && m.K == K && m.rows == rows) {
            *out = m.map;
            return true;
        }
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t row_bytes = (cuuint64_t)(K / 256) * kSB;
    const cuuint64_t dims[2] = {row_bytes, (cuuint64_t)N};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)kSB, (cuuint32_t)rows};
    const cuuint32_t estr[2] = {1u, 1u};
    MapEntry& e = cache[next];
    if (fn(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        e.w = nullptr;
        return false;
    }
    e.w = w;
    e.N = N;
    e.K = K;
    e.rows = rows;
    *out = e.map;
    next = (next + 1) % 16;
    return true;
}

// Shared memory: [staged xhat K*4][(S_j, 2^(22+e_j)) per sub-block][reduction 2*4*16*32 + 16 floats]
//                [mbarriers 16*3*8, error word][nw rings of D slots of 4608 bytes]. Warps: the super-blocks per row
// spread evenly over at most 16 warps; depth: 2 (3 on request) if it fits, fewer warps for the longest
// inputs (up to K = 48384).
template <int NS, bool PURE>
cudaError_t run_rows(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x, const float* gamma,
                     float eps, int N, int K, bool swiglu, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    RowParams p;
    p.y0 = y0;
    p.y1 = y1;
    p.w0 = w0;
    p.w1 = w1;
    p.x = x;
    p.gamma = gamma;
    p.eps = eps;
    p.swiglu = swiglu ? 1 : 0;
    p.N = N;
    p.K = K;
    p.nsb = K / 256;
    p.tiles = (N + 32 / NS - 1) / (32 / NS);
    p.wait_cycles = wait_limit_cycles();
    p.nb = kGroupMax;
    p.fault = device_fault_word(di.device);
    if (!p.fault) return cudaErrorInvalidSymbol;
    if (!weight_map(&p.tm0, w0, N, K, 32 / NS)) return cudaErrorNotSupported;
    if (NS == 2 && !weight_map(&p.tm1, w1, N, K, 32 / NS)) return cudaErrorNotSupported;
    const int per_warp = (p.nsb + kMaxWarps - 1) / kMaxWarps;
    const int nw = (p.nsb + per_warp - 1) / per_warp;
    p.xs_off = 0;
    p.ss_off = PURE ? 0u : (uint32_t)K * 4u;
    p.red_off = p.ss_off + (PURE ? 0u : round_up_u32((uint32_t)(K / 32) * 8u, 128u));
    p.bar_off = p.red_off + round_up_u32((uint32_t)(2 * kGroupMax * kMaxWarps * 32 + kMaxWarps) * 4u, 128u);
    p.slots_off = p.bar_off + round_up_u32((uint32_t)(kMaxWarps * 3 * 8 + 4), 128u);
    // ring depth 2 (the measured best), fewer warps for the longest inputs
    for (int w = nw; w >= 1; --w) {
        const uint32_t smem = p.slots_off + (uint32_t)(w * 2) * kSlot;
        if (smem <= (uint32_t)di.max_smem_optin) return launch_rows_fixed<NS, 2, PURE, true>(di, p, w, smem, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_q4k_rows_gemv(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x,
                                 const float* gamma, float eps, int N, int K, bool swiglu, cudaStream_t s) {
    if (w1) return run_rows<2, false>(y0, y1, w0, w1, x, gamma, eps, N, K, swiglu, s);
    return run_rows<1, false>(y0, nullptr, w0, nullptr, x, gamma, eps, N, K, false, s);
}

cudaError_t launch_q4k_rows_pure_read(float* sink, const uint8_t* w, int N, int K, cudaStream_t s) {
    return run_rows<1, true>(sink, nullptr, w, nullptr, nullptr, nullptr, 0.f, N, K, false, s);
}

}  // namespace q4
