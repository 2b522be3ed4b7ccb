// Row-per-lane Q4_K decode GEMV for sm_103a: fused RMSNorm + GEMV, fused gate+up (two weight streams
// against one staged input, RMSNorm optional, optional SwiGLU epilogue) and the pure-read instrument.
//
// Format (trueno-gpu `fused.rs`, FusedRmsNormQ4KGemvKernel phase 3): a row is K/256 super-blocks of 144
// bytes: f16 d, f16 dmin, 12 bytes of packed 6-bit scales/mins, 128 quant bytes. Chunk c (32 bytes) holds
// sub-block 2c in its low nibbles and sub-block 2c+1 in its high nibbles; weight value d*sc_j*q - dmin*m_j.
//
// Kernel shape (one persistent CTA of W <= 16 warps per SM):
//  * a tile is 32 lane rows: 32 rows of the one matrix, or rows r0..r0+15 of gate (lanes 0-15) and of up
//    (lanes 16-31). The W warps form G groups of KS warps; each group takes tiles of its own (groups numbered
//    across CTAs first) and warp k of a group takes super-blocks k, k + KS, ... of every row of the tile, so a
//    stage is one super-block of 32 lane rows (4608 bytes), moved by one 2-D tensor copy per stream into the
//    warp's ring of D slots (mbarrier per slot, bounded waits). KS is chosen per problem so that the groups
//    cover the tiles evenly with the fewest stages per warp;
//  * prologue: one stage per warp is requested, then (after the previous kernel in the stream is done) each
//    thread loads its eight elements of x and gamma in one round trip: sum(x^2) for r = rsqrt(sum/K + eps)
//    comes from the same registers that are then staged as x * gamma (r, one scalar for the whole row sum,
//    multiplies the row totals at the end), per 32-element sub-block j pre-scaled for the bias-free decode
//    with its own exponent bound e_j; beside it (S_j, 2^(22+e_j)), where S_j * 2^(-22-e_j) is the sub-block's
//    FMA chain run on codes of 1, formed by the four lanes of the sub-block through shuffles;
//  * lane l decodes the header of its own row's super-block once: each 6-bit scale or min becomes the float
//    2^23 + v by one byte permute, and one FMA with d (or dmin) and -d * 2^23 gives d * sc exactly;
//  * per word: one shift and eight ANDs, then packed fp32x2 FMAs against the staged input (every lane reads
//    the same input quads, so each shared load is one broadcast wavefront), one accumulator A_j per sub-block;
//    each sub-block is folded as fl(d*sc_j*2^(22+e_j) * A_j) - fl(dmin*m_j * S_j) with unfused rounded
//    operations, so a sub-block whose weights d*sc_j*q - dmin*m_j are all zero (sc_j = m_j = 0, or a constant
//    power-of-two code with d*sc_j*q = dmin*m_j) contributes exactly zero;
//  * at the end of a tile the KS per-lane partial sums meet in shared memory (double-buffered by tile parity)
//    at the group's named barrier, and warp 0 of the group adds them in warp order and stores the rows (or
//    silu(gate) * up, the up total arriving by one shuffle);
//  * a stage wait that runs out of its limit makes the warp stop issuing copies and contribute NaN partials, so
//    every row its group stores from then on is NaN (kFaultWaitTimeout); before exiting the warp waits,
//    bounded, for the copies it had issued.
// Inputs whose staged value reaches 2^83 in magnitude are outside the supported range (non-finite result).
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>


#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

constexpr int kSB = 144;                   // bytes per super-block
constexpr uint32_t kSlot = 32u * kSB;      // one stage: a super-block of each of the 32 lane rows
constexpr int kMaxWarps = 16;

struct RowParams {
    CUtensorMap tm0, tm1;  // weight matrices as 2-D byte tensors [N][row bytes], box 144 x rows per stream
    float* y0;
    float* y1;
    const float* x;
    const float* gamma;  // nullptr: no RMSNorm
    float eps;
    int swiglu;          // two streams only: y0 = silu(gate) * up, y1 unused
    int N, K, nsb;
    int tiles;           // ceil(N / rows per tile)
    int KS;              // warps per tile; W = KS * G warps per CTA
    int G;               // groups per CTA
    long long wait_cycles;  // limit of one stage wait
    unsigned* fault;        // device fault word
    uint32_t xs_off, ss_off, red_off, bar_off, slots_off;
};


// 2-D tensor tile (x bytes in, y rows down) into shared memory, completing on the mbarrier's transaction count
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

template <int NS, int D, bool PURE>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) q4k_rows_kernel(const __grid_constant__ RowParams p) {
    constexpr int TR = 32 / NS;  // rows per tile and stream
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nthreads = (int)blockDim.x;
    const uint32_t s_base = smem_addr(smem);
    const uint32_t bars = s_base + p.bar_off + (uint32_t)(warp * D) * 8u;  // this warp's mbarriers, one per slot
    const uint64_t pol = policy_evict_first();
    const int nwarps = nthreads / 32;
    if ((int)threadIdx.x < nwarps * D) {
        mbar_init(s_base + p.bar_off + 8u * threadIdx.x, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Warp wi belongs to group wi / KS (tiles gid, gid + G*grid, ...) as its warp k = wi % KS (super-blocks k,
    // k + KS, ... of each tile). Its stage j is tile j / spw of the group, super-block k + (j % spw) * KS, into
    // slot j % D of the warp's ring.
    const int gstep = p.G * (int)gridDim.x;
    struct Plan {
        int k, spw, gid, tiles, total;
    };
    auto plan_of = [&](int wi) {
        Plan w;
        const int gi = wi / p.KS;
        w.k = wi - gi * p.KS;
        w.spw = w.k < p.nsb ? (p.nsb - 1 - w.k) / p.KS + 1 : 0;  // 0 when KS > nsb: the warp only meets barriers
        w.gid = gi * (int)gridDim.x + (int)blockIdx.x;
        w.tiles = w.gid < p.tiles ? (p.tiles - 1 - w.gid) / gstep + 1 : 0;  // the same for every warp of a group
        w.total = w.tiles * w.spw;
        return w;
    };
    auto issue_for = [&](int wi, const Plan& w, int j) {
        const int jt = j / w.spw;
        const int sb = w.k + (j - jt * w.spw) * p.KS;
        const int r0 = (w.gid + jt * gstep) * TR;
        const uint32_t bar = s_base + p.bar_off + (uint32_t)(wi * D + j % D) * 8u;
        const uint32_t dst = s_base + p.slots_off + (uint32_t)(wi * D + j % D) * kSlot;
        mbar_expect_tx(bar, kSlot);
        tma_load_2d(dst, &p.tm0, sb * kSB, r0, bar, pol);  // rows past N arrive zero-filled
        if constexpr (NS == 2) tma_load_2d(dst + (uint32_t)(TR * kSB), &p.tm1, sb * kSB, r0, bar, pol);
    };
    const Plan me = plan_of(warp);
    const int g = warp / p.KS, k = me.k, spw = me.spw, gid = me.gid, total = me.total;
    const int my_tiles = me.tiles;  // every warp of the group takes part in each tile's barrier
    // A slot is refilled only after every lane of the warp has read it (the __syncwarp before each refill), and a
    // proxy fence orders those reads before the tensor copy's writes.
    auto issue = [&](int j) {
        if (lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_for(warp, me, j);
        }
    };
    if (total > 0) issue(0);

    // The weights are constant; x, gamma and the outputs may belong to the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();
    // The other slots of every ring are requested by the lanes of the last warp, while the rest stage the input
    // (a burst of copies from one SM is accepted at a limited rate; spread over the warps it would hold each of
    // them for that long).
    if (warp == nwarps - 1 && lane < nwarps) {
        const Plan w = plan_of(lane);
        for (int j = 1; j < min(D, w.total); ++j) issue_for(lane, w, j);
    }
    int issued = min(D, total);

    float* const red = reinterpret_cast<float*>(smem + p.red_off);  // [2][G][KS][32] partials, then [2][G] flags
    int* const red_bad = reinterpret_cast<int*>(red + 2 * kMaxWarps * 32);
    float* const part = reinterpret_cast<float*>(red_bad + 2 * kMaxWarps);  // one sum of squares per warp
    float r = 1.0f;  // RMSNorm factor, applied to the row sums
    if constexpr (PURE) {
        if (threadIdx.x < 2 * kMaxWarps) red_bad[threadIdx.x] = 0;
        __syncthreads();
    } else {
        // Each thread holds elements 8t .. 8t+7 (t = its lane within a group of four) of sub-block thr / 4 of x
        // and gamma in registers, loaded in one round trip: sum(x^2) comes from them and x * gamma is staged
        // from them. The factor r = rsqrt(sum/K + eps) is a scalar of the whole row sum, so it multiplies the
        // row results at the end and the staging does not wait for the block-wide sum (K/32 is a multiple of
        // 8, so every loop runs whole warps and the group shuffles see 32 lanes).
        constexpr int kIt = 4;  // sub-block quarters a thread keeps in registers; longer inputs load twice
        const int nsub = p.K / 32;
        const int iters = (nsub * 4 + nthreads - 1) / nthreads;
        const bool keep = iters <= kIt;
        const bool norm = p.gamma != nullptr;
        const int t4 = lane & 3;
        float4 xa[kIt], xb[kIt], ga[kIt], gb[kIt];
        auto load_xg = [&](int thr, float4& a, float4& b, float4& c, float4& e) {
            const int q = (thr >> 2) * 8 + 2 * t4;
            a = __ldg(reinterpret_cast<const float4*>(p.x) + q);
            b = __ldg(reinterpret_cast<const float4*>(p.x) + q + 1);
            if (norm) {
                c = __ldg(reinterpret_cast<const float4*>(p.gamma) + q);
                e = __ldg(reinterpret_cast<const float4*>(p.gamma) + q + 1);
            }
        };
        auto sumsq = [](float ss, float4 a, float4 b) {
            ss = fmaf(a.x, a.x, ss);
            ss = fmaf(a.y, a.y, ss);
            ss = fmaf(a.z, a.z, ss);
            ss = fmaf(a.w, a.w, ss);
            ss = fmaf(b.x, b.x, ss);
            ss = fmaf(b.y, b.y, ss);
            ss = fmaf(b.z, b.z, ss);
            return fmaf(b.w, b.w, ss);
        };
        if (keep) {
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int thr = (int)threadIdx.x + it * nthreads;
                if (it < iters && thr < nsub * 4) load_xg(thr, xa[it], xb[it], ga[it], gb[it]);
            }
        }
        // xhat / r staged per sub-block j in element order, pre-scaled for the code positions of the low (j even)
        // or high (j odd) nibbles, and S_j from the chain of the sub-block's quads 0..7 on codes of 1: the four
        // lanes of the group take their two quads in turn, passing the running pair by shuffles.
        float4* const xs = reinterpret_cast<float4*>(smem + p.xs_off);
        float2* const ssum = reinterpret_cast<float2*>(smem + p.ss_off);
        const Word8s c1 = decode_word_sub(0x11111111u);
        float ss = 0.f;
        for (int it = 0, thr = threadIdx.x; thr < nsub * 4; ++it, thr += nthreads) {
            const int js = thr >> 2;
            float4 a, b, c, e;
            if (keep) {
                a = xa[0];
                b = xb[0];
                c = ga[0];
                e = gb[0];
#pragma unroll
                for (int q = 1; q < kIt; ++q)
                    if (it == q) {
                        a = xa[q];
                        b = xb[q];
                        c = ga[q];
                        e = gb[q];
                    }
            } else {
                load_xg(thr, a, b, c, e);
            }
            if (norm) {
                ss = sumsq(ss, a, b);
                a = make_float4(a.x * c.x, a.y * c.y, a.z * c.z, a.w * c.w);
                b = make_float4(b.x * e.x, b.y * e.y, b.z * e.z, b.w * e.w);
            }
            const int hi = js & 1;
            const Stage4 st = stage_block4(a, b, hi);
            xs[js * 8 + 2 * t4] = st.a;
            xs[js * 8 + 2 * t4 + 1] = st.b;
            const float2 p01 = hi ? c1.hi01 : c1.lo01, p23 = hi ? c1.hi23 : c1.lo23;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                float2 m = ffma2(p01, make_float2(st.a.x, st.a.y), acc);
                m = ffma2(p23, make_float2(st.a.z, st.a.w), m);
                m = ffma2(p01, make_float2(st.b.x, st.b.y), m);
                m = ffma2(p23, make_float2(st.b.z, st.b.w), m);
                acc.x = __shfl_sync(0xffffffffu, m.x, (lane & ~3) + t);
                acc.y = __shfl_sync(0xffffffffu, m.y, (lane & ~3) + t);
            }
            if (t4 == 0) {
                const float f = block_factor(st.e);
                ssum[js] = make_float2((acc.x + acc.y) * f, f);
            }
        }
        if (norm) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) part[warp] = ss;
        }
        __syncthreads();
    }

    bool aborted = false;  // a stage wait ran out: no more copies, this warp's partials are NaN
    int consumed = 0;
    const uint8_t* const ring_p = smem + p.slots_off + (size_t)(warp * D) * kSlot + (size_t)lane * kSB;
    for (int t = 0; t < my_tiles; ++t) {
        float2 tot2 = make_float2(0.f, 0.f);
        uint32_t fold = 0u;
        for (int s = 0; s < spw; ++s) {
            const int j = t * spw + s;
            const uint32_t slot = (uint32_t)(j % D);
            if (!aborted) {
                if (warp_wait_bounded(bars + 8u * slot, (uint32_t)((j / D) & 1), p.wait_cycles)) {
                    consumed = j + 1;
                } else {
                    aborted = true;
                    if (lane == 0) atomicOr(p.fault, kFaultWaitTimeout);
                }
            }
            if (aborted) continue;
            const uint8_t* const sp = ring_p + slot * kSlot;
            const int sb = k + s * p.KS;
            const uint4 hdr = *reinterpret_cast<const uint4*>(sp);
            if constexpr (PURE) {
                uint32_t f = hdr.x ^ hdr.y ^ hdr.z ^ hdr.w;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint4 w = *reinterpret_cast<const uint4*>(sp + 16 + 16 * u);
                    f ^= w.x ^ w.y ^ w.z ^ w.w;
                }
                fold ^= f;
            } else {
                const float d = __half2float(__ushort_as_half((unsigned short)(hdr.x & 0xFFFFu)));
                const float dmin = __half2float(__ushort_as_half((unsigned short)(hdr.x >> 16)));
                const float nd23 = -d * 8388608.0f, dmin23 = dmin * 8388608.0f;  // exact
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
                    // d*sc and -dmin*m, exact: the byte as the float 2^23 + v, then one FMA
                    const uint32_t jl = (uint32_t)((2 * c) & 3), jh = (uint32_t)((2 * c + 1) & 3);
                    const float dsl = fmaf(d, __uint_as_float(__byte_perm(scw, 0x4B000000u, 0x7540u + jl)), nd23);
                    const float dsh = fmaf(d, __uint_as_float(__byte_perm(scw, 0x4B000000u, 0x7540u + jh)), nd23);
                    const float mnl = fmaf(-dmin, __uint_as_float(__byte_perm(mw, 0x4B000000u, 0x7540u + jl)), dmin23);
                    const float mnh = fmaf(-dmin, __uint_as_float(__byte_perm(mw, 0x4B000000u, 0x7540u + jh)), dmin23);
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
                    // fl(d*sc*f * A) - fl(dmin*m * S) per sub-block (d*sc*f exact), with scalar rounded operations,
                    // which the compiler never fuses into an FMA (a fused form would leave the product's
                    // rounding error instead of an exact zero)
                    tot2.x = __fadd_rn(tot2.x, __fadd_rn(__fmul_rn(dsl * sf.y, aL.x + aL.y), __fmul_rn(mnl, sf.x)));
                    tot2.y = __fadd_rn(tot2.y, __fadd_rn(__fmul_rn(dsh * sf.w, aH.x + aH.y), __fmul_rn(mnh, sf.z)));
                }
            }
            __syncwarp();  // every lane is done with the slot before it is refilled
            if (issued < total) issue(issued++);
        }
        // the tile's partials meet at the group's named barrier (double-buffered by tile parity)
        const int par = t & 1;
        float* const gbuf = red + (par * kMaxWarps + g * p.KS) * 32;
        gbuf[k * 32 + lane] = aborted ? NAN : PURE ? __uint_as_float(fold) : tot2.x + tot2.y;
        if (PURE && aborted && lane == 0) red_bad[par * kMaxWarps + g] = 1;
        if (p.KS > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(p.KS * 32) : "memory");
        if (k == 0) {
            const int r0 = (gid + t * gstep) * TR;
            const int rr = lane % TR;
            if constexpr (PURE) {
                uint32_t f = 0u;
                for (int w = 0; w < p.KS; ++w) f ^= __float_as_uint(gbuf[w * 32 + lane]);
                const bool bad = red_bad[par * kMaxWarps + g] != 0;
                __syncwarp();
                if (lane == 0) red_bad[par * kMaxWarps + g] = 0;
                if (r0 + rr < p.N) (NS == 2 && lane >= TR ? p.y1 : p.y0)[r0 + rr] = bad ? NAN : __uint_as_float(f);
            } else {
                if (t == 0 && p.gamma) {  // the RMSNorm factor, from the per-warp sums of squares
                    float tot = 0.f;
                    for (int w = 0; w < nwarps; ++w) tot += part[w];
                    r = rsqrtf(tot / (float)p.K + p.eps);
                }
                float v = 0.f;
                for (int w = 0; w < p.KS; ++w) v += gbuf[w * 32 + lane];
                v *= r;
                if (NS == 2 && p.swiglu) {
                    const float up = __shfl_down_sync(0xffffffffu, v, TR);
                    if (lane < TR && r0 + rr < p.N) p.y0[r0 + rr] = silu(v) * up;
                } else if (r0 + rr < p.N) {
                    (NS == 2 && lane >= TR ? p.y1 : p.y0)[r0 + rr] = v;
                }
            }
        }
    }
    // tensor copies issued but not consumed (only after a wait ran out): let them land before the CTA exits
    for (int st = consumed; st < issued; ++st)
        if (!warp_wait_bounded(bars + 8u * (uint32_t)(st % D), (uint32_t)((st / D) & 1), kDrainCycles) && lane == 0)
            atomicOr(p.fault, kFaultCopyLost);
}

inline uint32_t round_up_u32(uint32_t a, uint32_t b) { return (a + b - 1) / b * b; }

template <int NS, int D, bool PURE>
cudaError_t launch_rows_fixed(const DeviceInfo& di, const RowParams& p, int nw, uint32_t smem, cudaStream_t s) {
    static std::once_flag attr_once[64];
    auto kern = q4k_rows_kernel<NS, D, PURE>;
    cudaError_t err = cudaSuccess;
    std::call_once(attr_once[di.device & 63], [&] {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (err != cudaSuccess) return err;
    const int grid = std::min(di.sm_count, (p.tiles + p.G - 1) / p.G);
    return launch_kernel(kern, grid, nw * 32, smem, s, p);
}

// Tensor map of a Q4_K weight matrix as a 2-D byte tensor [N][K/256*144], box 144 bytes x `rows`.
bool weight_map(CUtensorMap* out, const uint8_t* w, int N, int K, int rows) {
    return cached_tensor_map_2d(out, w, (uint64_t)(K / 256) * kSB, (uint64_t)N, (uint32_t)kSB, (uint32_t)rows, false);
}

// Shared memory: [staged xhat K*4][(S_j, 2^(22+e_j)) per sub-block][partials 2*16*32 floats, flags, per-warp
// sums][mbarriers 16*2*8][W rings of 2 slots of 4608 bytes]. Plan: W = 16 warps in groups of KS (a power of two)
// warps per tile, KS chosen so that the tiles spread over the groups with the fewest stages on the slowest warp
// (ties to fewer warps per tile); fewer warps for the longest inputs.
template <int NS, bool PURE>
cudaError_t run_rows(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x, const float* gamma,
                     float eps, int N, int K, bool swiglu, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    RowParams p;
    p.y0 = y0;
    p.y1 = y1;
    p.x = x;
    p.gamma = gamma;
    p.eps = eps;
    p.swiglu = swiglu ? 1 : 0;
    p.N = N;
    p.K = K;
    p.nsb = K / 256;
    p.tiles = (N + 32 / NS - 1) / (32 / NS);
    p.wait_cycles = wait_limit_cycles();
    p.fault = device_fault_word(di.device);
    if (!p.fault) return cudaErrorInvalidSymbol;
    if (!weight_map(&p.tm0, w0, N, K, 32 / NS)) return cudaErrorNotSupported;
    if (NS == 2 && !weight_map(&p.tm1, w1, N, K, 32 / NS)) return cudaErrorNotSupported;
    constexpr int D = 2;
    p.xs_off = 0;
    p.ss_off = PURE ? 0u : (uint32_t)K * 4u;
    p.red_off = p.ss_off + (PURE ? 0u : round_up_u32((uint32_t)(K / 32) * 8u, 128u));
    p.bar_off = p.red_off + round_up_u32((uint32_t)(2 * kMaxWarps * 32 + 2 * kMaxWarps + kMaxWarps) * 4u, 128u);
    p.slots_off = p.bar_off + round_up_u32((uint32_t)(kMaxWarps * D * 8), 128u);
    for (int W = kMaxWarps; W >= 1; W /= 2) {
        const uint32_t smem = p.slots_off + (uint32_t)(W * D) * kSlot;
        if (smem > (uint32_t)di.max_smem_optin) continue;
        int best_ks = W, best_cost = 1 << 30;
        for (int ks = 1; ks <= W; ks *= 2) {
            const int groups = (W / ks) * di.sm_count;
            const int cost = ((p.tiles + groups - 1) / groups) * ((p.nsb + ks - 1) / ks);
            if (cost < best_cost) {
                best_cost = cost;
                best_ks = ks;
            }
        }
        p.KS = best_ks;
        p.G = W / best_ks;
        return launch_rows_fixed<NS, D, PURE>(di, p, W, smem, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The encoder comes from the driver through the runtime's entry-point query.
static EncodeTiledFn encode_tiled() {
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

bool cached_tensor_map_2d(CUtensorMap* out, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                          uint32_t box_rows, bool swizzle128) {
    struct Entry {
        const void* base = nullptr;
        uint64_t row_bytes = 0, rows = 0;
        uint32_t box_bytes = 0, box_rows = 0;
        bool swz = false;
        CUtensorMap map;
    };
    static std::mutex mu;
    static Entry cache[32];
    static int next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& m : cache)
        if (m.base == base && m.row_bytes == row_bytes && m.rows == rows && m.box_bytes == box_bytes &&
            m.box_rows == box_rows && m.swz == swizzle128) {
            *out = m.map;
            return true;
        }
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes, box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    Entry& e = cache[next];
    if (fn(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        e.base = nullptr;
        return false;
    }
    e.base = base;
    e.row_bytes = row_bytes;
    e.rows = rows;
    e.box_bytes = box_bytes;
    e.box_rows = box_rows;
    e.swz = swizzle128;
    *out = e.map;
    next = (next + 1) % 32;
    return true;
}

cudaError_t launch_q4k_rows_gemv(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x,
                                 const float* gamma, float eps, int N, int K, bool swiglu, cudaStream_t s) {
    if (w1) return run_rows<2, false>(y0, y1, w0, w1, x, gamma, eps, N, K, swiglu, s);
    return run_rows<1, false>(y0, nullptr, w0, nullptr, x, gamma, eps, N, K, false, s);
}

cudaError_t launch_q4k_rows_pure_read(float* sink, const uint8_t* w, int N, int K, cudaStream_t s) {
    return run_rows<1, true>(sink, nullptr, w, nullptr, nullptr, nullptr, 0.f, N, K, false, s);
}

}  // namespace q4
