// Planar Q4 decode GEMV for one input vector, with the input held in registers (sm_103a).
//
// Format (inferencelayer `kernel_lab.rs`, shader GEMV_F16S): row n is K/32 blocks; block b has 16 packed bytes
// qs[n][b][0..15] (byte j: weight j in the low nibble, weight j+16 in the high nibble) and an f16 scale
// d[n][b]; the weight is (q - 8) * d.
//
// Kernel shape (one persistent CTA of W warps per SM):
//  * lane l always works on the units (16-byte blocks) l, l+32, ... of a row, so the staged input it needs is
//    the same for every row: after one cooperative staging pass through shared memory, each lane keeps its
//    UPL units of x (pre-scaled for the bias-free decode, 32 floats per unit) plus each unit's factor and
//    -8 offset term in registers, and the unit loop reads nothing but weights from shared memory;
//  * every warp owns a ring of D slots of R whole rows (quants, then scales), each filled by two bulk copies
//    on the slot's mbarrier; the whole ring is requested before the kernel waits for its predecessor in the
//    stream, and a slot is refilled as soon as the warp has consumed it;
//  * per unit and row: one shift and eight ANDs per word turn codes into floats, four packed fp32x2 FMAs
//    per word accumulate in the common chain order (word_fma), t = A * 2^(22+e) + bias, and the row adds
//    d * t; the R row totals of a job meet in one transposing warp reduction;
//  * a stage wait that runs out of its limit makes the warp stop: it issues no more copies, writes its
//    remaining rows as NaN, records kFaultWaitTimeout, and before exiting waits (bounded) for the copies it
//    had already issued, so no copy lands in the shared memory of an exited CTA.
// Lane l's units are visited in increasing order with the same fold and the same reduction tree as the
// batched kernel (q4_dense.cuh), so a row's result is bit-identical to that kernel's row for the same input.
#pragma once

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {
namespace xr {

struct XrParams {
    float* y;
    const uint8_t* qs;
    const uint16_t* d;
    const float* x;
    int N, nblk;
    int jobs;               // row groups of R rows
    long long wait_cycles;  // limit of one stage wait
    unsigned* fault;        // device fault word
    uint32_t slot_bytes;
    uint32_t xs_off, fac_off, slots_off;  // mbarriers at offset 0
};

__host__ __device__ constexpr uint32_t round_up(uint32_t a, uint32_t b) { return (a + b - 1) / b * b; }

// 16 bits from shared memory into a 16-bit register (an f16 scale, converted without masking)
__device__ __forceinline__ unsigned short lds_h16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// R rows per job, W warps, ring depth D, UPL units per lane (K/32 <= 32*UPL), PRE stages requested before the
// dependency wait (the rest right after the input is staged), FULL: K/32 == 32*UPL (no short last unit).
template <int R, int W, int D, int UPL, int PRE, bool FULL, bool PURE>
__global__ void __launch_bounds__(W * 32, 1) q4_xr_kernel(const XrParams p) {
    static_assert(PRE >= 1 && PRE <= D, "stages before the dependency wait");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t s_base = smem_addr(smem);
    const uint32_t bars = s_base + (uint32_t)(warp * D) * 8u;
    // whole rows of exactly 32*UPL blocks: row strides and the slot size are compile-time constants
    const uint32_t QROW = FULL ? 512u * UPL : (uint32_t)p.nblk * 16u;
    const uint32_t SROW = FULL ? 64u * UPL : (uint32_t)p.nblk * 2u;
    const uint32_t SLOT = FULL ? (R * 576u * UPL + 127u) / 128u * 128u : p.slot_bytes;
    const uint32_t ring = s_base + p.slots_off + (uint32_t)(warp * D) * SLOT;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < D; ++k) mbar_init(bars + 8u * k, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    // Warps are numbered across CTAs first, so a small job count still spreads over all SMs.
    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;
    const int Wtot = (int)gridDim.x * W;
    const int my_jobs = gw < p.jobs ? (p.jobs - 1 - gw) / Wtot + 1 : 0;
    const uint64_t pol = policy_evict_first();

    // stage j of this warp (job gw + j * Wtot) into slot j % D
    auto issue = [&](int j) {
        if (lane == 0) {
            const int r0 = (gw + j * Wtot) * R;
            const uint32_t rv = (uint32_t)min(R, p.N - r0);
            const uint32_t bar = bars + 8u * (uint32_t)(j % D);
            const uint32_t dst = ring + (uint32_t)(j % D) * SLOT;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(bar, rv * (QROW + SROW));
            bulk_copy(dst, p.qs + (size_t)r0 * QROW, rv * QROW, bar, pol);
            bulk_copy(dst + R * QROW, p.d + (size_t)r0 * p.nblk, rv * SROW, bar, pol);
        }
    };
    // the weights are constant, so their first stages need not wait for the previous kernel
    int issued = min(PRE, my_jobs);
    for (int j = 0; j < issued; ++j) issue(j);

    // The input and the outputs may belong to the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();

    if constexpr (!PURE) {
        // Stage x: four lanes per 32-element block (lane t of a group holds elements 8t .. 8t+7), quads stored
        // lane-major per unit (float4 [UPL][8][32 + 1 pad], the rows of the chunk-major layout) so that each
        // lane's register loads and the four lanes' stores are conflict-free. Every thread issues all of its
        // loads before using any, so staging costs one round trip to the L2.
        float4* const xs = reinterpret_cast<float4*>(smem + p.xs_off);
        float* const fs = reinterpret_cast<float*>(smem + p.fac_off);
        constexpr int kIter = (32 * UPL * 4 + W * 32 - 1) / (W * 32);  // block-quarters per thread
        const int t4 = lane & 3;
        float4 xa[kIter], xb[kIter];
#pragma unroll
        for (int j = 0; j < kIter; ++j) {
            const int blk = ((int)threadIdx.x + j * W * 32) >> 2;
            const float4* src = reinterpret_cast<const float4*>(p.x) + (size_t)blk * 8 + 2 * t4;
            const bool in = blk < p.nblk;
            xa[j] = in ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
            xb[j] = in ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        int ej[kIter];
        stage_blocks4<kIter>(xa, xb, t4 >> 1, ej);  // every lane takes part in the shuffles
#pragma unroll
        for (int j = 0; j < kIter; ++j) {
            const int blk = ((int)threadIdx.x + j * W * 32) >> 2;
            if (blk < p.nblk) {
                float4* q = xs + ((blk >> 5) * 8 + 2 * t4) * kXRow + (blk & 31);
                q[0] = xa[j];
                q[kXRow] = xb[j];
                if (t4 == 0) fs[blk] = block_factor(ej[j]);
            }
        }
        __syncthreads();
    }
    for (int j = issued; j < min(D, my_jobs); ++j) issue(j);
    issued = min(D, my_jobs);

    // Lane l's input for unit i (quads, factor and -8 offset term) in registers, loaded during the first job just
    // before the unit is first used, so the loads overlap the decode of the units before it.
    float4 xr[PURE ? 1 : UPL][8];
    float fac[PURE ? 1 : UPL], bias[PURE ? 1 : UPL];
    auto load_unit = [&](int i) {
        if constexpr (!PURE) {
            const float4* const xs = reinterpret_cast<const float4*>(smem + p.xs_off);
            const bool in = FULL || i * 32 + lane < p.nblk;
#pragma unroll
            for (int q = 0; q < 8; ++q) xr[i][q] = in ? xs[(i * 8 + q) * kXRow + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
            fac[i] = in ? reinterpret_cast<const float*>(smem + p.fac_off)[i * 32 + lane] : 1.0f;
            bias[i] = in ? q4_block_bias(xr[i], fac[i]) : 0.0f;
        }
    };

    // A job's R row totals are reduced across the warp after the next job's wait, so that the shuffles can
    // overlap that job's first loads.
    constexpr int P2R = NextPow2<R>::value;
    constexpr int LR = log2_const<P2R>();
    float prev[P2R];
    int prev_g = -1;
    bool prev_nan = false;
    bool aborted = false;
    int consumed = 0;
    auto reduce_store = [&]() {
        warp_transpose_reduce<P2R>(prev, lane);
        const int idx = lane >> (5 - LR);
        const int row = (gw + prev_g * Wtot) * R + idx;
        if ((lane & ((1 << (5 - LR)) - 1)) == 0 && idx < R && row < p.N) p.y[row] = prev_nan ? NAN : prev[0];
    };

    // One job: wait for its stage, decode and accumulate its R rows, refill the slot.
    auto job = [&](int g, auto first) {
        constexpr bool FIRST = decltype(first)::value;
        const uint32_t slot = (uint32_t)(g % D);
        if (!aborted) {
            if (warp_wait_bounded(bars + 8u * slot, (uint32_t)((g / D) & 1), p.wait_cycles)) {
                consumed = g + 1;
            } else {
                aborted = true;
                if (lane == 0) atomicOr(p.fault, kFaultWaitTimeout);
            }
        }
        if constexpr (!PURE) {
            if (prev_g >= 0) reduce_store();
        }
        float cur[P2R];
#pragma unroll
        for (int r = 0; r < P2R; ++r) cur[r] = 0.f;
        if (!aborted) {
            const uint32_t sq = ring + slot * SLOT + (uint32_t)lane * 16u;
            const uint32_t sd = ring + slot * SLOT + R * QROW + (uint32_t)lane * 2u;
            uint32_t fold[R];
#pragma unroll
            for (int r = 0; r < R; ++r) fold[r] = 0u;
#pragma unroll
            for (int i = 0; i < UPL; ++i) {
                if constexpr (FIRST) load_unit(i);
                if (!FULL && i == UPL - 1 && i * 32 + lane >= p.nblk) break;  // a short last unit round
                uint4 w[R];
                unsigned short db[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    w[r] = lds128(sq + (uint32_t)r * QROW + (uint32_t)(i * 512));
                    db[r] = lds_h16(sd + (uint32_t)r * SROW + (uint32_t)(i * 64));
                }
                if constexpr (PURE) {
#pragma unroll
                    for (int r = 0; r < R; ++r) fold[r] ^= w[r].x ^ w[r].y ^ w[r].z ^ w[r].w ^ (uint32_t)db[r];
                } else {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float2 a = word_fma(decode_word_sub(w[r].x), xr[i][0], xr[i][4], make_float2(0.f, 0.f));
                        a = word_fma(decode_word_sub(w[r].y), xr[i][1], xr[i][5], a);
                        a = word_fma(decode_word_sub(w[r].z), xr[i][2], xr[i][6], a);
                        a = word_fma(decode_word_sub(w[r].w), xr[i][3], xr[i][7], a);
                        const float t = fmaf(a.x + a.y, fac[i], bias[i]);
                        cur[r] = fmaf(__half2float(__ushort_as_half(db[r])), t, cur[r]);
                    }
                }
            }
            __syncwarp();  // every lane is done with the slot before it is refilled
            if (issued < my_jobs) issue(issued++);
            if constexpr (PURE) {
                const int r0 = (gw + g * Wtot) * R;
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) fold[r] ^= __shfl_xor_sync(0xffffffffu, fold[r], off);
                    if (lane == 0 && r0 + r < p.N) p.y[r0 + r] = __uint_as_float(fold[r]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < P2R; ++r) prev[r] = cur[r];
        prev_g = g;
        prev_nan = aborted;  // rows of a job whose wait ran out (or any later job) are NaN
    };

    if (my_jobs > 0) {
        job(0, std::true_type{});
        for (int g = 1; g < my_jobs; ++g) job(g, std::false_type{});
        if constexpr (!PURE) reduce_store();
    }
    if constexpr (PURE) {
        // rows of jobs after a timed-out wait were never written: store NaN there
        for (int g = consumed; g < my_jobs; ++g) {
            const int r0 = (gw + g * Wtot) * R;
            if (lane < R && r0 + lane < p.N) p.y[r0 + lane] = NAN;
        }
    }
    // copies issued but not consumed (only after a wait ran out): let them land before the CTA exits
    for (int s = consumed; s < issued; ++s)
        if (!warp_wait_bounded(bars + 8u * (uint32_t)(s % D), (uint32_t)((s / D) & 1), kDrainCycles) && lane == 0)
            atomicOr(p.fault, kFaultCopyLost);
}

// Shared memory: [mbarriers W*D*8, 512 B][staged x UPL*4 KB][factors UPL*128 B][rings W*D*slot].
template <int R, int W, int D, int UPL, int PRE, bool PURE>
cudaError_t launch_xr(const DeviceInfo& di, float* y, const uint8_t* qs, const uint16_t* d, const float* x, int N,
                      int K, cudaStream_t s) {
    static_assert(W * D * 8 <= 512, "mbarrier area");
    const int nblk = K / 32;
    if (nblk % 8 != 0 || nblk > 32 * UPL || nblk <= 32 * (UPL - 1) || (reinterpret_cast<uintptr_t>(d) & 15u) != 0)
        return cudaErrorNotSupported;
    XrParams p;
    p.y = y;
    p.qs = qs;
    p.d = d;
    p.x = x;
    p.N = N;
    p.nblk = nblk;
    p.jobs = (N + R - 1) / R;
    p.wait_cycles = wait_limit_cycles();
    p.fault = device_fault_word(di.device);
    if (!p.fault) return cudaErrorInvalidSymbol;
    p.slot_bytes = round_up((uint32_t)(R * nblk * 18), 128u);
    p.xs_off = 512;
    p.fac_off = p.xs_off + (PURE ? 0u : (uint32_t)UPL * 8u * kXRow * 16u);
    p.slots_off = round_up(p.fac_off + (PURE ? 0u : (uint32_t)UPL * 128u), 128u);
    const uint32_t smem = p.slots_off + (uint32_t)(W * D) * p.slot_bytes;
    if (smem > (uint32_t)di.max_smem_optin) return cudaErrorNotSupported;
    auto kern = nblk == 32 * UPL ? q4_xr_kernel<R, W, D, UPL, PRE, true, PURE> : q4_xr_kernel<R, W, D, UPL, PRE, false, PURE>;
    static std::once_flag attr_once[2][64];
    cudaError_t err = cudaSuccess;
    std::call_once(attr_once[nblk == 32 * UPL ? 1 : 0][di.device & 63], [&] {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (err != cudaSuccess) return err;
    const int grid = std::min(di.sm_count, p.jobs);
    return launch_kernel(kern, grid, W * 32, smem, s, p);
}

}  // namespace xr
}  // namespace q4
