// Planar Q4 decode GEMV kernel template (sm_103a): single vector, small batch (V <= 16 vectors sharing one
// sweep over the weights) and the pure-read ceiling instrument. Included by the kernels_q4*.cu translation
// units, which instantiate disjoint sets of batch widths so that they compile in parallel.
//
// Format (inferencelayer `kernel_lab.rs`, shader GEMV_F16S): row n of the weight matrix is K/32 blocks;
// block b of row n has 16 packed bytes qs[n][b][0..15] and one f16 scale d[n][b]. Byte j holds weight j
// in its low nibble and weight j+16 in its high nibble; the weight is (q - 8) * d.
//
// Kernel shape (one persistent CTA of W warps per SM):
//  * the V input vectors are staged once per CTA in shared memory, block by block: each element is
//    pre-scaled for the bit position of its code and its block's exponent bound, and beside each block sit
//    its factor 2^(22+e) and the -8 offset term of the block (q4_block_bias: the unit chain on codes of 8, so
//    a block of zero weights contributes exactly zero; device_common.cuh, bias-free decode);
//  * every warp owns a ring of D shared-memory slots; a slot holds R consecutive rows x CB = 32*UPL blocks
//    (quants, then scales), so each weight byte is read from HBM once and all V vectors use it. Whole rows of
//    exactly CB blocks travel as two bulk copies (quants, scales) issued by lane 0 on the slot's mbarrier;
//    chunks of longer rows by warp-cooperative 16-byte cp.async;
//  * lane l handles units l, l+32, ... of every row in the slot, in increasing order whatever CB is, so
//    the per-row summation order depends only on K: batched rows equal single-vector calls bit for bit;
//  * per 32-bit word: one shift and eight ANDs turn the codes into floats, and four packed fp32x2 FMAs per
//    vector accumulate against the staged quads in the common chain order (word_fma); per block:
//    t = A * 2^(22+e) + bias, then d * t;
//  * the per-stage control is incremental (no division in the loop) and full chunks run unguarded;
//  * at the end of a row group the R*V totals are summed across the warp with a transposing shuffle
//    reduction and stored;
//  * a stage wait (bulk mode) that runs out of its limit makes the warp stop issuing copies and store its
//    remaining rows as NaN (kFaultWaitTimeout); before exiting it waits, bounded, for the copies it issued.
#pragma once

#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {
namespace dense {

struct Q4Params {
    float* y;
    const uint8_t* qs;
    const uint16_t* d;
    const float* x;
    int N, K, nblk;
    int S;      // chunks per row
    int jobs;   // row groups of R rows
    int dcopy;  // scales move by 16-byte copies (else the warp loads them into the slot itself)
    int bulk;   // every stage is whole rows: one bulk copy each for quants and scales, on a slot mbarrier
    long long wait_cycles;  // limit of one stage wait
    unsigned* fault;        // device fault word
    uint32_t xs_off, aux_off, bar_off, slots_off;
};

__host__ __device__ constexpr uint32_t round_up_u(uint32_t a, uint32_t b) { return (a + b - 1) / b * b; }

template <int R, int UPL>
__host__ __device__ constexpr uint32_t slot_bytes() {
    return round_up_u((uint32_t)(R * 32 * UPL * 16 + R * 32 * UPL * 2), 128u);
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

template <int V, int R, int W, int D, int UPL, bool PURE>
__global__ void __launch_bounds__(W * 32, 1) q4_gemv_kernel(const Q4Params p) {
    constexpr int CB = 32 * UPL;
    constexpr uint32_t QROW = CB * 16u;
    constexpr uint32_t QBYTES = R * QROW;
    constexpr uint32_t SLOT = slot_bytes<R, UPL>();
    constexpr int kThreads = W * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;

    const uint32_t s_base = smem_addr(smem);
    const uint32_t xs = s_base + p.xs_off;
    const uint32_t aux = s_base + p.aux_off;
    const uint32_t ring = s_base + p.slots_off + (uint32_t)warp * (uint32_t)(D * SLOT);
    const uint32_t bars = s_base + p.bar_off + (uint32_t)(warp * D) * 8u;  // one mbarrier per slot (bulk mode)
    if (p.bulk) {
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < D; ++k) mbar_init(bars + 8u * k, 1u);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
    }

    // Warps are numbered across CTAs first so that a small job count still spreads over all SMs.
    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;
    const int Wtot = (int)gridDim.x * W;
    const uint64_t pol = policy_evict_first();

    // Issue pointer: the next stage to copy (job, chunk) and its slot. One commit group per call, empty
    // once this warp has no stage left, so the wait below always counts D - 1 groups ahead.
    int ijob = gw, ic = 0, islot = 0;
    int nissued = 0;        // stages issued (bulk mode)
    bool aborted = false;   // a stage wait ran out: no more copies, the warp's remaining rows are NaN
    auto issue = [&]() {
        if (ijob < p.jobs && !aborted) {
            const int r0 = ijob * R;
            const int rv = min(R, p.N - r0);
            const int b0 = ic * CB;
            const int nb = min(CB, p.nblk - b0);
            const uint32_t slot = ring + (uint32_t)islot * SLOT;
            if (p.bulk) {
                // lane 0 moves the rows' quants and scales; this warp's earlier reads of the slot are ordered
                // before the asynchronous write
                if (lane == 0) {
                    const uint32_t bar = bars + 8u * (uint32_t)islot;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(bar, (uint32_t)rv * (QROW + CB * 2));
                    bulk_copy(slot, p.qs + (size_t)r0 * QROW, (uint32_t)rv * QROW, bar, pol);
                    bulk_copy(slot + QBYTES, p.d + (size_t)r0 * CB, (uint32_t)(rv * CB * 2), bar, pol);
                }
                ++nissued;
            } else if (nb == CB && p.S == 1) {
                warp_copy_async(slot, p.qs + (size_t)r0 * QROW, (uint32_t)rv * QROW, lane, pol);
                if (p.dcopy)
                    warp_copy_async(slot + QBYTES, p.d + (size_t)r0 * CB, (uint32_t)(rv * CB * 2), lane, pol);
            } else {
                for (int r = 0; r < rv; ++r) {
                    const size_t rb = (size_t)(r0 + r) * p.nblk + b0;
                    warp_copy_async(slot + (uint32_t)r * QROW, p.qs + rb * 16, (uint32_t)(nb * 16), lane, pol);
                    if (p.dcopy)
                        warp_copy_async(slot + QBYTES + (uint32_t)(r * CB * 2), p.d + rb, (uint32_t)(nb * 2), lane,
                                        pol);
                }
            }
            if (!p.dcopy) {
                // scales that cannot move by 16-byte copies (not 16-byte aligned, or K/32 not a multiple of 8)
                // go into the slot by plain loads, so the unit loop always reads them from shared memory
                uint16_t* const ds =
                    reinterpret_cast<uint16_t*>(smem + p.slots_off + (size_t)(warp * D + islot) * SLOT + QBYTES);
                for (int r = 0; r < rv; ++r)
                    for (int u = lane; u < nb; u += 32) ds[r * CB + u] = __ldg(p.d + (size_t)(r0 + r) * p.nblk + b0 + u);
            }
            if (++ic == p.S) {
                ic = 0;
                ijob += Wtot;
            }
            islot = islot + 1 == D ? 0 : islot + 1;
        }
        if (!p.bulk) cp_async_commit();
    };

#pragma unroll
    for (int k = 0; k < D - 1; ++k) issue();

    // The weights are constant; the input and the outputs may belong to the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();

    if constexpr (!PURE) {
        // Stage the V vectors (X is [V][K]): four lanes per 32-element block, lane t of the group holding
        // float4 2t and 2t+1 (quads 2t, 2t+1 of the unit); loads are issued kStageU/2 blocks ahead. The loop
        // covers whole warps (the block count rounded up to 8) so the group shuffles always see 32 lanes.
        const int nb_all = V * p.nblk;
        const int t4 = lane & 3;
        const int nthr = ((nb_all * 4 + 31) & ~31);
        // each thread issues the loads of kBatch block quarters before using any (batches sized so that one
        // batch covers a thread's quarters of 2 to 4 vectors at K = 4096: one L2 round trip), then stages them
        // together
        constexpr int kBatch = V >= 3 ? 8 : V == 2 ? 4 : kStageU / 2;
        for (int base = threadIdx.x; base < nthr; base += kThreads * kBatch) {
            float4 xa[kBatch], xb[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int blk = (base + j * kThreads) >> 2;
                const bool in = blk < nb_all;
                const float4* src = reinterpret_cast<const float4*>(p.x) + (size_t)blk * 8 + 2 * t4;
                xa[j] = in ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
                xb[j] = in ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            int ej[kBatch];
            stage_blocks4<kBatch>(xa, xb, t4 >> 1, ej);  // quarters past the end stage zeros and are not stored
            DivWalk vu(base >> 2, kThreads >> 2, p.nblk);  // (vector, block) of quarter j's block
#pragma unroll
            for (int j = 0; j < kBatch; ++j, vu.next()) {
                const int blk = (base + j * kThreads) >> 2;
                if (blk < nb_all) {
                    const int v = vu.q;
                    const uint32_t u = (uint32_t)vu.r;
                    const uint32_t a0 = xs + xs_chunk_offset((uint32_t)v, (uint32_t)(2 * t4), u, (uint32_t)V);
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "f"(xa[j].x), "f"(xa[j].y),
                                 "f"(xa[j].z), "f"(xa[j].w)
                                 : "memory");
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + kXRow * 16u), "f"(xb[j].x),
                                 "f"(xb[j].y), "f"(xb[j].z), "f"(xb[j].w)
                                 : "memory");
                    if (t4 == 0)
                        asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(aux + aux_offset((uint32_t)v, u, (uint32_t)V)),
                                     "f"(block_factor(ej[j])), "f"(0.0f)
                                     : "memory");
                }
            }
        }
        __syncthreads();
        // each block's -8 offset term: the unit chain on codes of 8 over its staged quads
        DivWalk vu((int)threadIdx.x, kThreads, p.nblk);
        for (int b = threadIdx.x; b < nb_all; b += kThreads, vu.next()) {
            const int v = vu.q;
            const uint32_t u = (uint32_t)vu.r;
            float4 xq[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) xq[q] = lds128f(xs + xs_chunk_offset((uint32_t)v, (uint32_t)q, u, (uint32_t)V));
            const uint32_t a = aux + aux_offset((uint32_t)v, u, (uint32_t)V);
            const float bias = q4_block_bias(xq, lds32f(a));
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(a + 4u), "f"(bias) : "memory");
        }
    }
    __syncthreads();

    // Plain pointers into the shared array (not asm address operands), so that the unit offsets below fold
    // into the loads' immediates.
    const float4* const xs_p = reinterpret_cast<const float4*>(smem + p.xs_off) + lane;
    const float2* const aux_p = reinterpret_cast<const float2*>(smem + p.aux_off) + lane;
    const uint8_t* const ring_p = smem + p.slots_off + (size_t)warp * (D * SLOT);

    float tot[R][V];
    uint32_t fold[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        fold[r] = 0u;
#pragma unroll
        for (int v = 0; v < V; ++v) tot[r][v] = 0.f;
    }

    const int my_jobs = gw < p.jobs ? (p.jobs - 1 - gw) / Wtot + 1 : 0;
    const int total = my_jobs * p.S;
    int job = gw, c = 0, cslot = 0;
    uint32_t cphase = 0u;
    int consumed = 0;  // stages whose wait completed (bulk mode)
    for (int g = 0; g < total; ++g) {
        issue();  // stage g + D - 1 into the slot consumed at g - 1
        // stage g has landed: its slot's mbarrier completed phase cphase (bounded wait), or its commit group
        if (p.bulk) {
            if (!aborted) {
                if (warp_wait_bounded(bars + 8u * (uint32_t)cslot, cphase, p.wait_cycles)) {
                    consumed = g + 1;
                } else {
                    aborted = true;
                    if (lane == 0) atomicOr(p.fault, kFaultWaitTimeout);
                }
            }
        } else {
            cp_async_wait<D - 1>();
        }
        __syncwarp();
        const uint8_t* const slot_p = ring_p + cslot * SLOT;
        const int r0 = job * R;
        const int rv = min(R, p.N - r0);
        const int b0 = c * CB;
        const int nb = min(CB, p.nblk - b0);
        const uint4* const qb = reinterpret_cast<const uint4*>(slot_p) + lane;
        const uint16_t* const db = reinterpret_cast<const uint16_t*>(slot_p + QBYTES) + lane;
        const float4* const xb = xs_p + (b0 >> 5) * (V * 8 * (int)kXRow);
        const float2* const ab = aux_p + (b0 >> 5) * (V * 32);

        auto unit = [&](const int it) {
            uint4 w[R];
            float dsc[R];
            uint32_t dbits[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                w[r] = qb[r * (QROW / 16) + it * 32];
                dbits[r] = db[r * CB + it * 32];
                dsc[r] = f16_bits_to_f32(dbits[r]);
            }
            if constexpr (PURE) {
#pragma unroll
                for (int r = 0; r < R; ++r) fold[r] ^= w[r].x ^ w[r].y ^ w[r].z ^ w[r].w ^ dbits[r];
            } else {
                // one fp32x2 chain per row and vector, in the common word order
                float2 acc[R][V];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    Word8s d8[R];
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        d8[r] = decode_word_sub(i == 0 ? w[r].x : i == 1 ? w[r].y : i == 2 ? w[r].z : w[r].w);
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const float4* const xa = xb + (it * V + v) * (8 * (int)kXRow) + i * (int)kXRow;
                        const float4 xl = xa[0];
                        const float4 xh = xa[4 * (int)kXRow];
#pragma unroll
                        for (int r = 0; r < R; ++r)
                            acc[r][v] = word_fma(d8[r], xl, xh, i == 0 ? make_float2(0.f, 0.f) : acc[r][v]);
                    }
                }
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float2 fa = ab[(it * V + v) * 32];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float t = fmaf(acc[r][v].x + acc[r][v].y, fa.x, fa.y);
                        tot[r][v] = fmaf(dsc[r], t, tot[r][v]);
                    }
                }
            }
        };
        if (aborted) {
            // no compute after a timed-out wait; the rows are stored as NaN below
        } else if constexpr (R * V <= 2) {
            // short bodies: unrolled, so neighbouring units overlap; full chunks run unguarded
            if (nb == CB) {
#pragma unroll
                for (int it = 0; it < UPL; ++it) unit(it);
            } else {
#pragma unroll
                for (int it = 0; it < UPL; ++it)
                    if (it * 32 + lane < nb) unit(it);
            }
        } else {
            // long bodies (R*V independent chains already): one copy of the unit, so the loop stays in the
            // instruction cache
#pragma unroll 1
            for (int it = 0; it < UPL; ++it)
                if (it * 32 + lane < nb) unit(it);
        }
        __syncwarp();  // every lane is done with this slot before a later stage overwrites it

        if (c == p.S - 1) {
            if constexpr (PURE) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) fold[r] ^= __shfl_xor_sync(0xffffffffu, fold[r], off);
                    if (lane == 0 && r < rv) p.y[r0 + r] = aborted ? NAN : __uint_as_float(fold[r]);
                    fold[r] = 0u;
                }
            } else {
                constexpr int NV = R * V;
                constexpr int P2 = NextPow2<NV>::value;
                constexpr int L2 = log2_const<P2>();
                float vals[P2];
#pragma unroll
                for (int i = 0; i < P2; ++i) vals[i] = 0.f;
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        vals[r * V + v] = tot[r][v];
                        tot[r][v] = 0.f;
                    }
                warp_transpose_reduce<P2>(vals, lane);
                const int idx = lane >> (5 - L2);
                const bool leader = (lane & ((1 << (5 - L2)) - 1)) == 0;
                if (leader && idx < NV) {
                    const int r = idx / V;
                    const int v = idx - r * V;
                    if (r < rv)
                        p.y[(size_t)v * p.N + r0 + r] = aborted ? NAN : vals[0];
                }
            }
        }
        if (++c == p.S) {
            c = 0;
            job += Wtot;
        }
        if (++cslot == D) {
            cslot = 0;
            cphase ^= 1u;
        }
    }
    // bulk copies issued but not consumed (only after a wait ran out): let them land before the CTA exits
    for (int st = consumed; st < nissued; ++st)
        if (!warp_wait_bounded(bars + 8u * (uint32_t)(st % D), (uint32_t)((st / D) & 1), kDrainCycles) && lane == 0)
            atomicOr(p.fault, kFaultCopyLost);
}

template <int V, int R, int W, int D, int UPL, bool PURE>
cudaError_t launch_fixed(const DeviceInfo& di, float* y, const uint8_t* qs, const uint16_t* d, const float* x, int N,
                         int K, bool dcopy, cudaStream_t s) {
    constexpr int CB = 32 * UPL;
    const uint32_t nblk = (uint32_t)K / 32u;
    const uint32_t xsb = PURE ? 0u : xs_chunk_bytes((uint32_t)V, nblk);
    const uint32_t axb = PURE ? 0u : aux_bytes((uint32_t)V, nblk);
    const uint32_t barb = round_up_u((uint32_t)(W * D * 8), 128u);  // slot mbarriers
    const uint32_t smem = xsb + axb + barb + (uint32_t)(W * D) * slot_bytes<R, UPL>();
    if (smem > (uint32_t)di.max_smem_optin) return cudaErrorNotSupported;
    auto kern = q4_gemv_kernel<V, R, W, D, UPL, PURE>;
    static std::once_flag attr_once[64];
    cudaError_t err = cudaSuccess;
    std::call_once(attr_once[di.device & 63], [&] {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (err != cudaSuccess) return err;
    Q4Params p;
    p.y = y;
    p.qs = qs;
    p.d = d;
    p.x = x;
    p.N = N;
    p.K = K;
    p.nblk = (int)nblk;
    p.S = (int)((nblk + CB - 1) / CB);
    p.jobs = (N + R - 1) / R;
    p.dcopy = dcopy ? 1 : 0;
    p.bulk = (dcopy && p.S == 1 && (int)nblk == CB) ? 1 : 0;
    p.wait_cycles = wait_limit_cycles();
    p.fault = device_fault_word(di.device);
    if (!p.fault) return cudaErrorInvalidSymbol;
    p.xs_off = 0;
    p.aux_off = xsb;
    p.bar_off = xsb + axb;
    p.slots_off = xsb + axb + barb;
    const int grid = std::min(di.sm_count, p.jobs);
    return launch_kernel(kern, grid, W * 32, smem, s, p);
}

// The deepest ring among the instantiated depths {2, 3, 4, 5, 6, 8} not above DMAX nor `want` that fits.
template <int V, int R, int W, int DMAX, int UPL, bool PURE>
cudaError_t launch_upl(const DeviceInfo& di, float* y, const uint8_t* qs, const uint16_t* d, const float* x, int N,
                       int K, bool dcopy, int want, cudaStream_t s) {
    cudaError_t e = cudaErrorNotSupported;
#define Q4_TRY_DEPTH(DD)                                                                              \
    if constexpr (DMAX >= DD)                                                                         \
        if (e == cudaErrorNotSupported && want >= DD)                                                 \
            e = launch_fixed<V, R, W, DD, UPL, PURE>(di, y, qs, d, x, N, K, dcopy, s);
    Q4_TRY_DEPTH(8)
    Q4_TRY_DEPTH(6)
    Q4_TRY_DEPTH(5)
    Q4_TRY_DEPTH(4)
    Q4_TRY_DEPTH(3)
#undef Q4_TRY_DEPTH
    if (e == cudaErrorNotSupported) e = launch_fixed<V, R, W, 2, UPL, PURE>(di, y, qs, d, x, N, K, dcopy, s);
    return e;
}

// Units per lane: the whole row in one chunk up to min(K/32, 32*upl_max) blocks (UPL = 1, 2, 4), longer rows
// in chunks of that size; smaller chunks when the rings would not fit beside the staged input.
template <int V, int R, int W, int DMAX, bool PURE>
cudaError_t launch(const DeviceInfo& di, float* y, const uint8_t* qs, const uint16_t* d, const float* x, int N, int K,
                   int depth, int upl_max, cudaStream_t s) {
    const int nblk = K / 32;
    const bool dcopy = (nblk % 8 == 0) && ((reinterpret_cast<uintptr_t>(d) & 15u) == 0);
    depth = std::min(depth, DMAX);
    const int upl0 = std::min(nblk <= 32 ? 1 : nblk <= 64 ? 2 : 4, upl_max);
    cudaError_t e = cudaErrorNotSupported;
    if (upl0 == 4) e = launch_upl<V, R, W, DMAX, 4, PURE>(di, y, qs, d, x, N, K, dcopy, depth, s);
    if (e == cudaErrorNotSupported && upl0 >= 2)
        e = launch_upl<V, R, W, DMAX, 2, PURE>(di, y, qs, d, x, N, K, dcopy, depth, s);
    if (e == cudaErrorNotSupported) e = launch_upl<V, R, W, DMAX, 1, PURE>(di, y, qs, d, x, N, K, dcopy, depth, s);
    return e;
}

// Per-translation-unit entry points (kernels_q4_*.cu).
cudaError_t gemv_v1(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int N, int K,
                    cudaStream_t s);
cudaError_t gemv_v2_4(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V,
                      int N, int K, cudaStream_t s);
cudaError_t gemv_v5_8(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V,
                      int N, int K, cudaStream_t s);
cudaError_t gemv_v9_16(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V,
                       int N, int K, cudaStream_t s);

}  // namespace dense
}  // namespace q4
