// Batched (unfused) Q4_K decode GEMV for sm_103a: Y[v][n] = sum_k W[n][k] * X[v][k] for v < V <= 8, reading
// every weight byte once for all V vectors.
//
// Format: trueno-gpu `fused.rs`, FusedRmsNormQ4KGemvKernel phase 3 (144-byte super-blocks of 256 weights;
// value d*sc_j*q - dmin*m_j); the page also names an unfused Q4KGemvKernel. Batched contract as the planar
// form (spark_model `gemm_quant.rs`, dense_gemv_batchm: one sweep for all rows).
//
// Kernel shape (one persistent CTA of W warps per SM), the Q4_K kernel's with V vectors:
//  * the V vectors are staged once per CTA, each 32-element sub-block with its own exponent bound e_{j,v}
//    (bias-free decode, device_common.cuh), with the two code halves interleaved: quad 2i + g of a unit (16 quant
//    bytes: half of sub-block 2c in the low nibbles, the same half of 2c+1 in the high ones) holds the inputs of
//    word i's bytes 2g and 2g+1 as (low, high, low, high), so one packed FMA takes a byte's low code into the .x
//    lane and its high code into the .y lane of one accumulator; beside each unit sit (S_lo, S_hi, f_lo, f_hi):
//    f = 2^(22+e) of the two sub-blocks and S = f times the unit's FMA chain run on codes of 1 over each half;
//  * each warp streams R rows (whole rows when they fit) through its own ring of cp.async slots;
//  * lane l takes unit l (+32, ...) of every row: chunk c = (l%8)/2, half l%2; the 8 lanes of a super-block
//    each decode one sub-block's header entry (d*sc_j and dmin*m_j), shared with the group by shuffles;
//  * per word: one shift + eight ANDs per row, then for each vector two staged-input loads (shared by the R
//    rows) and four packed FMAs per row into the row's (low half, high half) accumulator pair; per unit and
//    vector the two halves fold as fl(d*sc*f * A) - fl(dmin*m * S) with unfused rounded operations, so halves
//    whose weights are all zero (sc = m = 0, or a constant power-of-two code with d*sc*q = dmin*m) contribute
//    exactly zero;
//  * the R*V totals are summed over the warp with the transposing shuffle reduction and stored.
#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

struct Q4KBParams {
    float* y;
    const uint8_t* w;
    const float* x;
    int N, K, nsb;
    int CS, S, jobs, slot_bytes;
    uint32_t xs_off, ssum_off, slots_off;
};

// The 8 codes of a word as (low, high) pairs of its bytes 0..3, at the bit positions of decode_word_sub.
struct Word4p {
    float2 b0, b1, b2, b3;
};
__device__ __forceinline__ Word4p decode_word_pairs(uint32_t w) {
    const uint32_t s = w >> 12;
    Word4p r;
    r.b0 = make_float2(__uint_as_float(w & 0x0000000Fu), __uint_as_float(w & 0x000000F0u));
    r.b1 = make_float2(__uint_as_float(w & 0x00000F00u), __uint_as_float(w & 0x0000F000u));
    r.b2 = make_float2(__uint_as_float(w & 0x000F0000u), __uint_as_float(s & 0x00000F00u));
    r.b3 = make_float2(__uint_as_float(s & 0x0000F000u), __uint_as_float(s & 0x000F0000u));
    return r;
}
// One word of a unit for one row and vector: quads q0 = (lo0, hi0, lo1, hi1) and q1 = (lo2, hi2, lo3, hi3).
__device__ __forceinline__ float2 word_fma_pairs(const Word4p& d, float4 q0, float4 q1, float2 a) {
    a = ffma2(d.b0, make_float2(q0.x, q0.y), a);
    a = ffma2(d.b1, make_float2(q0.z, q0.w), a);
    a = ffma2(d.b2, make_float2(q1.x, q1.y), a);
    a = ffma2(d.b3, make_float2(q1.z, q1.w), a);
    return a;
}

__device__ __forceinline__ float byte_as_float_b(uint32_t w, int j) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + (uint32_t)j)) - 8388608.0f;
}

template <int V, int R, int W, int D>
__global__ void __launch_bounds__(W * 32, 1) q4k_batched_kernel(const Q4KBParams p) {
    constexpr int kThreads = W * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t U = (uint32_t)(p.K / 32);
    const int nsub = p.K / 32;

    const uint32_t s_base = smem_addr(smem);
    const uint32_t xs = s_base + p.xs_off;      // float[V][8 quads][U][4]
    const uint32_t ssum = s_base + p.ssum_off;  // float4[V][K/32] per unit: (S_lo, S_hi, f_lo, f_hi)
    const uint32_t ring = s_base + p.slots_off + (uint32_t)(warp * D * p.slot_bytes);

    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;
    const int Wtot = (int)gridDim.x * W;
    const uint64_t pol = policy_evict_first();
    const size_t row_bytes = (size_t)p.nsb * 144;

    int ijob = gw, ic = 0, islot = 0;
    auto issue = [&]() {
        if (ijob < p.jobs) {
            const int r0 = ijob * R;
            const int rv = min(R, p.N - r0);
            const int sb0 = ic * p.CS;
            const int cs = min(p.CS, p.nsb - sb0);
            const uint32_t slot = ring + (uint32_t)(islot * p.slot_bytes);
            const uint8_t* src = p.w + (size_t)r0 * row_bytes + (size_t)sb0 * 144;
            if (p.S == 1) {
                warp_copy_async(slot, src, (uint32_t)(rv * cs * 144), lane, pol);
            } else {
                for (int r = 0; r < rv; ++r)
                    warp_copy_async(slot + (uint32_t)(r * cs * 144), src + (size_t)r * row_bytes, (uint32_t)(cs * 144),
                                    lane, pol);
            }
            if (++ic == p.S) {
                ic = 0;
                ijob += Wtot;
            }
            islot = islot + 1 == D ? 0 : islot + 1;
        }
        cp_async_commit();
    };

#pragma unroll
    for (int k = 0; k < D - 1; ++k) issue();

    // The weights are constant; X and Y may belong to the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();

    // Stage the V vectors: four lanes per sub-block (whole warps: V*K/32*4 is a multiple of 32). Each thread issues
    // the loads of up to kBatch of its sub-block quarters before using any of them (one L2 round trip per batch).
    {
        const int t4 = lane & 3;
        const int nthr = V * nsub * 4;
        constexpr int kBatch = V <= 2 ? 2 : 8;  // two quarters per thread cover two vectors at 512 threads and K <= 4096
        for (int base = threadIdx.x; base < nthr; base += kThreads * kBatch) {
        float4 xa[kBatch], xb[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int thr = base + j * kThreads;
            const bool in = thr < nthr;
            const float4* src = reinterpret_cast<const float4*>(p.x) + (size_t)(in ? thr >> 2 : 0) * 8 + 2 * t4;
            xa[j] = in ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
            xb[j] = in ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // a thread's quarters all lie in sub-blocks of one parity (kThreads / 4 and nsub are even), so they share
        // the code half k
        const int k = (base >> 2) & 1;
        int ej[kBatch];
        stage_blocks4<kBatch>(xa, xb, k, ej);  // quarters past the end stage zeros and are not stored
        DivWalk vs(base >> 2, kThreads >> 2, nsub);  // (vector, sub-block) of quarter jb's sub-block
#pragma unroll
        for (int jb = 0; jb < kBatch; ++jb, vs.next()) {
            const int thr = base + jb * kThreads;
            if (thr >= nthr) break;  // warp-uniform
            const int v = vs.q;
            const int js = vs.r;
            const Stage4 st = {ej[jb], xa[jb], xb[jb]};
            const uint32_t u = (uint32_t)(js & ~1) + (uint32_t)(t4 >> 1);
            // this quarter holds words i0 and i0 + 1 of unit u in one code half (k); lane ^ 4 holds the same words
            // in the other half. The low-half lane writes word i0 and the high-half lane word i0 + 1, each as its
            // two interleaved quads
            const uint32_t i0 = (uint32_t)((2 * t4) & 3);
            const float4 send = k ? st.a : st.b;
            const float4 recv = make_float4(__shfl_xor_sync(0xffffffffu, send.x, 4), __shfl_xor_sync(0xffffffffu, send.y, 4),
                                            __shfl_xor_sync(0xffffffffu, send.z, 4), __shfl_xor_sync(0xffffffffu, send.w, 4));
            const float4 lo = k ? recv : st.a, hi = k ? st.b : recv;
            const uint32_t a0 = xs + xs_index((uint32_t)v, 2u * (i0 + (uint32_t)k), u, U) * 4u;
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "f"(lo.x), "f"(hi.x), "f"(lo.y),
                         "f"(hi.y)
                         : "memory");
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + U * 16u), "f"(lo.z), "f"(hi.z),
                         "f"(lo.w), "f"(hi.w)
                         : "memory");
            if (t4 == 0) {
                // f of sub-block js goes to both units of its chunk (.z for the low sub-block, .w for the high)
                const uint32_t ua = ssum + ((uint32_t)v * U + (uint32_t)(js & ~1)) * 16u + 8u + (uint32_t)k * 4u;
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(ua), "f"(block_factor(st.e)) : "memory");
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(ua + 16u), "f"(block_factor(st.e)) : "memory");
            }
        }
        }
        __syncthreads();
        // S of each unit's two halves: the unit chain on codes of 1, in the main loop's order (.x low, .y high)
        const Word4p c1 = decode_word_pairs(0x11111111u);
        DivWalk vu((int)threadIdx.x, kThreads, (int)U);
        for (int t = threadIdx.x; t < V * (int)U; t += kThreads, vu.next()) {
            const uint32_t v = (uint32_t)vu.q, u = (uint32_t)vu.r;
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                a = word_fma_pairs(c1, lds128f(xs + xs_index(v, (uint32_t)(2 * i), u, U) * 4u),
                                   lds128f(xs + xs_index(v, (uint32_t)(2 * i + 1), u, U) * 4u), a);
            const uint32_t ua = ssum + ((uint32_t)v * U + u) * 16u;
            const float2 f = lds64f(ua + 8u);
            asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(ua), "f"(a.x * f.x), "f"(a.y * f.y)
                         : "memory");
        }
    }
    __syncthreads();

    float2 tot[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) tot[r][v] = make_float2(0.f, 0.f);

    const uint32_t cpos = (uint32_t)(lane & 7);
    const uint32_t jj = cpos & 3u;
    const int gbase = lane & ~7;
    const uint32_t qstride = U * 16u;
    const uint32_t vstride = 8u * U * 16u;
    const int my_jobs = gw < p.jobs ? (p.jobs - 1 - gw) / Wtot + 1 : 0;
    const int total = my_jobs * p.S;
    int job = gw, c = 0, cslot = 0;
    for (int g = 0; g < total; ++g) {
        issue();
        cp_async_wait<D - 1>();
        __syncwarp();
        const uint32_t slot = ring + (uint32_t)(cslot * p.slot_bytes);
        const int r0 = job * R;
        const int rv = min(R, p.N - r0);
        const int sb0 = c * p.CS;
        const int cs = min(p.CS, p.nsb - sb0);
        const int nunits = 8 * cs;

        // Uniform trip count over the warp (lanes past the chunk use a clamped super-block and add nothing),
        // so every lane takes part in the shuffles.
#pragma unroll 1
        for (int ul0 = 0; ul0 < nunits; ul0 += 32) {
            const int ul = ul0 + lane;
            const bool valid = ul < nunits;
            const int sbl = valid ? (ul >> 3) : 0;
            const uint32_t u = (uint32_t)(8 * (sb0 + sbl)) + cpos;  // unit index = sub-block index of j = cpos
            uint4 w[R];
            float dlo[R], dhi[R], mlo[R], mhi[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t it = (uint32_t)(r * cs + sbl);
                const uint4 hdr = lds128(slot + it * 144u);
                const uint32_t scw = cpos < 4 ? (hdr.y & 0x3F3F3F3Fu)
                                              : ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u));
                const uint32_t mw = cpos < 4 ? (hdr.z & 0x3F3F3F3Fu)
                                             : (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u));
                const float dsc = f16_bits_to_f32(hdr.x) * byte_as_float_b(scw, (int)jj);
                const float dmm = -(f16_bits_to_f32(hdr.x >> 16) * byte_as_float_b(mw, (int)jj));
                dlo[r] = __shfl_sync(0xffffffffu, dsc, gbase + (int)(cpos & ~1u));
                dhi[r] = __shfl_sync(0xffffffffu, dsc, gbase + (int)(cpos | 1u));
                mlo[r] = __shfl_sync(0xffffffffu, dmm, gbase + (int)(cpos & ~1u));
                mhi[r] = __shfl_sync(0xffffffffu, dmm, gbase + (int)(cpos | 1u));
                w[r] = lds128(slot + it * 144u + 16u + cpos * 16u);
            }
            float2 acc[R][V];  // (low half, high half) of the unit
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                Word4p d4[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    d4[r] = decode_word_pairs(i == 0 ? w[r].x : i == 1 ? w[r].y : i == 2 ? w[r].z : w[r].w);
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const uint32_t xa = xs + (uint32_t)v * vstride + u * 16u;
                    const float4 q0 = lds128f(xa + (uint32_t)(2 * i) * qstride);
                    const float4 q1 = lds128f(xa + (uint32_t)(2 * i + 1) * qstride);
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        acc[r][v] = word_fma_pairs(d4[r], q0, q1, i == 0 ? make_float2(0.f, 0.f) : acc[r][v]);
                }
            }
            if (valid) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    // (S_lo, S_hi, f_lo, f_hi) of this unit for vector v
                    const float4 sf = lds128f(ssum + ((uint32_t)v * U + u) * 16u);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        // fl(d*sc*f * A) - fl(dmin*m * S) per half (d*sc*f and dmin*m are exact), with scalar
                        // rounded operations that the compiler never fuses into an FMA
                        const float ul = __fmul_rn(dlo[r] * sf.z, acc[r][v].x);
                        const float uh = __fmul_rn(dhi[r] * sf.w, acc[r][v].y);
                        tot[r][v].x = __fadd_rn(tot[r][v].x, __fadd_rn(ul, __fmul_rn(mlo[r], sf.x)));
                        tot[r][v].y = __fadd_rn(tot[r][v].y, __fadd_rn(uh, __fmul_rn(mhi[r], sf.y)));
                    }
                }
            }
        }
        __syncwarp();  // every lane is done with this slot before a later stage reuses it

        if (c == p.S - 1) {
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
                    vals[r * V + v] = tot[r][v].x + tot[r][v].y;
                    tot[r][v] = make_float2(0.f, 0.f);
                }
            warp_transpose_reduce<P2>(vals, lane);
            const int idx = lane >> (5 - L2);
            const bool leader = (lane & ((1 << (5 - L2)) - 1)) == 0;
            if (leader && idx < NV) {
                const int r = idx / V;
                const int v = idx - r * V;
                if (r < rv) p.y[(size_t)v * p.N + r0 + r] = vals[0];
            }
        }
        if (++c == p.S) {
            c = 0;
            job += Wtot;
        }
        cslot = cslot + 1 == D ? 0 : cslot + 1;
    }
}

inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Shared memory: [staged X V*K*4][(S_lo, S_hi, f_lo, f_hi) per unit V*K/32*16][W rings of D slots of R rows x CS super-blocks];
// whole rows first, then smaller chunks, then depth 2.
template <int V, int R, int W>
cudaError_t run_batched(const DeviceInfo& di, float* Y, const uint8_t* w, const float* X, int N, int K,
                        cudaStream_t s) {
    const int nsb = K / 256;
    Q4KBParams p;
    p.y = Y;
    p.w = w;
    p.x = X;
    p.N = N;
    p.K = K;
    p.nsb = nsb;
    const uint32_t xsb = (uint32_t)round_up(V * K * 4, 128);
    const uint32_t ssb = (uint32_t)round_up(V * (K / 32) * 16, 128);
    p.xs_off = 0;
    p.ssum_off = xsb;
    p.slots_off = xsb + ssb;
    for (int dd = 3; dd >= 2; --dd) {
        for (int cs0 = 16; cs0 >= 1; cs0 /= 2) {
            const int cs = std::min(cs0, nsb);
            const int slot = round_up(R * cs * 144, 128);
            const uint32_t smem = p.slots_off + (uint32_t)(W * dd * slot);
            if (smem > (uint32_t)di.max_smem_optin) continue;
            p.CS = cs;
            p.S = (nsb + cs - 1) / cs;
            p.jobs = (N + R - 1) / R;
            p.slot_bytes = slot;
            const int grid = std::min(di.sm_count, p.jobs);
            cudaError_t err = cudaSuccess;
            if (dd == 3) {
                auto kern = q4k_batched_kernel<V, R, W, 3>;
                static std::once_flag once3[64];
                std::call_once(once3[di.device & 63], [&] {
                    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
                });
                if (err != cudaSuccess) return err;
                return launch_kernel(kern, grid, W * 32, smem, s, p);
            }
            auto kern = q4k_batched_kernel<V, R, W, 2>;
            static std::once_flag once2[64];
            std::call_once(once2[di.device & 63], [&] {
                err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
            });
            if (err != cudaSuccess) return err;
            return launch_kernel(kern, grid, W * 32, smem, s, p);
        }
    }
    return cudaErrorNotSupported;
}

}  // namespace

// Variant per batch width: 16 warps x 2 rows for one or two vectors, 8 warps x 2 rows for three, 8 x 4 for four
// and 8 x 3 for five to eight (each staged quad serves more rows; four rows at eight vectors would spill).
cudaError_t launch_q4k_gemv_batched(float* Y, const uint8_t* w, const float* X, int V, int N, int K, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    switch (V) {
        case 1:
            // one input: the row-per-lane kernel of the fused calls, without normalisation
            e = launch_q4k_rows_gemv(Y, nullptr, w, nullptr, X, nullptr, 0.f, N, K, false, s);
            return e == cudaErrorNotSupported ? run_batched<1, 2, 16>(di, Y, w, X, N, K, s) : e;
        case 2: return run_batched<2, 2, 16>(di, Y, w, X, N, K, s);
        case 3: return run_batched<3, 2, 8>(di, Y, w, X, N, K, s);
        case 4: return run_batched<4, 4, 8>(di, Y, w, X, N, K, s);
        case 5: return run_batched<5, 3, 8>(di, Y, w, X, N, K, s);
        case 6: return run_batched<6, 3, 8>(di, Y, w, X, N, K, s);
        case 7: return run_batched<7, 3, 8>(di, Y, w, X, N, K, s);
        case 8: return run_batched<8, 3, 8>(di, Y, w, X, N, K, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace q4
