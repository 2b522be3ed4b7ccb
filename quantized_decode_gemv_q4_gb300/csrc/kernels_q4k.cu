// Q4_K decode GEMVs for sm_103a: fused RMSNorm + GEMV, fused gate+up (two weight streams against one
// staged input, RMSNorm optional), the pure-read ceiling instrument and the bit-exact dequant dump.
//
// Format (trueno-gpu `fused.rs`, FusedRmsNormQ4KGemvKernel phase 3): a row is K/256 super-blocks of 144
// bytes: f16 d, f16 dmin, 12 bytes of packed 6-bit scales/mins, 128 quant bytes. Weight e of a super-block
// lives in chunk c = e/64: low nibbles of the chunk's 32 bytes are sub-block 2c, high nibbles sub-block 2c+1;
// its value is d*sc_j*q - dmin*m_j for its sub-block j.
//
// Kernel shape (one CTA of W warps per SM, persistent), as the planar Q4 kernels:
//  * prologue: every warp issues its first weight copies, then the CTA computes sum(x^2) (block reduction),
//    r = rsqrt(sum/K + eps) and xhat = x * r * gamma, which it keeps in shared memory only (permuted and
//    pre-scaled per nibble position), together with the 32-element sub-block sums S_j of xhat;
//  * each warp streams R rows of each of NS weight matrices through its own ring of cp.async slots;
//  * per slot, the warp first decodes each super-block header once: d*sc_j into a small table, and the
//    whole min term dmin * sum_j m_j * S_j straight into its row accumulators;
//  * then lane l takes 16-byte quant unit l (+32, ...): chunk c = (l%8)/2, half h = l%2 of a super-block,
//    i.e. 16 codes of sub-block 2c and 16 of 2c+1, all against the same 32 staged inputs, and folds them
//    with d*sc_2c and d*sc_2c+1 from the table;
//  * row totals are summed over the warp and stored. The NS matrices share every staged-input load.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

struct Q4KParams {
    float* y0;
    float* y1;
    const uint8_t* w0;
    const uint8_t* w1;
    const float* x;
    const float* gamma;  // nullptr: no RMSNorm
    float eps;
    int N, K, nsb;
    int CS;          // super-blocks per chunk
    int S;           // chunks per row
    int jobs;        // row groups of R rows (per stream)
    int slot_bytes;  // multiple of 128
    int table_bytes; // per warp
    uint32_t xs_off, ssum_off, red_off, tables_off, slots_off;
};

template <int NS, int R, int W, int D, bool PURE>
__global__ void __launch_bounds__(W * 32, 1) q4k_gemv_kernel(const Q4KParams p) {
    constexpr int kThreads = W * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t U = (uint32_t)(p.K / 32);  // 16-byte quant units per row

    const uint32_t s_base = smem_addr(smem);
    const uint32_t xs = s_base + p.xs_off;
    const uint32_t ssum = s_base + p.ssum_off;
    const uint32_t red = s_base + p.red_off;
    const uint32_t table = s_base + p.tables_off + (uint32_t)(warp * p.table_bytes);
    const uint32_t slots = s_base + p.slots_off + (uint32_t)(warp * D * p.slot_bytes);

    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;
    const int Wtot = (int)gridDim.x * W;
    const int my_jobs = gw < p.jobs ? (p.jobs - 1 - gw) / Wtot + 1 : 0;
    const int total = my_jobs * p.S;
    const uint64_t pol = policy_evict_first();
    const size_t row_bytes = (size_t)p.nsb * 144;

    // Stage g of this warp -> slot g % D; one commit group per stage (empty when g >= total).
    auto issue = [&](int g) {
        if (g < total) {
            const int job = gw + (g / p.S) * Wtot;
            const int c = g % p.S;
            const int r0 = job * R;
            const int rv = min(R, p.N - r0);
            const int sb0 = c * p.CS;
            const int cs = min(p.CS, p.nsb - sb0);
            const uint32_t slot = slots + (uint32_t)((g % D) * p.slot_bytes);
#pragma unroll
            for (int s = 0; s < NS; ++s) {
                const uint8_t* src = (s == 0 ? p.w0 : p.w1) + (size_t)r0 * row_bytes + (size_t)sb0 * 144;
                const uint32_t dst = slot + (uint32_t)(s * R * cs * 144);
                if (p.S == 1) {
                    warp_copy_async(dst, src, (uint32_t)(rv * cs * 144), lane, pol);
                } else {
                    for (int r = 0; r < rv; ++r)
                        warp_copy_async(dst + (uint32_t)(r * cs * 144), src + (size_t)r * row_bytes,
                                        (uint32_t)(cs * 144), lane, pol);
                }
            }
        }
        cp_async_commit();
    };

    for (int g = 0; g < D - 1; ++g) issue(g);

    // The weights are constant; x, gamma and the outputs may belong to the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();

    if constexpr (!PURE) {
        const int K4 = p.K >> 2;
        float r = 1.0f;
        if (p.gamma) {
            // sum of squares over K: per-thread partials, warp shuffles, then one value per warp
            float ss = 0.f;
            for (int idx = threadIdx.x; idx < K4; idx += kThreads) {
                const float4 xv = __ldg(reinterpret_cast<const float4*>(p.x) + idx);
                ss = fmaf(xv.x, xv.x, ss);
                ss = fmaf(xv.y, xv.y, ss);
                ss = fmaf(xv.z, xv.z, ss);
                ss = fmaf(xv.w, xv.w, ss);
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) asm volatile("st.shared.f32 [%0], %1;" ::"r"(red + (uint32_t)warp * 4u), "f"(ss) : "memory");
            __syncthreads();
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) tot += lds32f(red + (uint32_t)w * 4u);
            r = rsqrtf(tot / (float)p.K + p.eps);
        }
        // xhat = (x * r) * gamma, staged permuted and pre-scaled; S_j = sum of xhat over sub-block j.
        // A warp covers 32 consecutive float4 = 4 whole sub-blocks, and K/4 is a multiple of 64, so every
        // lane of a warp takes the same number of trips and the 8-lane shuffles below are complete.
        for (int idx = threadIdx.x; idx < K4; idx += kThreads) {
            const uint32_t k = (uint32_t)idx * 4u;
            float4 xv = __ldg(reinterpret_cast<const float4*>(p.x) + idx);
            if (p.gamma) {
                const float4 gv = __ldg(reinterpret_cast<const float4*>(p.gamma) + idx);
                xv.x = (xv.x * r) * gv.x;
                xv.y = (xv.y * r) * gv.y;
                xv.z = (xv.z * r) * gv.z;
                xv.w = (xv.w * r) * gv.w;
            }
            float part = (xv.x + xv.y) + (xv.z + xv.w);
            part += __shfl_xor_sync(0xffffffffu, part, 4);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            if ((lane & 7) == 0)
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(ssum + (k >> 5) * 4u), "f"(part) : "memory");
            uint32_t u, q, jj;
            int hi;
            q4k_elem_place(k, u, q, jj, hi);
            const uint32_t a = xs + xs_index(0u, q, u, U) * 4u;
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(xv.x * pos_scale_dev(hi, 0)),
                         "f"(xv.y * pos_scale_dev(hi, 1)), "f"(xv.z * pos_scale_dev(hi, 2)),
                         "f"(xv.w * pos_scale_dev(hi, 3))
                         : "memory");
        }
    }
    __syncthreads();

    float2 tot[NS][R];
    float mins[NS][R];
    uint32_t fold[NS][R];
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            tot[s][r] = make_float2(0.f, 0.f);
            mins[s][r] = 0.f;
            fold[s][r] = 0u;
        }

    const uint32_t cpos = (uint32_t)(lane & 7);  // unit position inside a super-block: chunk cpos/2, half cpos%2

    for (int g = 0; g < total; ++g) {
        issue(g + D - 1);
        cp_async_wait<D - 1>();
        __syncwarp();
        const uint32_t slot = slots + (uint32_t)((g % D) * p.slot_bytes);

        const int job = gw + (g / p.S) * Wtot;
        const int c = g % p.S;
        const int r0 = job * R;
        const int rv = min(R, p.N - r0);
        const int sb0 = c * p.CS;
        const int cs = min(p.CS, p.nsb - sb0);

        // 1) headers: one lane per (stream, row, super-block)
        for (int t = lane; t < NS * R * cs; t += 32) {
            const int sr = t / cs;  // stream * R + row
            const int sbl = t - sr * cs;
            const uint4 hdr = lds128(slot + (uint32_t)((sr * cs + sbl) * 144));
            if constexpr (PURE) {
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        if (s * R + r == sr) fold[s][r] ^= hdr.x ^ hdr.y ^ hdr.z ^ hdr.w;
            } else {
                const float d = f16_bits_to_f32(hdr.x);
                const float dmin = f16_bits_to_f32(hdr.x >> 16);
                const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu;
                const uint32_t m_lo = hdr.z & 0x3F3F3F3Fu;
                const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
                const uint32_t m_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
                const uint32_t sg = (uint32_t)(sb0 + sbl) * 8u;  // first sub-block index in the row
                const float4 s0 = lds128f(ssum + sg * 4u);
                const float4 s1 = lds128f(ssum + sg * 4u + 16u);
                float dsc[8];
                float msum = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    dsc[j] = d * (float)((sc_lo >> (8 * j)) & 0xFFu);
                    dsc[j + 4] = d * (float)((sc_hi >> (8 * j)) & 0xFFu);
                }
                msum = fmaf((float)(m_lo & 0xFFu), s0.x, msum);
                msum = fmaf((float)((m_lo >> 8) & 0xFFu), s0.y, msum);
                msum = fmaf((float)((m_lo >> 16) & 0xFFu), s0.z, msum);
                msum = fmaf((float)(m_lo >> 24), s0.w, msum);
                msum = fmaf((float)(m_hi & 0xFFu), s1.x, msum);
                msum = fmaf((float)((m_hi >> 8) & 0xFFu), s1.y, msum);
                msum = fmaf((float)((m_hi >> 16) & 0xFFu), s1.z, msum);
                msum = fmaf((float)(m_hi >> 24), s1.w, msum);
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        if (s * R + r == sr) mins[s][r] = fmaf(dmin, msum, mins[s][r]);
                const uint32_t te = table + (uint32_t)((sr * cs + sbl) * 64);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(te + (uint32_t)cc * 16u),
                                 "f"(dsc[2 * cc]), "f"(dsc[2 * cc]), "f"(dsc[2 * cc + 1]), "f"(dsc[2 * cc + 1])
                                 : "memory");
            }
        }
        __syncwarp();

        // 2) quant units
        for (int ul = lane; ul < 8 * cs; ul += 32) {
            const int sbl = ul >> 3;
            const uint32_t u = (uint32_t)(8 * (sb0 + sbl)) + cpos;
            if constexpr (PURE) {
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint4 w = lds128(slot + (uint32_t)(((s * R + r) * cs + sbl) * 144 + 16) + cpos * 16u);
                        fold[s][r] ^= w.x ^ w.y ^ w.z ^ w.w;
                    }
            } else {
                float4 xl[4], xh[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xl[i] = lds128f(xs + xs_index(0u, (uint32_t)i, u, U) * 4u);
                    xh[i] = lds128f(xs + xs_index(0u, (uint32_t)(4 + i), u, U) * 4u);
                }
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t blk = (uint32_t)(((s * R + r) * cs + sbl) * 144);
                        const uint4 w = lds128(slot + blk + 16u + cpos * 16u);
                        float2 aL = make_float2(0.f, 0.f), aH = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t word = i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
                            const Word8 d8 = decode_word<0>(word);
                            aL = ffma2(d8.lo01, make_float2(xl[i].x, xl[i].y), aL);
                            aL = ffma2(d8.lo23, make_float2(xl[i].z, xl[i].w), aL);
                            aH = ffma2(d8.hi01, make_float2(xh[i].x, xh[i].y), aH);
                            aH = ffma2(d8.hi23, make_float2(xh[i].z, xh[i].w), aH);
                        }
                        const float4 tb =
                            lds128f(table + (uint32_t)(((s * R + r) * cs + sbl) * 64) + (cpos >> 1) * 16u);
                        tot[s][r] = ffma2(make_float2(tb.x, tb.y), aL, tot[s][r]);
                        tot[s][r] = ffma2(make_float2(tb.z, tb.w), aH, tot[s][r]);
                    }
            }
        }

        __syncwarp();  // every lane is done with this slot (and its table) before later stages reuse them

        if (c == p.S - 1) {
            if constexpr (PURE) {
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1)
                            fold[s][r] ^= __shfl_xor_sync(0xffffffffu, fold[s][r], off);
                        if (lane == 0 && r < rv) (s == 0 ? p.y0 : p.y1)[r0 + r] = __uint_as_float(fold[s][r]);
                        fold[s][r] = 0u;
                    }
            } else {
                constexpr int NV = NS * R;
                constexpr int P2 = NextPow2<NV>::value;
                constexpr int L2 = log2_const<P2>();
                float vals[P2];
#pragma unroll
                for (int i = 0; i < P2; ++i) vals[i] = 0.f;
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        vals[s * R + r] = (tot[s][r].x + tot[s][r].y) - mins[s][r];
                        tot[s][r] = make_float2(0.f, 0.f);
                        mins[s][r] = 0.f;
                    }
                warp_transpose_reduce<P2>(vals, lane);
                const int idx = lane >> (5 - L2);
                const bool leader = (lane & ((1 << (5 - L2)) - 1)) == 0;
                if (leader && idx < NV) {
                    const int s = idx / R;
                    const int r = idx - s * R;
                    if (r < rv) (s == 0 ? p.y0 : p.y1)[r0 + r] = vals[0];
                }
            }
        }
    }
}

// One thread per 16-byte quant unit: 32 weights, each d*sc*q - dmin*m rounded once to fp32.
__global__ void q4k_dequant_kernel(float* __restrict__ W, const uint8_t* __restrict__ w, long long nunits, int nsb) {
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nunits) return;
    const long long sbi = t >> 3;  // super-block (row-major over rows and super-blocks)
    const int cpos = (int)(t & 7);
    const int c = cpos >> 1, h = cpos & 1;
    const uint8_t* blk = w + sbi * 144;
    const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(blk));
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(blk + 16 + 16 * cpos));
    const uint8_t* s = reinterpret_cast<const uint8_t*>(&hdr) + 4;
    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
    float dsc[2], dm[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int j = 2 * c + k;
        int sc, m;
        if (j < 4) {
            sc = s[j] & 63;
            m = s[j + 4] & 63;
        } else {
            sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
        dsc[k] = __fmul_rn(d, (float)sc);
        dm[k] = __fmul_rn(dmin, (float)m);
    }
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
    // element index inside the super-block: low nibble of byte b -> 64c + 16h + b, high -> +32
    float* row = W + (sbi / nsb) * (long long)nsb * 256 + (sbi % nsb) * 256;
    float lo[16], hi[16];
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const uint32_t byte = (words[b >> 2] >> (8 * (b & 3))) & 0xFFu;
        lo[b] = __fsub_rn(__fmul_rn(dsc[0], (float)(byte & 15u)), dm[0]);
        hi[b] = __fsub_rn(__fmul_rn(dsc[1], (float)(byte >> 4)), dm[1]);
    }
    float4* dl = reinterpret_cast<float4*>(row + 64 * c + 16 * h);
    float4* dh = reinterpret_cast<float4*>(row + 64 * c + 32 + 16 * h);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        dl[i] = make_float4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
        dh[i] = make_float4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
    }
}

inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

void plan_override(int* cs, int* d) {
    static int o_cs = -1, o_d = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* e = getenv("Q4GEMV_Q4K_PLAN");
        if (e) sscanf(e, "%d,%d", &o_cs, &o_d);
    });
    if (o_cs > 0) *cs = o_cs;
    if (o_d > 0) *d = o_d;
}

struct Args {
    float *y0, *y1;
    const uint8_t *w0, *w1;
    const float *x, *gamma;
    float eps;
    int N, K;
};

template <int NS, int R, int W, int D, bool PURE>
cudaError_t launch_plan(const DeviceInfo& di, Q4KParams p, uint32_t smem, cudaStream_t s) {
    static std::once_flag attr_once[64];
    auto kern = q4k_gemv_kernel<NS, R, W, D, PURE>;
    cudaError_t err = cudaSuccess;
    std::call_once(attr_once[di.device & 63], [&] {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (err != cudaSuccess) return err;
    const int grid = std::min(di.sm_count, p.jobs);
    return launch_kernel(kern, grid, W * 32, smem, s, p);
}

// Shared memory: [staged xhat K*4][sub-block sums K/32*4][W reduction floats][W header tables]
//                [W rings of D slots]. Chunk (super-blocks per slot) and depth shrink until it fits.
template <int NS, int R, int W, bool PURE>
cudaError_t run(const DeviceInfo& di, const Args& a, int CS, int D, cudaStream_t s) {
    const int nsb = a.K / 256;
    plan_override(&CS, &D);
    D = std::max(2, std::min(4, D));
    Q4KParams p;
    bool ok = false;
    uint32_t smem = 0;
    int depth = D;
    for (int dd = D; dd >= 2 && !ok; --dd) {
        for (int cs0 = CS; cs0 >= 1 && !ok; cs0 /= 2) {
            const int cs = std::min(cs0, nsb);
            const int slot = round_up(NS * R * cs * 144, 128);
            const int tbytes = round_up(NS * R * cs * 64, 128);
            const uint32_t xs_bytes = PURE ? 0u : (uint32_t)(a.K * 4);
            const uint32_t ss_bytes = PURE ? 0u : (uint32_t)round_up(a.K / 32 * 4, 128);
            const uint32_t red_bytes = (uint32_t)round_up(W * 4, 128);
            p.xs_off = 0;
            p.ssum_off = xs_bytes;
            p.red_off = p.ssum_off + ss_bytes;
            p.tables_off = p.red_off + red_bytes;
            p.slots_off = p.tables_off + (uint32_t)(W * tbytes);
            smem = p.slots_off + (uint32_t)(W * dd * slot);
            if (smem <= (uint32_t)di.max_smem_optin) {
                ok = true;
                p.CS = cs;
                p.slot_bytes = slot;
                p.table_bytes = tbytes;
                depth = dd;
            }
        }
    }
    if (!ok) return cudaErrorNotSupported;
    p.y0 = a.y0;
    p.y1 = a.y1;
    p.w0 = a.w0;
    p.w1 = a.w1;
    p.x = a.x;
    p.gamma = a.gamma;
    p.eps = a.eps;
    p.N = a.N;
    p.K = a.K;
    p.nsb = nsb;
    p.S = (nsb + p.CS - 1) / p.CS;
    p.jobs = (a.N + R - 1) / R;
    switch (depth) {
        case 2: return launch_plan<NS, R, W, 2, PURE>(di, p, smem, s);
        case 3: return launch_plan<NS, R, W, 3, PURE>(di, p, smem, s);
        default: return launch_plan<NS, R, W, 4, PURE>(di, p, smem, s);
    }
}

}  // namespace

cudaError_t launch_q4k_gemv(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x,
                            const float* gamma, float eps, int N, int K, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    const Args a{y0, y1, w0, w1, x, gamma, eps, N, K};
    if (w1) return run<2, 1, 16, false>(di, a, 14, 2, s);
    return run<1, 2, 16, false>(di, a, 14, 2, s);
}

cudaError_t launch_q4k_pure_read(float* sink, const uint8_t* w, int N, int K, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    const Args a{sink, nullptr, w, nullptr, nullptr, nullptr, 0.f, N, K};
    return run<1, 2, 16, true>(di, a, 14, 2, s);
}

cudaError_t launch_q4k_dequant(float* W, const uint8_t* w, int N, int K, cudaStream_t s) {
    const int nsb = K / 256;
    const long long nunits = (long long)N * nsb * 8;
    const int threads = 256;
    const long long blocks = (nunits + threads - 1) / threads;
    q4k_dequant_kernel<<<(unsigned)blocks, threads, 0, s>>>(W, w, nunits, nsb);
    return cudaGetLastError();
}

}  // namespace q4
