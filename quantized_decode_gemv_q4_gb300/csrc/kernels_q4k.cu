// Q4_K decode GEMVs for sm_103a: fused RMSNorm + GEMV, fused gate+up (two weight streams against one
// staged input, RMSNorm optional), the pure-read ceiling instrument and the bit-exact dequant dump.
//
// Format (trueno-gpu `fused.rs`, FusedRmsNormQ4KGemvKernel phase 3): a row is K/256 super-blocks of 144
// bytes: f16 d, f16 dmin, 12 bytes of packed 6-bit scales/mins, 128 quant bytes. Weight e of a super-block
// lives in chunk c = e/64: low nibbles of the chunk's 32 bytes are sub-block 2c, high nibbles sub-block 2c+1;
// its value is d*sc_j*q - dmin*m_j for its sub-block j.
//
// Kernel shape (one persistent CTA of W warps per SM):
//  * prologue: every warp issues its first weight copies; after the previous kernel in the stream is done
//    the CTA computes sum(x^2) (block reduction), r = rsqrt(sum/K + eps) and xhat = x * r * gamma, which it
//    keeps in shared memory only: each 32-element sub-block j is staged pre-scaled with its own exponent
//    bound e_j (the bias-free decode of device_common.cuh), next to (S_j = sum of xhat over j, 2^(22+e_j));
//  * each warp streams R rows of each of NS weight matrices (whole rows when they fit) through its own ring
//    of cp.async slots, with incremental per-stage control;
//  * lane l takes 16-byte quant unit l (+32, ...): chunk c = (l%8)/2, half h = l%2 of a super-block, i.e.
//    16 codes of sub-block 2c and 16 of 2c+1 against the same 32 staged inputs: one shift and eight ANDs per
//    word, packed fp32x2 FMAs into one accumulator per sub-block. The 8 lanes of a super-block each decode
//    one sub-block's header entry (j = l%8): d*sc_j*2^(22+e_j), shared with the group by two shuffles, and
//    the min term dmin*m_j*S_j, added to the lane's own accumulator (the warp reduction sums them);
//  * row totals are summed over the warp and stored. The NS matrices share every staged-input load.
// Inputs whose staged value reaches 2^83 in magnitude are outside the supported range (non-finite result).
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

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
    int swiglu;          // two streams only: y0 = silu(gate) * up, y1 unused
    int N, K, nsb;
    int CS;           // super-blocks per chunk
    int S;            // chunks per row
    int jobs;         // row groups of R rows (per stream)
    int slot_bytes;   // multiple of 128
    uint32_t xs_off, ssum_off, red_off, slots_off;
};

// byte j of w as an exact float (0x4B000000 | b is 2^23 + b)
__device__ __forceinline__ float byte_as_float(uint32_t w, int j) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + (uint32_t)j)) - 8388608.0f;
}

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
    const uint32_t ring = s_base + p.slots_off + (uint32_t)(warp * D * p.slot_bytes);

    // Warps are numbered across CTAs first so that a small job count still spreads over all SMs.
    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;
    const int Wtot = (int)gridDim.x * W;
    const uint64_t pol = policy_evict_first();
    const size_t row_bytes = (size_t)p.nsb * 144;

    // Issue pointer (job, chunk, slot); one commit group per call, empty once this warp has nothing left.
    int ijob = gw, ic = 0, islot = 0;
    auto issue = [&]() {
        if (ijob < p.jobs) {
            const int r0 = ijob * R;
            const int rv = min(R, p.N - r0);
            const int sb0 = ic * p.CS;
            const int cs = min(p.CS, p.nsb - sb0);
            const uint32_t slot = ring + (uint32_t)(islot * p.slot_bytes);
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

    // The weights are constant; x, gamma and the outputs may belong to the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();

    if constexpr (!PURE) {
        const int K4 = p.K >> 2;
        float r = 1.0f;
        if (p.gamma) {
            // sum of squares over K: per-thread partials (loads issued ahead), warp shuffles, one value per warp
            float ss = 0.f;
            for (int base = threadIdx.x; base < K4; base += kThreads * kStageU) {
                float4 xv[kStageU];
#pragma unroll
                for (int j = 0; j < kStageU; ++j) {
                    const int idx = base + j * kThreads;
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
            if (lane == 0) asm volatile("st.shared.f32 [%0], %1;" ::"r"(red + (uint32_t)warp * 4u), "f"(ss) : "memory");
            __syncthreads();
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) tot += lds32f(red + (uint32_t)w * 4u);
            r = rsqrtf(tot / (float)p.K + p.eps);
        }
        // xhat = (x * r) * gamma, four lanes per 32-element sub-block (lane t of the group holds float4 2t,
        // 2t+1): the group's sum S_j and largest magnitude, then the block staged pre-scaled with its exponent
        // bound e_j. Sub-block j = 8*sb + 2c + k holds the low (k = 0) or high (k = 1) codes of units
        // 8*sb + 2c + h, h = element/16; its float4 f lands in quad 4k + f%4 of unit 8*sb + 2c + f/4.
        // K/32 is a multiple of 8, so whole warps take part in every group shuffle.
        const int nsub = p.K / 32;
        const int t4 = lane & 3;
        for (int thr = threadIdx.x; thr < nsub * 4; thr += kThreads) {
            const int js = thr >> 2;
            const float4* src = reinterpret_cast<const float4*>(p.x) + js * 8 + 2 * t4;
            float4 xa = __ldg(src), xb = __ldg(src + 1);
            if (p.gamma) {
                const float4* gsrc = reinterpret_cast<const float4*>(p.gamma) + js * 8 + 2 * t4;
                const float4 ga = __ldg(gsrc), gb = __ldg(gsrc + 1);
                xa = make_float4((xa.x * r) * ga.x, (xa.y * r) * ga.y, (xa.z * r) * ga.z, (xa.w * r) * ga.w);
                xb = make_float4((xb.x * r) * gb.x, (xb.y * r) * gb.y, (xb.z * r) * gb.z, (xb.w * r) * gb.w);
            }
            const int k = js & 1;
            const Stage4 st = stage_block4(xa, xb, k);
            const uint32_t ubase = (uint32_t)(js & ~1);  // 8*sb + 2c
            const int f0 = 2 * t4;                        // float4 index of xa inside the sub-block
            const uint32_t u = ubase + (uint32_t)(f0 >> 2);
            const uint32_t q0 = (uint32_t)(4 * k + (f0 & 3));
            const uint32_t a0 = xs + xs_index(0u, q0, u, U) * 4u;
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "f"(st.a.x), "f"(st.a.y), "f"(st.a.z),
                         "f"(st.a.w)
                         : "memory");
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + U * 16u), "f"(st.b.x), "f"(st.b.y),
                         "f"(st.b.z), "f"(st.b.w)
                         : "memory");
            if (t4 == 0)
                asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(ssum + (uint32_t)js * 8u), "f"(st.sum),
                             "f"(block_factor(st.e))
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
    const int my_jobs = gw < p.jobs ? (p.jobs - 1 - gw) / Wtot + 1 : 0;
    const int total = my_jobs * p.S;
    int job = gw, c = 0, cslot = 0;
    for (int g = 0; g < total; ++g) {
        issue();                 // stage g + D - 1 into the slot consumed at g - 1
        cp_async_wait<D - 1>();  // stage g has landed
        __syncwarp();
        const uint32_t slot = ring + (uint32_t)(cslot * p.slot_bytes);
        const int r0 = job * R;
        const int rv = min(R, p.N - r0);
        const int sb0 = c * p.CS;
        const int cs = min(p.CS, p.nsb - sb0);

        // Quant units: lane l takes unit l (+32, ...) of the chunk, i.e. super-block ul/8 at position
        // cpos = ul%8 (chunk cpos/2, half cpos%2). The trip count is uniform over the warp (lanes past the
        // chunk work on a clamped super-block and add nothing), so every lane takes part in the shuffles.
        // Each lane decodes the header entry of sub-block j = cpos of its super-block: d*sc_j*2^(22+e_j)
        // (exchanged within the 8-lane group: a unit needs sub-blocks 2c and 2c+1) and its own min term
        // dmin*m_j*S_j, which it adds to its row accumulator; the warp reduction sums all eight.
        const int nunits = 8 * cs;
        const int gbase = lane & ~7;
#pragma unroll 1
        for (int ul0 = 0; ul0 < nunits; ul0 += 32) {
            const int ul = ul0 + lane;
            const bool valid = ul < nunits;
            const int sbl = valid ? (ul >> 3) : 0;
            const uint32_t u = (uint32_t)(8 * (sb0 + sbl)) + cpos;
            if constexpr (PURE) {
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int rr = 0; rr < R; ++rr) {
                        const int it = (s * R + rr) * cs + sbl;
                        const uint4 w = lds128(slot + (uint32_t)(it * 144 + 16) + cpos * 16u);
                        uint32_t f = w.x ^ w.y ^ w.z ^ w.w;
                        if (cpos == 0) {
                            const uint4 hdr = lds128(slot + (uint32_t)(it * 144));
                            f ^= hdr.x ^ hdr.y ^ hdr.z ^ hdr.w;
                        }
                        if (valid) fold[s][rr] ^= f;
                    }
            } else {
                const float2 sf = lds64f(ssum + u * 8u);  // (S_j, 2^(22+e_j)) of sub-block j = cpos of this super-block
                const uint32_t xa = xs + u * 16u;
                const uint32_t qstride = U * 16u;
                float4 xl[4], xh[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xl[i] = lds128f(xa + (uint32_t)i * qstride);
                    xh[i] = lds128f(xa + (uint32_t)(4 + i) * qstride);
                }
                const uint32_t jj = cpos & 3u;
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int rr = 0; rr < R; ++rr) {
                        const int it = (s * R + rr) * cs + sbl;
                        const uint4 hdr = lds128(slot + (uint32_t)(it * 144));
                        // 6-bit scale and min of sub-block j = cpos
                        const uint32_t scw = cpos < 4 ? (hdr.y & 0x3F3F3F3Fu)
                                                      : ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u));
                        const uint32_t mw = cpos < 4 ? (hdr.z & 0x3F3F3F3Fu)
                                                     : (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u));
                        const float d = f16_bits_to_f32(hdr.x);
                        const float dmin = f16_bits_to_f32(hdr.x >> 16);
                        const float dsc = (d * byte_as_float(scw, (int)jj)) * sf.y;
                        const float mterm = (dmin * byte_as_float(mw, (int)jj)) * sf.x;
                        const float dlo = __shfl_sync(0xffffffffu, dsc, gbase + (int)(cpos & ~1u));
                        const float dhi = __shfl_sync(0xffffffffu, dsc, gbase + (int)(cpos | 1u));
                        const uint4 w = lds128(slot + (uint32_t)(it * 144 + 16) + cpos * 16u);
                        float2 aL = make_float2(0.f, 0.f), aH = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const Word8s d8 = decode_word_sub(i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w);
                            aL = ffma2(d8.lo01, make_float2(xl[i].x, xl[i].y), aL);
                            aL = ffma2(d8.lo23, make_float2(xl[i].z, xl[i].w), aL);
                            aH = ffma2(d8.hi01, make_float2(xh[i].x, xh[i].y), aH);
                            aH = ffma2(d8.hi23, make_float2(xh[i].z, xh[i].w), aH);
                        }
                        if (valid) {
                            tot[s][rr] = ffma2(make_float2(dlo, dlo), aL, tot[s][rr]);
                            tot[s][rr] = ffma2(make_float2(dhi, dhi), aH, tot[s][rr]);
                            mins[s][rr] += mterm;
                        }
                    }
            }
        }

        __syncwarp();  // every lane is done with this slot before a later stage reuses it

        if (c == p.S - 1) {
            if constexpr (PURE) {
#pragma unroll
                for (int s = 0; s < NS; ++s)
#pragma unroll
                    for (int rr = 0; rr < R; ++rr) {
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1)
                            fold[s][rr] ^= __shfl_xor_sync(0xffffffffu, fold[s][rr], off);
                        if (lane == 0 && rr < rv) (s == 0 ? p.y0 : p.y1)[r0 + rr] = __uint_as_float(fold[s][rr]);
                        fold[s][rr] = 0u;
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
                    for (int rr = 0; rr < R; ++rr) {
                        vals[s * R + rr] = (tot[s][rr].x + tot[s][rr].y) - mins[s][rr];
                        tot[s][rr] = make_float2(0.f, 0.f);
                        mins[s][rr] = 0.f;
                    }
                warp_transpose_reduce<P2>(vals, lane);
                const int idx = lane >> (5 - L2);
                const bool leader = (lane & ((1 << (5 - L2)) - 1)) == 0;
                if (NS == 2 && p.swiglu) {
                    // row rr's up total sits R lane groups after its gate total
                    const float up = __shfl_down_sync(0xffffffffu, vals[0], R << (5 - L2));
                    if (leader && idx < R && idx < rv) p.y0[r0 + idx] = silu(vals[0]) * up;
                } else if (leader && idx < NV) {
                    const int s = idx / R;
                    const int rr = idx - s * R;
                    if (rr < rv) (s == 0 ? p.y0 : p.y1)[r0 + rr] = vals[0];
                }
            }
        }
        if (++c == p.S) {
            c = 0;
            job += Wtot;
        }
        cslot = cslot + 1 == D ? 0 : cslot + 1;
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

// Developer override of the launch plan, read once from Q4GEMV_Q4K_PLAN="CS,depth,variant" (super-blocks
// per chunk, ring depth; variant 2: gate+up as 2 rows x 8 warps instead of 1 row x 16 warps). Used for
// tuning sweeps; the defaults come from such sweeps.
void plan_override(int* cs, int* d, int* variant) {
    static int o_cs = -1, o_d = -1, o_v = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* e = getenv("Q4GEMV_Q4K_PLAN");
        if (e) sscanf(e, "%d,%d,%d", &o_cs, &o_d, &o_v);
    });
    if (o_cs > 0) *cs = o_cs;
    if (o_d > 0) *d = o_d;
    if (o_v > 0) *variant = o_v;
}

struct Args {
    float *y0, *y1;
    const uint8_t *w0, *w1;
    const float *x, *gamma;
    float eps;
    int N, K;
    bool swiglu;
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

// Shared memory: [staged xhat K*4][(S_j, 2^(22+e_j)) per sub-block K/32*8][W reduction floats]
//                [W rings of D slots]. Chunk (super-blocks per slot) and depth shrink until it fits.
template <int NS, int R, int W, bool PURE>
cudaError_t run(const DeviceInfo& di, const Args& a, int CS, int D, cudaStream_t s) {
    const int nsb = a.K / 256;
    D = std::max(2, std::min(4, D));
    Q4KParams p;
    bool ok = false;
    uint32_t smem = 0;
    int depth = D;
    for (int dd = D; dd >= 2 && !ok; --dd) {
        for (int cs0 = CS; cs0 >= 1 && !ok; cs0 /= 2) {
            const int cs = std::min(cs0, nsb);
            const int slot = round_up(NS * R * cs * 144, 128);
            const uint32_t xs_bytes = PURE ? 0u : (uint32_t)(a.K * 4);
            const uint32_t ss_bytes = PURE ? 0u : (uint32_t)round_up(a.K / 32 * 8, 128);
            const uint32_t red_bytes = (uint32_t)round_up(W * 4, 128);
            p.xs_off = 0;
            p.ssum_off = xs_bytes;
            p.red_off = p.ssum_off + ss_bytes;
            p.slots_off = p.red_off + red_bytes;
            smem = p.slots_off + (uint32_t)(W * dd * slot);
            if (smem <= (uint32_t)di.max_smem_optin) {
                ok = true;
                p.CS = cs;
                p.slot_bytes = slot;
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
    p.swiglu = a.swiglu ? 1 : 0;
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

// Developer switch to the warp-per-row-group kernels above, read once from Q4GEMV_Q4K_IMPL=warp; the
// row-per-lane kernels are the default.
bool use_warp_impl() {
    static bool w = false;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* e = getenv("Q4GEMV_Q4K_IMPL");
        w = e && std::string(e) == "warp";
    });
    return w;
}

cudaError_t launch_q4k_gemv(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x,
                            const float* gamma, float eps, int N, int K, bool swiglu, cudaStream_t s) {
    if (!use_warp_impl()) return launch_q4k_rows_gemv(y0, y1, w0, w1, x, gamma, eps, N, K, swiglu, s);
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    const Args a{y0, y1, w0, w1, x, gamma, eps, N, K, swiglu && w1 != nullptr};
    int cs = 16, depth = 2, variant = 1;
    plan_override(&cs, &depth, &variant);
    if (w1) {
        if (variant == 2) return run<2, 2, 8, false>(di, a, cs, depth, s);
        if (variant == 3) return run<2, 1, 24, false>(di, a, cs, depth, s);
        return run<2, 1, 16, false>(di, a, cs, depth, s);
    }
    if (variant == 2) return run<1, 4, 8, false>(di, a, cs, depth, s);
    return run<1, 2, 16, false>(di, a, cs, depth, s);
}

cudaError_t launch_q4k_pure_read(float* sink, const uint8_t* w, int N, int K, cudaStream_t s) {
    if (!use_warp_impl()) return launch_q4k_rows_pure_read(sink, w, N, K, s);
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    const Args a{sink, nullptr, w, nullptr, nullptr, nullptr, 0.f, N, K, false};
    int cs = 16, depth = 2, variant = 1;
    plan_override(&cs, &depth, &variant);
    return run<1, 2, 16, true>(di, a, cs, depth, s);
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
