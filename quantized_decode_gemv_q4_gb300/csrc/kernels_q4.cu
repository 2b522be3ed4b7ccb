// Planar Q4 decode GEMV for sm_103a: single vector, small batch (V <= 8 vectors sharing one sweep
// over the weights), the pure-read ceiling instrument and the bit-exact dequant dump.
//
// Format (inferencelayer `kernel_lab.rs`, shader GEMV_F16S): row n of the weight matrix is K/32 blocks;
// block b of row n has 16 packed bytes qs[n][b][0..15] and one f16 scale d[n][b]. Byte j holds weight j
// in its low nibble and weight j+16 in its high nibble; the weight is (q - 8) * d.
//
// Kernel shape (one CTA of 8 warps per SM, persistent):
//  * the input vectors are staged once per CTA in shared memory (permuted and pre-scaled, see
//    device_common.cuh), so no weight byte ever waits on a global load of x;
//  * every warp owns a ring of D shared-memory slots filled by warp-cooperative cp.async copies; a slot
//    holds R consecutive rows x CB blocks of quants plus their scales, so each weight byte is read from HBM
//    exactly once and all V vectors use it;
//  * lane l handles block unit l (+32, +64, ...) of every row in the slot: R rows share each staged-input
//    load; the 8 codes of a packed word become floats with one LOP3 each, one packed fp32x2 add removes
//    the bias exactly, and packed fp32x2 FMAs accumulate in fp32;
//  * each block's partial sum is scaled by its f16 scale; at the end of a row group the R*V totals are
//    summed across the warp with a transposing shuffle reduction and stored.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {


struct Q4Params {
    float* y;
    const uint8_t* qs;
    const uint16_t* d;
    const float* x;
    int N, K, nblk;
    int CB;          // blocks per chunk (multiple of 8)
    int S;           // chunks per row
    int jobs;        // row groups of R rows
    int slot_bytes;  // bytes per slot (multiple of 128)
    int d_off;       // offset of the scale region inside a slot
    int dcopy;       // scales travel in the slot (else read from global)
    uint32_t xs_off, slots_off;
};

template <int V, int R, int W, int D, bool PURE>
__global__ void __launch_bounds__(W * 32, 1) q4_gemv_kernel(const Q4Params p) {
    constexpr int kWarps = W;
    constexpr int kThreads = W * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t U = (uint32_t)p.nblk;

    const uint32_t s_base = smem_addr(smem);
    const uint32_t xs = s_base + p.xs_off;
    const uint32_t slots = s_base + p.slots_off + (uint32_t)(warp * D * p.slot_bytes);

    // Warps are numbered across CTAs first so that a small job count still spreads over all SMs.
    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;
    const int Wtot = (int)gridDim.x * kWarps;
    const int my_jobs = gw < p.jobs ? (p.jobs - 1 - gw) / Wtot + 1 : 0;
    const int total = my_jobs * p.S;
    const uint64_t pol = policy_evict_first();

    // Stage g of this warp -> slot g % D; one commit group per stage (empty when g >= total).
    auto issue = [&](int g) {
        if (g < total) {
            const int job = gw + (g / p.S) * Wtot;
            const int c = g % p.S;
            const int r0 = job * R;
            const int rv = min(R, p.N - r0);
            const int b0 = c * p.CB;
            const int nb = min(p.CB, p.nblk - b0);
            const uint32_t slot = slots + (uint32_t)((g % D) * p.slot_bytes);
            if (p.S == 1) {
                warp_copy_async(slot, p.qs + (size_t)r0 * p.nblk * 16, (uint32_t)(rv * nb * 16), lane, pol);
                if (p.dcopy)
                    warp_copy_async(slot + (uint32_t)p.d_off, p.d + (size_t)r0 * p.nblk, (uint32_t)(rv * nb * 2), lane,
                                    pol);
            } else {
                for (int r = 0; r < rv; ++r) {
                    const size_t row_blk = (size_t)(r0 + r) * p.nblk + b0;
                    warp_copy_async(slot + (uint32_t)(r * nb * 16), p.qs + row_blk * 16, (uint32_t)(nb * 16), lane,
                                    pol);
                    if (p.dcopy)
                        warp_copy_async(slot + (uint32_t)(p.d_off + r * nb * 2), p.d + row_blk, (uint32_t)(nb * 2),
                                        lane, pol);
                }
            }
        }
        cp_async_commit();
    };

    for (int g = 0; g < D - 1; ++g) issue(g);

    if constexpr (!PURE) {
        // Stage the V input vectors: permuted into per-unit quads and pre-scaled by 2^(23-p).
        const int K4 = p.K >> 2;
        for (int idx = threadIdx.x; idx < V * K4; idx += kThreads) {
            const int v = idx / K4;
            const uint32_t k = (uint32_t)(idx - v * K4) * 4u;
            const float4 xv = __ldg(reinterpret_cast<const float4*>(p.x + (size_t)v * p.K + k));
            uint32_t u, q, jj;
            int hi;
            q4_elem_place(k, u, q, jj, hi);
            const uint32_t a = xs + xs_index((uint32_t)v, q, u, U) * 4u;
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(xv.x * pos_scale_dev(hi, 0)),
                         "f"(xv.y * pos_scale_dev(hi, 1)), "f"(xv.z * pos_scale_dev(hi, 2)),
                         "f"(xv.w * pos_scale_dev(hi, 3))
                         : "memory");
        }
    }
    __syncthreads();

    float2 tot[R][V];
    uint32_t fold[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        fold[r] = 0u;
#pragma unroll
        for (int v = 0; v < V; ++v) tot[r][v] = make_float2(0.f, 0.f);
    }

    for (int g = 0; g < total; ++g) {
        issue(g + D - 1);
        cp_async_wait<D - 1>();
        __syncwarp();
        const uint32_t slot = slots + (uint32_t)((g % D) * p.slot_bytes);

        const int job = gw + (g / p.S) * Wtot;
        const int c = g % p.S;
        const int r0 = job * R;
        const int rv = min(R, p.N - r0);
        const int b0 = c * p.CB;
        const int nb = min(p.CB, p.nblk - b0);

        for (int ul = lane; ul < nb; ul += 32) {
            const uint32_t u = (uint32_t)(b0 + ul);
            uint4 w[R];
            float dsc[R];
            uint32_t dbits[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                w[r] = lds128(slot + (uint32_t)((r * nb + ul) * 16));
                if (p.dcopy) {
                    const uint32_t a = slot + (uint32_t)(p.d_off + (r * nb + ul) * 2);
                    uint32_t bits;
                    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(bits) : "r"(a));
                    dbits[r] = bits;
                } else {
                    dbits[r] = r < rv ? (uint32_t)__ldg(p.d + (size_t)(r0 + r) * p.nblk + u) : 0u;
                }
                dsc[r] = f16_bits_to_f32(dbits[r]);
            }
            if constexpr (PURE) {
#pragma unroll
                for (int r = 0; r < R; ++r) fold[r] ^= w[r].x ^ w[r].y ^ w[r].z ^ w[r].w ^ dbits[r];
            } else {
                float2 acc[R][V];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    Word8 d8[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t word = i == 0 ? w[r].x : i == 1 ? w[r].y : i == 2 ? w[r].z : w[r].w;
                        d8[r] = decode_word<8>(word);
                    }
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const float4 xl = lds128f(xs + xs_index((uint32_t)v, (uint32_t)i, u, U) * 4u);
                        const float4 xh = lds128f(xs + xs_index((uint32_t)v, (uint32_t)(4 + i), u, U) * 4u);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            float2 a = i == 0 ? make_float2(0.f, 0.f) : acc[r][v];
                            a = ffma2(d8[r].lo01, make_float2(xl.x, xl.y), a);
                            a = ffma2(d8[r].lo23, make_float2(xl.z, xl.w), a);
                            a = ffma2(d8[r].hi01, make_float2(xh.x, xh.y), a);
                            a = ffma2(d8[r].hi23, make_float2(xh.z, xh.w), a);
                            acc[r][v] = a;
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int v = 0; v < V; ++v) tot[r][v] = ffma2(make_float2(dsc[r], dsc[r]), acc[r][v], tot[r][v]);
            }
        }

        __syncwarp();  // every lane is done with this slot before a later stage overwrites it

        if (c == p.S - 1) {
            if constexpr (PURE) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) fold[r] ^= __shfl_xor_sync(0xffffffffu, fold[r], off);
                    if (lane == 0 && r < rv) p.y[r0 + r] = __uint_as_float(fold[r]);
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
        }
    }
}

// One thread per 32-weight block; each weight is (q - 8) * d, exact in fp32.
__global__ void q4_dequant_kernel(float* __restrict__ W, const uint8_t* __restrict__ qs,
                                  const uint16_t* __restrict__ d, long long nunits) {
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nunits) return;
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(qs) + t);
    const float s = f16_bits_to_f32(__ldg(d + t));
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    float out[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t byte = (words[j >> 2] >> (8 * (j & 3))) & 0xFFu;
        out[j] = __fmul_rn((float)((int)(byte & 15u) - 8), s);
        out[j + 16] = __fmul_rn((float)((int)(byte >> 4) - 8), s);
    }
    float4* dst = reinterpret_cast<float4*>(W + t * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_float4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
}

struct Plan {
    int CB, D, slot_bytes, d_off, dcopy;
    uint32_t xs_off, slots_off, smem;
    int jobs, S, grid;
};

inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Developer override of the chunk size and ring depth (blocks per chunk, slots per warp), read once from
// Q4GEMV_Q4_PLAN="CB,D". Used for tuning sweeps; the defaults in launch_q4_gemv come from such sweeps.
void plan_override(int* cb, int* d) {
    static int o_cb = -1, o_d = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* e = getenv("Q4GEMV_Q4_PLAN");
        if (e) sscanf(e, "%d,%d", &o_cb, &o_d);
    });
    if (o_cb > 0) *cb = o_cb;
    if (o_d > 0) *d = o_d;
}

// Shared memory: [staged input V*K*4][W rings of D slots]. A slot holds R rows x cb blocks of quants
// (and their scales when those can travel by 16-byte copies).
bool make_plan(const DeviceInfo& di, int V, int R, int W, bool pure, int N, int K, bool dcopy, int CB, int D,
               Plan* pl) {
    const int nblk = K / 32;
    const uint32_t xs_bytes = pure ? 0u : (uint32_t)(V * K * 4);
    const int cb = std::min(round_up(CB, 8), round_up(nblk, 8));
    const int d_off = R * cb * 16;
    const int slot = round_up(d_off + round_up(R * cb * 2, 16), 128);
    const uint32_t smem = xs_bytes + (uint32_t)(W * D * slot);
    if (smem > (uint32_t)di.max_smem_optin) return false;
    pl->CB = cb;
    pl->D = D;
    pl->slot_bytes = slot;
    pl->d_off = d_off;
    pl->dcopy = dcopy ? 1 : 0;
    pl->xs_off = 0;
    pl->slots_off = xs_bytes;
    pl->smem = smem;
    pl->S = (nblk + cb - 1) / cb;
    pl->jobs = (N + R - 1) / R;
    pl->grid = std::min(di.sm_count, pl->jobs);
    return true;
}

template <int V, int R, int W, int D, bool PURE>
cudaError_t launch_plan(const DeviceInfo& di, const Plan& pl, float* y, const uint8_t* qs, const uint16_t* d,
                        const float* x, int N, int K, cudaStream_t s) {
    static std::once_flag attr_once[64];
    auto kern = q4_gemv_kernel<V, R, W, D, PURE>;
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
    p.nblk = K / 32;
    p.CB = pl.CB;
    p.S = pl.S;
    p.jobs = pl.jobs;
    p.slot_bytes = pl.slot_bytes;
    p.d_off = pl.d_off;
    p.dcopy = pl.dcopy;
    p.xs_off = pl.xs_off;
    p.slots_off = pl.slots_off;
    kern<<<pl.grid, W * 32, pl.smem, s>>>(p);
    return cudaGetLastError();
}

// Plan (largest chunk first, then the requested depth, shrinking until it fits) and launch.
template <int V, int R, int W, bool PURE>
cudaError_t run(const DeviceInfo& di, float* y, const uint8_t* qs, const uint16_t* d, const float* x, int N, int K,
                int CB, int D, cudaStream_t s) {
    const int nblk = K / 32;
    const bool dcopy = (nblk % 8 == 0) && ((reinterpret_cast<uintptr_t>(d) & 15u) == 0);
    plan_override(&CB, &D);
    D = std::max(2, std::min(4, D));
    Plan pl;
    bool ok = false;
    for (int dd = D; dd >= 2 && !ok; --dd)
        for (int cb = CB; cb >= 8 && !ok; cb /= 2) ok = make_plan(di, V, R, W, PURE, N, K, dcopy, cb, dd, &pl);
    if (!ok) return cudaErrorNotSupported;
    switch (pl.D) {
        case 2: return launch_plan<V, R, W, 2, PURE>(di, pl, y, qs, d, x, N, K, s);
        case 3: return launch_plan<V, R, W, 3, PURE>(di, pl, y, qs, d, x, N, K, s);
        default: return launch_plan<V, R, W, 4, PURE>(di, pl, y, qs, d, x, N, K, s);
    }
}

}  // namespace

// Variant per batch width: V <= 2 runs 16 warps x 2 rows (registers fit in 128 per thread); wider batches
// run 8 warps (more accumulators per thread).
cudaError_t launch_q4_gemv(float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V, int N, int K,
                           cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    switch (V) {
        case 1: return run<1, 2, 16, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        case 2: return run<2, 2, 16, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        case 3: return run<3, 4, 8, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        case 4: return run<4, 4, 8, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        case 5: return run<5, 2, 8, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        case 6: return run<6, 2, 8, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        case 7: return run<7, 2, 8, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        case 8: return run<8, 2, 8, false>(di, Y, qs, d, X, N, K, 128, 2, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_q4_pure_read(float* sink, const uint8_t* qs, const uint16_t* d, int N, int K, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    return run<1, 2, 16, true>(di, sink, qs, d, nullptr, N, K, 128, 2, s);
}

cudaError_t launch_q4_dequant(float* W, const uint8_t* qs, const uint16_t* d, int N, int K, cudaStream_t s) {
    const long long nunits = (long long)N * (K / 32);
    const int threads = 256;
    const long long blocks = (nunits + threads - 1) / threads;
    q4_dequant_kernel<<<(unsigned)blocks, threads, 0, s>>>(W, qs, d, nunits);
    return cudaGetLastError();
}

}  // namespace q4
