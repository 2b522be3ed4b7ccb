// Expert-gathered MoE gate+up GEMV over planar Q4 expert stores, for sm_103a, plus its pure-read
// ceiling instrument.
//
// Problem (inferencelayer `kernel_lab.rs`, moe_lab / MOE_PURE_READ): experts are stacked in one store of
// E*N rows per projection; slot (t, s) of token t uses expert e = ids[t*topk+s] and writes rows
// (t*topk+s)*N + r of the gate and up outputs.
//
// Kernel shape (one persistent CTA of 8 warps per SM):
//  * prologue (every CTA, no host synchronisation): read the T*topk ids, find for each slot the first slot
//    with the same expert and its rank among the slots of that expert, number the distinct experts in
//    order of first appearance, and cut each expert's slot list into groups of at most MAXC slots; slots
//    with an id outside [0, E) get NaN outputs (written by CTA 0) and raise a status bit;
//  * jobs are (group, row group of R rows); a warp streams the R gate rows and R up rows of its job through
//    its own ring of cp.async slots, so each selected expert's bytes are read once per call (once per group
//    when more than MAXC slots route to one expert) and every routed token reuses them;
//  * all T input vectors are staged once per CTA (permuted, pre-scaled), and each decoded weight pair feeds
//    one packed FMA per routed slot.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {

static __device__ unsigned g_fault_moe;

namespace {

constexpr int kMaxSlots = 512;  // T * topk
constexpr int kMaxC = 4;        // routed slots served per weight sweep

struct MoEParams {
    float* yg;
    float* yu;
    const uint8_t* qg;
    const uint16_t* dg;
    const uint8_t* qu;
    const uint16_t* du;
    const float* x;
    const int32_t* ids;
    int32_t* status;
    int T, topk, E, N, K, nblk;
    int CB, S, slot_bytes, d_off, dcopy;
    uint32_t route_off, xs_off, slots_off;
    unsigned* fault;
};

// Routing tables in shared memory (route_off): slot_ids[kMaxSlots], rank[kMaxSlots], owner[kMaxSlots],
// ucount[kMaxSlots], uoffset[kMaxSlots+1], list[kMaxSlots], group_ux[kMaxSlots], group_first[kMaxSlots],
// group_cnt[kMaxSlots], scalars[4] (number of distinct experts, number of groups).
constexpr int kRouteInts = 9 * kMaxSlots + 8;

template <int R, int W, int D, bool PURE>
__global__ void __launch_bounds__(W * 32, 1) moe_q4_kernel(const MoEParams p) {
    constexpr int kThreads = W * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int TK = p.T * p.topk;
    const uint32_t U = (uint32_t)p.nblk;

    int* route = reinterpret_cast<int*>(smem + p.route_off);
    int* slot_ids = route;
    int* rank = route + kMaxSlots;
    int* owner = route + 2 * kMaxSlots;
    int* ucount = route + 3 * kMaxSlots;
    int* uoffset = route + 4 * kMaxSlots;  // kMaxSlots + 1 entries
    int* list = route + 5 * kMaxSlots + 1;
    int* group_ux = route + 6 * kMaxSlots + 1;
    int* group_first = route + 7 * kMaxSlots + 1;
    int* group_cnt = route + 8 * kMaxSlots + 1;
    int* scalars = route + 9 * kMaxSlots + 1;

    // ---- routing -------------------------------------------------------------------------------------
    for (int i = threadIdx.x; i < TK; i += kThreads) {
        slot_ids[i] = __ldg(p.ids + i);
        ucount[i] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < TK; i += kThreads) {
        const int e = slot_ids[i];
        int first = -1, rk = 0;
        if (e >= 0 && e < p.E) {
            for (int j = 0; j < i; ++j) {
                if (slot_ids[j] == e) {
                    if (first < 0) first = j;
                    ++rk;
                }
            }
            if (first < 0) first = i;
        }
        owner[i] = first;  // -1: invalid id
        rank[i] = rk;
    }
    __syncthreads();
    if (warp == 0) {
        // number the distinct experts (first slots) in slot order
        int base = 0;
        for (int c0 = 0; c0 < TK; c0 += 32) {
            const int i = c0 + lane;
            const bool first = i < TK && owner[i] == i;
            const unsigned m = __ballot_sync(0xffffffffu, first);
            if (first) list[i] = base + __popc(m & ((1u << lane) - 1u));  // temporary: ux of first slot i
            base += __popc(m);
        }
        if (lane == 0) scalars[0] = base;
    }
    __syncthreads();
    const int nux = scalars[0];
    for (int i = threadIdx.x; i < TK; i += kThreads) {
        const int f = owner[i];
        if (f >= 0) {
            const int ux = list[f];
            owner[i] = ux;  // from here on: distinct-expert index of slot i
            atomicAdd(&ucount[ux], 1);
        }
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive prefix sums of slot counts and of groups per distinct expert
        int base = 0, gbase = 0;
        for (int c0 = 0; c0 < nux; c0 += 32) {
            const int u = c0 + lane;
            const int cnt = u < nux ? ucount[u] : 0;
            const int ng = (cnt + kMaxC - 1) / kMaxC;
            int incl = cnt, gincl = ng;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, incl, off);
                const int b = __shfl_up_sync(0xffffffffu, gincl, off);
                if (lane >= off) {
                    incl += a;
                    gincl += b;
                }
            }
            if (u < nux) {
                uoffset[u] = base + incl - cnt;
                const int g0 = gbase + gincl - ng;
                for (int gi = 0; gi < ng; ++gi) {
                    group_ux[g0 + gi] = u;
                    group_first[g0 + gi] = uoffset[u] + gi * kMaxC;
                    group_cnt[g0 + gi] = min(kMaxC, cnt - gi * kMaxC);
                }
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
            gbase += __shfl_sync(0xffffffffu, gincl, 31);
        }
        if (lane == 0) scalars[1] = gbase;
    }
    __syncthreads();
    const int ngroups = scalars[1];
    for (int i = threadIdx.x; i < TK; i += kThreads) {
        const int ux = owner[i];
        if (ux >= 0) list[uoffset[ux] + rank[i]] = i;
    }
    __syncthreads();
    // group -> expert id
    for (int gi = threadIdx.x; gi < ngroups; gi += kThreads) {
        const int ux = group_ux[gi];
        group_cnt[gi] |= slot_ids[list[uoffset[ux]]] << 8;  // low 8 bits: count, high bits: expert id
    }
    // invalid slots: NaN outputs and a status bit (CTA 0 only)
    if (blockIdx.x == 0) {
        for (int i = 0; i < TK; ++i) {
            if (owner[i] >= 0) continue;
            for (int r = threadIdx.x; r < p.N; r += kThreads) {
                p.yg[(size_t)i * p.N + r] = __int_as_float(0x7fc00000);
                p.yu[(size_t)i * p.N + r] = __int_as_float(0x7fc00000);
            }
            if (threadIdx.x == 0) {
                if (p.status) atomicOr(reinterpret_cast<unsigned*>(p.status), (unsigned)kFaultBadExpert);
                atomicOr(p.fault, (unsigned)kFaultBadExpert);
            }
        }
    }
    __syncthreads();

    // ---- weight streaming -----------------------------------------------------------------------------
    const uint32_t s_base = smem_addr(smem);
    const uint32_t xs = s_base + p.xs_off;
    const uint32_t slots = s_base + p.slots_off + (uint32_t)(warp * D * p.slot_bytes);
    const int rgs = (p.N + R - 1) / R;
    const int jobs = ngroups * rgs;
    const int gw = warp * (int)gridDim.x + (int)blockIdx.x;
    const int Wtot = (int)gridDim.x * W;
    const int my_jobs = gw < jobs ? (jobs - 1 - gw) / Wtot + 1 : 0;
    const int total = my_jobs * p.S;
    const uint64_t pol = policy_evict_first();

    // Stage g of this warp -> slot g % D; one commit group per stage (empty when g >= total).
    auto issue = [&](int g) {
        if (g < total) {
            const int job = gw + (g / p.S) * Wtot;
            const int grp = job / rgs;
            const int r0 = (job - grp * rgs) * R;
            const int e = group_cnt[grp] >> 8;
            const int c = g % p.S;
            const int rv = min(R, p.N - r0);
            const int b0 = c * p.CB;
            const int nb = min(p.CB, p.nblk - b0);
            const uint32_t slot = slots + (uint32_t)((g % D) * p.slot_bytes);
            const size_t row0 = (size_t)e * p.N + r0;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const uint8_t* q = s == 0 ? p.qg : p.qu;
                const uint16_t* d = s == 0 ? p.dg : p.du;
                const uint32_t qdst = slot + (uint32_t)(s * R * nb * 16);
                const uint32_t ddst = slot + (uint32_t)(p.d_off + s * R * nb * 2);
                if (p.S == 1) {
                    warp_copy_async(qdst, q + row0 * p.nblk * 16, (uint32_t)(rv * nb * 16), lane, pol);
                    if (p.dcopy) warp_copy_async(ddst, d + row0 * p.nblk, (uint32_t)(rv * nb * 2), lane, pol);
                } else {
                    for (int r = 0; r < rv; ++r) {
                        const size_t rb = (row0 + r) * p.nblk + b0;
                        warp_copy_async(qdst + (uint32_t)(r * nb * 16), q + rb * 16, (uint32_t)(nb * 16), lane, pol);
                        if (p.dcopy)
                            warp_copy_async(ddst + (uint32_t)(r * nb * 2), d + rb, (uint32_t)(nb * 2), lane, pol);
                    }
                }
            }
        }
        cp_async_commit();
    };

    for (int g = 0; g < D - 1; ++g) issue(g);

    if constexpr (!PURE) {
        const int K4 = p.K >> 2;
        for (int idx = threadIdx.x; idx < p.T * K4; idx += kThreads) {
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

    float2 tot[2][R][kMaxC];
    uint32_t fold[2][R];
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            fold[s][r] = 0u;
#pragma unroll
            for (int m = 0; m < kMaxC; ++m) tot[s][r][m] = make_float2(0.f, 0.f);
        }

    for (int g = 0; g < total; ++g) {
        issue(g + D - 1);
        cp_async_wait<D - 1>();
        __syncwarp();
        const uint32_t slot = slots + (uint32_t)((g % D) * p.slot_bytes);

        const int job = gw + (g / p.S) * Wtot;
        const int grp = job / rgs;
        const int r0 = (job - grp * rgs) * R;
        const int gc = group_cnt[grp];
        const int cnt = gc & 0xFF;
        const int e = gc >> 8;
        const int first = group_first[grp];
        const int c = g % p.S;
        const int rv = min(R, p.N - r0);
        const int b0 = c * p.CB;
        const int nb = min(p.CB, p.nblk - b0);
        int tok[kMaxC];
#pragma unroll
        for (int m = 0; m < kMaxC; ++m) tok[m] = m < cnt ? list[first + m] / p.topk : 0;

        for (int ul = lane; ul < nb; ul += 32) {
            const uint32_t u = (uint32_t)(b0 + ul);
            uint4 w[2][R];
            float dsc[2][R];
            uint32_t dbits[2][R];
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    w[s][r] = lds128(slot + (uint32_t)(((s * R + r) * nb + ul) * 16));
                    if (p.dcopy) {
                        uint32_t bits;
                        asm volatile("ld.shared.u16 %0, [%1];"
                                     : "=r"(bits)
                                     : "r"(slot + (uint32_t)(p.d_off + ((s * R + r) * nb + ul) * 2)));
                        dbits[s][r] = bits;
                    } else {
                        const uint16_t* d = s == 0 ? p.dg : p.du;
                        dbits[s][r] = r < rv ? (uint32_t)__ldg(d + ((size_t)e * p.N + r0 + r) * p.nblk + u) : 0u;
                    }
                    dsc[s][r] = f16_bits_to_f32(dbits[s][r]);
                }
            if constexpr (PURE) {
#pragma unroll
                for (int s = 0; s < 2; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r) fold[s][r] ^= w[s][r].x ^ w[s][r].y ^ w[s][r].z ^ w[s][r].w ^ dbits[s][r];
            } else {
                float2 acc[2][R][kMaxC];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    Word8 d8[2][R];
#pragma unroll
                    for (int s = 0; s < 2; ++s)
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t wd = i == 0 ? w[s][r].x : i == 1 ? w[s][r].y : i == 2 ? w[s][r].z : w[s][r].w;
                            d8[s][r] = decode_word<8>(wd);
                        }
#pragma unroll
                    for (int m = 0; m < kMaxC; ++m) {
                        if (m < cnt) {
                            const float4 xl = lds128f(xs + xs_index((uint32_t)tok[m], (uint32_t)i, u, U) * 4u);
                            const float4 xh = lds128f(xs + xs_index((uint32_t)tok[m], (uint32_t)(4 + i), u, U) * 4u);
#pragma unroll
                            for (int s = 0; s < 2; ++s)
#pragma unroll
                                for (int r = 0; r < R; ++r) {
                                    float2 a = i == 0 ? make_float2(0.f, 0.f) : acc[s][r][m];
                                    a = ffma2(d8[s][r].lo01, make_float2(xl.x, xl.y), a);
                                    a = ffma2(d8[s][r].lo23, make_float2(xl.z, xl.w), a);
                                    a = ffma2(d8[s][r].hi01, make_float2(xh.x, xh.y), a);
                                    a = ffma2(d8[s][r].hi23, make_float2(xh.z, xh.w), a);
                                    acc[s][r][m] = a;
                                }
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < kMaxC; ++m)
                    if (m < cnt) {
#pragma unroll
                        for (int s = 0; s < 2; ++s)
#pragma unroll
                            for (int r = 0; r < R; ++r)
                                tot[s][r][m] = ffma2(make_float2(dsc[s][r], dsc[s][r]), acc[s][r][m], tot[s][r][m]);
                    }
            }
        }

        __syncwarp();  // every lane is done with this slot before a later stage overwrites it

        if (c == p.S - 1) {
            if constexpr (PURE) {
#pragma unroll
                for (int s = 0; s < 2; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1)
                            fold[s][r] ^= __shfl_xor_sync(0xffffffffu, fold[s][r], off);
                        if (lane < cnt && r < rv) {
                            const int slot_i = list[first + lane];
                            (s == 0 ? p.yg : p.yu)[(size_t)slot_i * p.N + r0 + r] = __uint_as_float(fold[s][r]);
                        }
                        fold[s][r] = 0u;
                    }
            } else {
                constexpr int NV = 2 * R * kMaxC;
                constexpr int P2 = NextPow2<NV>::value;
                constexpr int L2 = log2_const<P2>();
                float vals[P2];
#pragma unroll
                for (int i = 0; i < P2; ++i) vals[i] = 0.f;
#pragma unroll
                for (int s = 0; s < 2; ++s)
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int m = 0; m < kMaxC; ++m) {
                            vals[(s * R + r) * kMaxC + m] = tot[s][r][m].x + tot[s][r][m].y;
                            tot[s][r][m] = make_float2(0.f, 0.f);
                        }
                warp_transpose_reduce<P2>(vals, lane);
                const int idx = lane >> (5 - L2);
                const bool leader = (lane & ((1 << (5 - L2)) - 1)) == 0;
                if (leader && idx < NV) {
                    const int sr = idx / kMaxC;
                    const int m = idx - sr * kMaxC;
                    const int s = sr / R;
                    const int r = sr - s * R;
                    if (r < rv && m < cnt) {
                        const int slot_i = list[first + m];
                        (s == 0 ? p.yg : p.yu)[(size_t)slot_i * p.N + r0 + r] = vals[0];
                    }
                }
            }
        }
    }
}

inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

void plan_override(int* cb, int* d) {
    static int o_cb = -1, o_d = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* e = getenv("Q4GEMV_MOE_PLAN");
        if (e) sscanf(e, "%d,%d", &o_cb, &o_d);
    });
    if (o_cb > 0) *cb = o_cb;
    if (o_d > 0) *d = o_d;
}

unsigned* fault_word(int device) {
    static unsigned* ptrs[64] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[device & 63]) {
        unsigned* p = nullptr;
        if (cudaGetSymbolAddress((void**)&p, g_fault_moe) != cudaSuccess) return nullptr;
        ptrs[device & 63] = p;
    }
    return ptrs[device & 63];
}

template <int R, int W, int D, bool PURE>
cudaError_t launch_plan(const DeviceInfo& di, const MoEParams& p, uint32_t smem, cudaStream_t s) {
    static std::once_flag attr_once[64];
    auto kern = moe_q4_kernel<R, W, D, PURE>;
    cudaError_t err = cudaSuccess;
    std::call_once(attr_once[di.device & 63], [&] {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (err != cudaSuccess) return err;
    // worst case: every slot its own group
    const long long max_jobs = (long long)(p.T * p.topk) * ((p.N + R - 1) / R);
    const int grid = (int)std::min<long long>(di.sm_count, std::max<long long>(1, max_jobs));
    kern<<<grid, W * 32, smem, s>>>(p);
    return cudaGetLastError();
}

// Shared memory: [routing tables][staged inputs T*K*4][W rings of D slots]; chunk and depth shrink until
// it fits.
template <int R, int W, bool PURE>
cudaError_t run(const DeviceInfo& di, MoEParams p, int CB, int D, cudaStream_t s) {
    plan_override(&CB, &D);
    D = std::max(2, std::min(4, D));
    const bool dcopy = (p.nblk % 8 == 0) && ((reinterpret_cast<uintptr_t>(p.dg) & 15u) == 0) &&
                       ((reinterpret_cast<uintptr_t>(p.du) & 15u) == 0);
    bool ok = false;
    uint32_t smem = 0;
    int depth = D;
    for (int dd = D; dd >= 2 && !ok; --dd) {
        for (int cb0 = CB; cb0 >= 8 && !ok; cb0 /= 2) {
            const int cb = std::min(round_up(cb0, 8), round_up(p.nblk, 8));
            const int d_off = 2 * R * cb * 16;
            const int slot = round_up(d_off + round_up(2 * R * cb * 2, 16), 128);
            const uint32_t route = (uint32_t)round_up(kRouteInts * 4, 128);
            const uint32_t xs_bytes = PURE ? 0u : (uint32_t)(p.T * p.K * 4);
            p.route_off = 0;
            p.xs_off = route;
            p.slots_off = p.xs_off + xs_bytes;
            smem = p.slots_off + (uint32_t)(W * dd * slot);
            if (smem <= (uint32_t)di.max_smem_optin) {
                ok = true;
                p.CB = cb;
                p.d_off = d_off;
                p.slot_bytes = slot;
                depth = dd;
            }
        }
    }
    if (!ok) return cudaErrorNotSupported;
    p.dcopy = dcopy ? 1 : 0;
    p.S = (p.nblk + p.CB - 1) / p.CB;
    p.fault = fault_word(di.device);
    if (!p.fault) return cudaErrorInvalidSymbol;
    switch (depth) {
        case 2: return launch_plan<R, W, 2, PURE>(di, p, smem, s);
        case 3: return launch_plan<R, W, 3, PURE>(di, p, smem, s);
        default: return launch_plan<R, W, 4, PURE>(di, p, smem, s);
    }
}

}  // namespace

cudaError_t launch_moe_q4_gemv(float* y_gate, float* y_up, const uint8_t* qs_gate, const uint16_t* d_gate,
                               const uint8_t* qs_up, const uint16_t* d_up, const float* x, const int32_t* ids,
                               int T, int topk, int E, int N, int K, int32_t* dev_status, bool pure_read,
                               cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    MoEParams p{};
    p.yg = y_gate;
    p.yu = y_up;
    p.qg = qs_gate;
    p.dg = d_gate;
    p.qu = qs_up;
    p.du = d_up;
    p.x = x;
    p.ids = ids;
    p.status = dev_status;
    p.T = T;
    p.topk = topk;
    p.E = E;
    p.N = N;
    p.K = K;
    p.nblk = K / 32;
    if (pure_read) return run<2, 8, true>(di, p, 64, 2, s);
    return run<2, 8, false>(di, p, 64, 2, s);
}

cudaError_t read_and_clear_fault_moe(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_fault_moe, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_moe, &zero, sizeof(unsigned));
    return e;
}

}  // namespace q4
