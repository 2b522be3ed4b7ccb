// Expert-gathered MoE gate+up GEMV over planar Q4 expert stores, for sm_103a, plus its pure-read
// ceiling instrument.
//
// Problem (inferencelayer `kernel_lab.rs`, moe_lab / MOE_PURE_READ): experts are stacked in one store of
// E*N rows per projection; slot (t, s) of token t uses expert e = ids[t*topk+s] and writes rows
// (t*topk+s)*N + r of the gate and up outputs.
//
// Kernel shape (one persistent CTA of W warps per SM):
//  * prologue (every CTA, no host synchronisation): read the T*topk ids, find for each slot the first slot
//    with the same expert and its rank among the slots of that expert, number the distinct experts in
//    order of first appearance, and cut each expert's slot list into groups of at most kMaxC slots; slots
//    with an id outside [0, E) get NaN outputs (written by CTA 0) and raise a status bit. Up to 64 slots, warp
//    0 does this alone from a 64-bit slot mask per expert (one shared-memory atomic OR per slot) while the
//    other warps stage the inputs; more slots take a table path run by all threads;
//  * jobs are (group, projection, row group of R rows), numbered group-major with the groups in order of slot
//    count; each warp owns one contiguous range of jobs of equal estimated cost, found in closed form from
//    the number of groups per slot count (or jobs dealt round-robin), so it streams whole-row stages of
//    consecutive rows through
//    its own ring of slots (bulk copies on a slot mbarrier, or cp.async for chunked rows) with incremental
//    control, and each selected expert's bytes are read once per call (once per group when more than kMaxC
//    slots route to one expert);
//  * all T input vectors are staged once per CTA, block by block, with the bias-free decode's per-block
//    scaling (device_common.cuh): float4[K/32 blocks / 32][T][8 quads][32 + 1 pad] and (2^(22+e), -8 offset term)
//    pairs float2[K/32 / 32][T][32] (the offset term is the unit chain on codes of 8, q4_block_bias, so zero
//    weights contribute exactly zero), and a lane's quads of a token sit at constant offsets from one base;
//  * a job's slot count C (1..kMaxC) selects a compiled variant of the stage body, so each decoded code
//    pair feeds exactly C packed FMAs in the common chain order (word_fma); per block t = A * 2^(22+e) + bias,
//    and the row accumulates d * t per routed slot;
//  * at the end of a row group the R*C totals are summed across the warp with a transposing shuffle
//    reduction and stored to each slot's output rows;
//  * a stage wait (bulk mode) that runs out of its limit makes the warp stop issuing copies and store its
//    remaining rows as NaN (kFaultWaitTimeout); before exiting it waits, bounded, for the copies it issued.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

constexpr int kMaxC = 4;        // routed slots served per weight sweep
// Grouped staging: a quad row holds the 32 blocks of a group and one 16-byte pad, so the four lanes that stage a
// block (quads 2t and 2t+1, rows 2t apart) store into distinct bank groups.
constexpr int kXGRow = 33;      // float4 per quad row

struct MoEParams {
    float* yg;
    float* yu;  // nullptr in the SwiGLU form (one output)
    const uint8_t* qg;
    const uint16_t* dg;
    const uint8_t* qu;
    const uint16_t* du;
    const float* x;
    const int32_t* ids;
    int32_t* status;
    int T, topk, E, N, K, nblk;
    int S, dcopy;
    int ms;    // routing table stride: T*topk rounded up to 32
    int deal;  // 1: jobs dealt round-robin over the warps; 0: contiguous cost-balanced ranges
    int cost_a, cost_b;
    int bulk;  // every stage is whole rows: bulk copies of quants and scales on a slot mbarrier
    uint32_t route_off, xs_off, aux_off, bar_off, slots_off;
    unsigned* fault;
    long long wait_cycles;  // limit of one stage wait
};

// Routing tables in shared memory (route_off), each of ms = T*topk rounded up to 32 entries: slot_ids, rank,
// owner, ucount, uoffset (ms+1), list, group_ux, group_first, group_cnt, scalars[4] (number of distinct experts,
// number of groups) and 3 spare entries, then the job order of the groups gorder (groups sorted by slot count),
// the token of each list entry ltok, the expert id of each group group_eid and the first job of each of the CTA's
// warps and of the next CTA (17 entries).
__host__ __device__ constexpr int route_ints(int ms) { return 9 * ms + 8 + 3 * ms + 17; }

// Relative cost of one job (R rows of one projection, all chunks) serving C routed slots: cost_a + cost_b * C
// (the decode and the streaming are shared, the FMAs grow with C; fitted to measured times of uniform
// routings with 1, 2 and 4 slots per expert). The pure-read instrument costs the same for every C.
__device__ __forceinline__ long long job_cost(int C, bool pure, int a, int b) { return pure ? 1 : a + (long long)b * C; }

// floor(a / b) for 0 <= a and 0 < b, as a 32-bit division whenever both fit (a 64-bit integer division is a long
// emulated sequence, and every warp needs a few at its start).
__device__ __forceinline__ long long floor_div(long long a, long long b) {
    if (a < 0x80000000LL && b < 0x80000000LL) return (long long)((uint32_t)a / (uint32_t)b);
    return a / b;
}

__host__ __device__ constexpr uint32_t moe_slot_bytes(int R, int UPL) {
    return (uint32_t)(((R * 32 * UPL * 18) + 127) / 128 * 128);
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// SWIGLU: a job streams R gate rows and the same R up rows of its expert (one slot of 2R rows) and writes
// silu(gate) * up per routed row; otherwise a job is R rows of one projection.
// XG: the tokens are staged in groups of 32 blocks (K/32 a multiple of 32), so a lane's quads sit at constant
// offsets; otherwise token-major with the quads K/32 * 16 bytes apart.
template <int R, int W, int D, int UPL, bool PURE, bool SWIGLU, bool XG>
__global__ void __launch_bounds__(W * 32, 1) moe_q4_kernel(const MoEParams p) {
    static_assert(!(PURE && SWIGLU), "the pure-read instrument streams one projection per job");
    constexpr int NP = SWIGLU ? 1 : 2;      // jobs per (group, row group)
    constexpr int RR = SWIGLU ? 2 * R : R;  // rows per slot
    constexpr int kThreads = W * 32;
    constexpr int CB = 32 * UPL;
    constexpr uint32_t QROW = CB * 16u;
    constexpr uint32_t QBYTES = RR * QROW;
    constexpr uint32_t SLOT = moe_slot_bytes(RR, UPL);
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int TK = p.T * p.topk;

    int* route = reinterpret_cast<int*>(smem + p.route_off);
    int* slot_ids = route;
    const int ms = p.ms;
    int* rank = route + ms;
    int* owner = route + 2 * ms;
    int* ucount = route + 3 * ms;
    int* uoffset = route + 4 * ms;  // ms + 1 entries
    int* list = route + 5 * ms + 1;
    int* group_ux = route + 6 * ms + 1;
    int* group_first = route + 7 * ms + 1;
    int* group_cnt = route + 8 * ms + 1;
    int* scalars = route + 9 * ms + 1;
    int* gorder = route + 9 * ms + 8;
    int* ltok = gorder + ms;  // token of each list entry (slot / topk), so stages divide nothing
    int* group_eid = ltok + ms;  // expert id of each group
    int* jr = group_eid + ms;    // job ranges of the CTA's warps: warp w takes [jr[w], jr[w + 1])

    const uint32_t s_base = smem_addr(smem);
    const uint32_t xs = s_base + p.xs_off;
    const uint32_t aux = s_base + p.aux_off;
    const int U = p.nblk;
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
    const int rgs = (p.N + R - 1) / R;
    // Groups run in order of slot count. Round-robin dealing (p.deal = 1): warp gw (numbered across CTAs
    // first) takes jobs gw, gw + Wtot, ..., so at any moment the grid sweeps neighbouring rows of one expert
    // matrix and the warps of an SM run the same compiled stage body. Range dealing (p.deal = 0): warps
    // numbered CTA by CTA own contiguous job ranges of equal estimated cost.
    const int gw = p.deal ? warp * (int)gridDim.x + (int)blockIdx.x : (int)blockIdx.x * W + warp;
    const int Wtot = (int)gridDim.x * W;

    // Single-warp routing (at most 64 slots) keeps a 64-bit slot mask per expert in the ring's shared memory, which
    // no copy reaches before the routing is over; the masks are cleared while the previous kernel finishes.
    const bool route1 = TK <= 64 && (long long)p.E * 8 <= (long long)W * D * SLOT;
    unsigned long long* const emask = reinterpret_cast<unsigned long long*>(smem + p.slots_off);
    if (route1) {
        for (int e = threadIdx.x; e < p.E; e += kThreads) emask[e] = 0ull;
        __syncthreads();
    }

    // Routing reads the expert ids and the first weight copies depend on it, so wait for the previous kernel
    // in the stream (it may have written ids, x or the outputs) before anything else.
    grid_dependency_wait();
    grid_launch_dependents();

    // Staging of the T inputs by threads t0 .. t0 + cnt - 1 (whole warps): four lanes per 32-element block, lane
    // t of the group holding quads 2t and 2t+1 (largest magnitude by two group shuffles). Each
    // thread issues the loads of up to kBatch of its block quarters before using any, so staging costs one round
    // trip to the L2 per kBatch quarters.
    constexpr int kBatch = 12;
    const int nb_all = p.T * U;
    const int nthr = (nb_all * 4 + 31) & ~31;  // whole warps, so the group shuffles always see 32 lanes
    auto stage_inputs = [&](int t0, int cnt) {
        if constexpr (!PURE) {
            const int me = (int)threadIdx.x - t0;
            const int t4 = lane & 3;
            for (int base = me; base < nthr; base += cnt * kBatch) {
                float4 xa[kBatch], xb[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int blk = (base + j * cnt) >> 2;
                    const bool in = blk < nb_all;
                    const float4* src = reinterpret_cast<const float4*>(p.x) + (size_t)(in ? blk : 0) * 8 + 2 * t4;
                    xa[j] = in ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xb[j] = in ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                int ej[kBatch];
                stage_blocks4<kBatch>(xa, xb, t4 >> 1, ej);  // quarters past the end stage zeros and are not stored
                DivWalk vu(base >> 2, cnt >> 2, U);            // (token, block) of quarter j's block
#pragma unroll
                for (int j = 0; j < kBatch; ++j, vu.next()) {
                    const int blk = (base + j * cnt) >> 2;
                    if (blk < nb_all) {
                        const int v = vu.q;
                        const int u = vu.r;
                        // XG layout: [group of 32 blocks][token][quad][block in group, then a pad]; otherwise
                        // [token][quad][block] (16 bytes each): the lanes of a warp read consecutive 16-byte pieces
                        const int grp32 = u >> 5, ul = u & 31;
                        const int q0 = 2 * t4;
                        const uint32_t a0 = xs + (uint32_t)(XG ? (((grp32 * p.T + v) * 8 + q0) * kXGRow + ul) * 16
                                                               : ((v * 8 + q0) * U + u) * 16);
                        const uint32_t qstep = XG ? kXGRow * 16u : (uint32_t)U * 16u;
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "f"(xa[j].x), "f"(xa[j].y),
                                     "f"(xa[j].z), "f"(xa[j].w)
                                     : "memory");
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + qstep), "f"(xb[j].x),
                                     "f"(xb[j].y), "f"(xb[j].z), "f"(xb[j].w)
                                     : "memory");
                        if (t4 == 0)
                            asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(aux + (uint32_t)((XG ? (grp32 * p.T + v) * 32 + ul
                                                                                                    : v * U + u) * 8)),
                                         "f"(block_factor(ej[j])), "f"(0.0f)
                                         : "memory");
                    }
                }
            }
        }
    };

    // Job order of the groups: stable by slot count (the groups of one slot in index order, then those of two, ...),
    // so the n_c groups of count c take the positions from N_c on (N_c: the groups of fewer slots). Each group has
    // NP * rgs jobs of cost job_cost(c), so the cost before class c is B_c = sum over c' < c of
    // n_c' * NP * rgs * job_cost(c'), and the job where the cost reaches x inside class c is
    // N_c * NP * rgs + floor((x - B_c) / job_cost(c)): each warp's share of the total cost becomes a contiguous job
    // range [j0, j1) with no table of cumulative costs and no search (groups with more routed slots spread over
    // more warps).
    auto order_and_ranges = [&]() {
        const int ngroups = scalars[1];
        const int jobs = ngroups * NP * rgs;
        const unsigned lt = (1u << lane) - 1u;
        int n[kMaxC + 1];  // groups per slot count (n[0] unused)
#pragma unroll
        for (int cc = 0; cc <= kMaxC; ++cc) n[cc] = 0;
        for (int c0 = 0; c0 < ngroups; c0 += 32) {
            const int gi = c0 + lane;
            const int c = gi < ngroups ? group_cnt[gi] : 0;
#pragma unroll
            for (int cc = 1; cc <= kMaxC; ++cc) n[cc] += __popc(__ballot_sync(0xffffffffu, c == cc));
        }
        int next[kMaxC + 1];  // next free position of each class
        next[1] = 0;
#pragma unroll
        for (int cc = 2; cc <= kMaxC; ++cc) next[cc] = next[cc - 1] + n[cc - 1];
        for (int c0 = 0; c0 < ngroups; c0 += 32) {
            const int gi = c0 + lane;
            const int c = gi < ngroups ? group_cnt[gi] : 0;
            int pos = 0;
#pragma unroll
            for (int cc = 1; cc <= kMaxC; ++cc) {
                const unsigned b = __ballot_sync(0xffffffffu, c == cc);
                if (c == cc) pos = next[cc] + __popc(b & lt);
                next[cc] += __popc(b);
            }
            if (gi < ngroups) gorder[pos] = gi;
        }
        // the first job of each of this CTA's warps and of the next CTA's first warp (range dealing)
        if (!p.deal && lane <= W) {
            long long bc[kMaxC + 2];  // B_c
            int nc[kMaxC + 2];        // N_c
            bc[1] = 0;
            nc[1] = 0;
#pragma unroll
            for (int cc = 1; cc <= kMaxC; ++cc) {
                nc[cc + 1] = nc[cc] + n[cc];
                bc[cc + 1] = bc[cc] + (long long)n[cc] * NP * rgs * job_cost(cc, PURE, p.cost_a, p.cost_b);
            }
            const long long cb = bc[kMaxC + 1];
            const long long x = floor_div(cb * ((int)blockIdx.x * W + lane), Wtot);
            int j = jobs;
            if (x < cb) {
                // the class holding cost x: the last non-empty class that starts at or before x
                long long b0 = 0, jc = job_cost(1, PURE, p.cost_a, p.cost_b);
                int n0 = 0;
#pragma unroll
                for (int cc = 2; cc <= kMaxC; ++cc)
                    if (n[cc] > 0 && bc[cc] <= x) {
                        b0 = bc[cc];
                        n0 = nc[cc];
                        jc = job_cost(cc, PURE, p.cost_a, p.cost_b);
                    }
                j = n0 * NP * rgs + (int)floor_div(x - b0, jc);
            }
            jr[lane] = j;
        }
    };

    // ---- routing, with the inputs staged beside it --------------------------------------------------
    if (route1) {
        // Warp 0 routes alone, two slots per lane (slots lane and lane + 32), while the other warps stage the
        // inputs. Each valid slot sets its bit in its expert's 64-bit slot mask (cleared before the dependency
        // wait); the mask then gives the slot's first equal slot, its rank among them and, on the first slot, their
        // count. The tables come out as the general path's.
        if (warp == 0) {
            const unsigned full = 0xffffffffu, lt = (1u << lane) - 1u;
            const int i0 = lane, i1 = lane + 32;
            const int e0 = i0 < TK ? __ldg(p.ids + i0) : -1;
            const int e1 = i1 < TK ? __ldg(p.ids + i1) : -1;
            const bool v0 = i0 < TK && e0 >= 0 && e0 < p.E, v1 = i1 < TK && e1 >= 0 && e1 < p.E;
            if (v0) atomicOr(emask + e0, 1ull << i0);
            if (v1) atomicOr(emask + e1, 1ull << i1);
            __syncwarp();
            const unsigned long long m0 = v0 ? emask[e0] : 0ull, m1 = v1 ? emask[e1] : 0ull;
            // the ring's copies overwrite the table once the routing is over
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const int rank0 = __popcll(m0 & ((1ull << i0) - 1ull)), first0 = v0 ? __ffsll((long long)m0) - 1 : i0;
            const int rank1 = __popcll(m1 & ((1ull << i1) - 1ull)), first1 = v1 ? __ffsll((long long)m1) - 1 : i1;
            const bool isf0 = v0 && first0 == i0, isf1 = v1 && first1 == i1;
            // distinct experts numbered by first appearance (slots 0..31, then 32..63)
            const unsigned b0 = __ballot_sync(full, isf0), b1 = __ballot_sync(full, isf1);
            const int nux0 = __popc(b0);
            const int uxf0 = __popc(b0 & lt), uxf1 = nux0 + __popc(b1 & lt);  // on first slots
            // each expert's slot count and group count on its first slot, then exclusive prefix sums in that order
            const int cnt0 = isf0 ? __popcll(m0) : 0, cnt1 = isf1 ? __popcll(m1) : 0;
            const int ng0 = (cnt0 + kMaxC - 1) / kMaxC, ng1 = (cnt1 + kMaxC - 1) / kMaxC;
            int ic0 = cnt0, ig0 = ng0, ic1 = cnt1, ig1 = ng1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int a = __shfl_up_sync(full, ic0, off), b = __shfl_up_sync(full, ig0, off);
                const int c = __shfl_up_sync(full, ic1, off), d = __shfl_up_sync(full, ig1, off);
                if (lane >= off) {
                    ic0 += a;
                    ig0 += b;
                    ic1 += c;
                    ig1 += d;
                }
            }
            const int tc0 = __shfl_sync(full, ic0, 31), tg0 = __shfl_sync(full, ig0, 31);
            const int ngroups_f = tg0 + __shfl_sync(full, ig1, 31);
            const int uoff0 = ic0 - cnt0, goff0 = ig0 - ng0;
            const int uoff1 = tc0 + ic1 - cnt1, goff1 = tg0 + ig1 - ng1;
            if (isf0)
                for (int gi = 0; gi < ng0; ++gi) {
                    group_ux[goff0 + gi] = uxf0;
                    group_first[goff0 + gi] = uoff0 + gi * kMaxC;
                    group_cnt[goff0 + gi] = min(kMaxC, cnt0 - gi * kMaxC);
                    group_eid[goff0 + gi] = e0;
                }
            if (isf1)
                for (int gi = 0; gi < ng1; ++gi) {
                    group_ux[goff1 + gi] = uxf1;
                    group_first[goff1 + gi] = uoff1 + gi * kMaxC;
                    group_cnt[goff1 + gi] = min(kMaxC, cnt1 - gi * kMaxC);
                    group_eid[goff1 + gi] = e1;
                }
            // each slot's expert index (the first slots before its own first slot) and list position (from its first
            // slot's lane)
            const unsigned long long fb = (unsigned long long)b0 | ((unsigned long long)b1 << 32);  // first slots
            const int ux0 = __popcll(fb & ((1ull << first0) - 1ull)), ux1 = __popcll(fb & ((1ull << first1) - 1ull));
            const int uo0 = __shfl_sync(full, uoff0, first0 & 31);
            const int uo1a = __shfl_sync(full, uoff0, first1 & 31), uo1b = __shfl_sync(full, uoff1, first1 & 31);
            const int uo1 = first1 < 32 ? uo1a : uo1b;
            if (i0 < TK) {
                slot_ids[i0] = e0;
                owner[i0] = v0 ? ux0 : -1;
                if (v0) {
                    list[uo0 + rank0] = i0;
                    ltok[uo0 + rank0] = i0 / p.topk;
                }
            }
            if (i1 < TK) {
                slot_ids[i1] = e1;
                owner[i1] = v1 ? ux1 : -1;
                if (v1) {
                    list[uo1 + rank1] = i1;
                    ltok[uo1 + rank1] = i1 / p.topk;
                }
            }
            if (lane == 0) {
                scalars[0] = nux0 + __popc(b1);
                scalars[1] = ngroups_f;
            }
            __syncwarp();
            order_and_ranges();
        } else {
            stage_inputs(32, kThreads - 32);
        }
        __syncthreads();
    } else {
        for (int i = threadIdx.x; i < TK; i += kThreads) {
            slot_ids[i] = __ldg(p.ids + i);
            ucount[i] = 0;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < TK; i += kThreads) {
            const int e = slot_ids[i];
            int first = -1, rk = 0;
            if (e >= 0 && e < p.E) {
                // the earlier slots four at a time (the table starts 16-byte aligned and has ms >= TK entries)
                const int4* const s4 = reinterpret_cast<const int4*>(slot_ids);
                for (int j = 0; j < i; j += 4) {
                    const int4 v = s4[j >> 2];
                    const bool m0 = v.x == e, m1 = v.y == e && j + 1 < i, m2 = v.z == e && j + 2 < i,
                               m3 = v.w == e && j + 3 < i;
                    if (first < 0) first = m0 ? j : m1 ? j + 1 : m2 ? j + 2 : m3 ? j + 3 : -1;
                    rk += (int)m0 + (int)m1 + (int)m2 + (int)m3;
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
        const int ngr = scalars[1];
        for (int i = threadIdx.x; i < TK; i += kThreads) {
            const int ux = owner[i];
            if (ux >= 0) {
                list[uoffset[ux] + rank[i]] = i;
                ltok[uoffset[ux] + rank[i]] = i / p.topk;
            }
        }
        __syncthreads();
        // group -> expert id
        for (int gi = threadIdx.x; gi < ngr; gi += kThreads) group_eid[gi] = slot_ids[list[uoffset[group_ux[gi]]]];
        __syncthreads();
        if (warp == 0) order_and_ranges();
        else stage_inputs(32, kThreads - 32);
        __syncthreads();
    }
    const int ngroups = scalars[1];

    // ---- jobs -------------------------------------------------------------------------------------------
    const int jobs = ngroups * NP * rgs;
    const int j0 = p.deal ? gw : jr[warp];
    const int j1 = p.deal ? (gw < jobs ? gw + ((jobs - 1 - gw) / Wtot + 1) : gw) : jr[warp + 1];
    const int jstep = p.deal ? Wtot : 1;  // job stride of this warp
    const uint64_t pol = policy_evict_first();

    // Job cursor: group, projection, row group, chunk. Jobs run group-major, then projection, then row
    // group, so a warp's stages walk consecutive rows of one expert matrix.
    struct Cursor {
        int grp, sp, rg, c;
    };
    auto cursor_at = [&](int j) {
        Cursor k;
        k.grp = j / (NP * rgs);
        const int rem = j - k.grp * NP * rgs;
        k.sp = NP == 2 && rem >= rgs ? 1 : 0;  // rem < NP * rgs
        k.rg = rem - k.sp * rgs;
        k.c = 0;
        return k;
    };
    auto advance = [&](Cursor& k) {
        if (++k.c == p.S) {
            k.c = 0;
            k.rg += jstep;
            while (k.rg >= rgs) {
                k.rg -= rgs;
                if (++k.sp == NP) {
                    k.sp = 0;
                    ++k.grp;
                }
            }
        }
    };

    const int total = (p.deal ? (j1 - j0) : (j1 - j0)) * p.S;  // jobs of this warp x chunks
    Cursor ik = cursor_at(j0);
    int issued = 0, islot = 0;
    bool aborted = false;  // a stage wait ran out: no more copies, the warp's remaining rows are NaN
    auto issue = [&]() {
        if (issued < total && !aborted) {
            const int e = group_eid[gorder[ik.grp]];
            const int r0 = ik.rg * R;
            const int rv = min(R, p.N - r0);
            const int b0 = ik.c * CB;
            const int nb = min(CB, p.nblk - b0);
            const size_t row0 = (size_t)e * p.N + r0;
            const uint32_t slot = ring + (uint32_t)islot * SLOT;
            if (p.bulk && lane == 0) {
                // this warp's earlier reads of the slot are ordered before the asynchronous writes
                const uint32_t bar = bars + 8u * (uint32_t)islot;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_expect_tx(bar, (uint32_t)((SWIGLU ? 2 : 1) * rv) * (QROW + CB * 2));
            }
#pragma unroll
            for (int sp = 0; sp < (SWIGLU ? 2 : 1); ++sp) {
                const int proj = SWIGLU ? sp : ik.sp;
                const uint8_t* q = proj == 0 ? p.qg : p.qu;
                const uint16_t* d = proj == 0 ? p.dg : p.du;
                const uint32_t qdst = slot + (uint32_t)(sp * R) * QROW;
                const uint32_t ddst = slot + QBYTES + (uint32_t)(sp * R * CB * 2);
                if (p.bulk) {
                    if (lane == 0) {
                        const uint32_t bar = bars + 8u * (uint32_t)islot;
                        bulk_copy(qdst, q + row0 * QROW, (uint32_t)rv * QROW, bar, pol);
                        bulk_copy(ddst, d + row0 * CB, (uint32_t)(rv * CB * 2), bar, pol);
                    }
                } else if (nb == CB && p.S == 1) {
                    warp_copy_async(qdst, q + row0 * QROW, (uint32_t)rv * QROW, lane, pol);
                    if (p.dcopy) warp_copy_async(ddst, d + row0 * CB, (uint32_t)(rv * CB * 2), lane, pol);
                } else {
                    for (int r = 0; r < rv; ++r) {
                        const size_t rb = (row0 + r) * p.nblk + b0;
                        warp_copy_async(qdst + (uint32_t)r * QROW, q + rb * 16, (uint32_t)(nb * 16), lane, pol);
                        if (p.dcopy)
                            warp_copy_async(ddst + (uint32_t)(r * CB * 2), d + rb, (uint32_t)(nb * 2), lane, pol);
                    }
                }
                if (!p.dcopy) {
                    // scales that cannot move by 16-byte copies (not 16-byte aligned, or K/32 not a multiple of
                    // 8) go into the slot by plain loads, so the stage body always reads them from shared memory
                    uint16_t* const ds = reinterpret_cast<uint16_t*>(smem + (ddst - s_base));
                    for (int r = 0; r < rv; ++r)
                        for (int u = lane; u < nb; u += 32) ds[r * CB + u] = __ldg(d + (row0 + r) * p.nblk + b0 + u);
                }
            }
            advance(ik);
            ++issued;
            islot = islot + 1 == D ? 0 : islot + 1;
        }
        if (!p.bulk) cp_async_commit();
    };

#pragma unroll
    for (int k = 0; k < D - 1; ++k) issue();

    // With the first copies in flight: each block's -8 offset term (the unit chain on codes of 8 over its staged
    // quads) and, in CTA 0, the invalid slots' NaN rows and status bit.
    if constexpr (!PURE) {
        DivWalk vu((int)threadIdx.x, kThreads, U);
        for (int b = threadIdx.x; b < nb_all; b += kThreads, vu.next()) {
            const int v = vu.q;
            const int u = vu.r;
            const int grp32 = u >> 5, ul = u & 31;
            const uint32_t q0 = xs + (uint32_t)(XG ? (((grp32 * p.T + v) * 8) * kXGRow + ul) * 16 : ((v * 8) * U + u) * 16);
            const uint32_t qstep = XG ? kXGRow * 16u : (uint32_t)U * 16u;
            float4 xq[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) xq[q] = lds128f(q0 + (uint32_t)q * qstep);
            const uint32_t a = aux + (uint32_t)((XG ? (grp32 * p.T + v) * 32 + ul : v * U + u) * 8);
            const float bias = q4_block_bias(xq, lds32f(a));
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(a + 4u), "f"(bias) : "memory");
        }
    }
    if (blockIdx.x == 0) {
        for (int i = 0; i < TK; ++i) {
            if (owner[i] >= 0) continue;
            for (int r = threadIdx.x; r < p.N; r += kThreads) {
                p.yg[(size_t)i * p.N + r] = __int_as_float(0x7fc00000);
                if constexpr (!SWIGLU) p.yu[(size_t)i * p.N + r] = __int_as_float(0x7fc00000);  // no y_up
            }
            if (threadIdx.x == 0) {
                if (p.status) atomicOr(reinterpret_cast<unsigned*>(p.status), (unsigned)kFaultBadExpert);
                atomicOr(p.fault, (unsigned)kFaultBadExpert);
            }
        }
    }
    __syncthreads();

    float tot[RR][kMaxC];
    uint32_t fold[RR];
#pragma unroll
    for (int r = 0; r < RR; ++r) {
        fold[r] = 0u;
#pragma unroll
        for (int m = 0; m < kMaxC; ++m) tot[r][m] = 0.f;
    }

    Cursor k = cursor_at(j0);
    int cslot = 0;
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
        const bool bad = aborted;
        const uint32_t slot = ring + (uint32_t)cslot * SLOT;
        const int grp = gorder[k.grp];
        const int cnt = group_cnt[grp];
        const int first = group_first[grp];
        const int r0 = k.rg * R;
        const int rv = min(R, p.N - r0);
        const int b0 = k.c * CB;
        const int nb = min(CB, p.nblk - b0);
        const uint32_t qb = slot + (uint32_t)lane * 16u;
        const uint32_t db = slot + QBYTES + (uint32_t)lane * 2u;

        // Stage body for C routed slots (compile-time), C = cnt.
        auto stage = [&](auto cc) {
            constexpr int C = decltype(cc)::value;
            // this lane's staged quads and block pairs of each routed token: from the stage's first group of 32
            // blocks of that token (x_it, a_it: the step to the next group)
            const float4* xq[C];
            const float2* aq[C];
            const int qs = XG ? kXGRow : U;  // quad stride (float4)
            const int x_it = XG ? p.T * 8 * kXGRow : 32, a_it = XG ? p.T * 32 : 32;
            (void)qs;  // the pure read uses none of these
            (void)x_it;
            (void)a_it;
#pragma unroll
            for (int m = 0; m < C; ++m) {
                const int tok = ltok[first + m];
                xq[m] = reinterpret_cast<const float4*>(smem + p.xs_off) +
                        (XG ? ((b0 >> 5) * p.T + tok) * 8 * kXGRow + lane : tok * 8 * U + b0 + lane);
                aq[m] = reinterpret_cast<const float2*>(smem + p.aux_off) +
                        (XG ? ((b0 >> 5) * p.T + tok) * 32 + lane : tok * U + b0 + lane);
            }
#pragma unroll 1
            for (int it = 0; it < UPL; ++it) {
                const int ul = it * 32 + lane;
                if (ul >= nb || bad) continue;
                uint4 w[RR];
                float dsc[RR];
                uint32_t dbits[RR];
#pragma unroll
                for (int r = 0; r < RR; ++r) {
                    // slot row r: projection (SWIGLU ? r / R : k.sp), expert row r0 + r % R
                    w[r] = lds128(qb + (uint32_t)r * QROW + (uint32_t)(it * 512));
                    dbits[r] = lds_u16(db + (uint32_t)(r * CB * 2 + it * 64));
                    dsc[r] = f16_bits_to_f32(dbits[r]);
                }
                if constexpr (PURE) {
#pragma unroll
                    for (int r = 0; r < RR; ++r) fold[r] ^= w[r].x ^ w[r].y ^ w[r].z ^ w[r].w ^ dbits[r];
                } else {
                    float2 acc[RR][C];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        Word8s d8[RR];
#pragma unroll
                        for (int r = 0; r < RR; ++r)
                            d8[r] = decode_word_sub(i == 0 ? w[r].x : i == 1 ? w[r].y : i == 2 ? w[r].z : w[r].w);
#pragma unroll
                        for (int m = 0; m < C; ++m) {
                            const float4 xl = xq[m][it * x_it + i * qs];
                            const float4 xh = xq[m][it * x_it + (4 + i) * qs];
#pragma unroll
                            for (int r = 0; r < RR; ++r)
                                acc[r][m] = word_fma(d8[r], xl, xh, i == 0 ? make_float2(0.f, 0.f) : acc[r][m]);
                        }
                    }
#pragma unroll
                    for (int m = 0; m < C; ++m) {
                        const float2 fa = aq[m][it * a_it];
#pragma unroll
                        for (int r = 0; r < RR; ++r) {
                            const float t = fmaf(acc[r][m].x + acc[r][m].y, fa.x, fa.y);
                            tot[r][m] = fmaf(dsc[r], t, tot[r][m]);
                        }
                    }
                }
            }
            __syncwarp();  // every lane is done with this slot before a later stage overwrites it

            if (k.c == p.S - 1) {
                float* y = k.sp == 0 ? p.yg : p.yu;
                (void)y;
                if constexpr (PURE) {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) fold[r] ^= __shfl_xor_sync(0xffffffffu, fold[r], off);
                        if (lane < cnt && r < rv)
                            y[(size_t)list[first + lane] * p.N + r0 + r] = bad ? NAN : __uint_as_float(fold[r]);
                        fold[r] = 0u;
                    }
                } else {
                    constexpr int NV = RR * C;
                    constexpr int P2 = NextPow2<NV>::value;
                    constexpr int L2 = log2_const<P2>();
                    float vals[P2];
#pragma unroll
                    for (int i = 0; i < P2; ++i) vals[i] = 0.f;
#pragma unroll
                    for (int r = 0; r < RR; ++r)
#pragma unroll
                        for (int m = 0; m < C; ++m) {
                            vals[r * C + m] = tot[r][m];
                            tot[r][m] = 0.f;
                        }
                    warp_transpose_reduce<P2>(vals, lane);
                    const int idx = lane >> (5 - L2);
                    const bool leader = (lane & ((1 << (5 - L2)) - 1)) == 0;
                    if constexpr (SWIGLU) {
                        // the up total of (row r, slot m) sits R*C lane groups after its gate total
                        const float up = __shfl_down_sync(0xffffffffu, vals[0], (R * C) << (5 - L2));
                        if (leader && idx < R * C) {
                            const int r = idx / C;
                            const int m = idx - r * C;
                            if (r < rv) p.yg[(size_t)list[first + m] * p.N + r0 + r] = bad ? NAN : silu(vals[0]) * up;
                        }
                    } else if (leader && idx < NV) {
                        const int r = idx / C;
                        const int m = idx - r * C;
                        if (r < rv) y[(size_t)list[first + m] * p.N + r0 + r] = bad ? NAN : vals[0];
                    }
                }
            }
        };
        if constexpr (PURE) {
            stage(std::integral_constant<int, 1>{});
        } else {
            switch (cnt) {
                case 1: stage(std::integral_constant<int, 1>{}); break;
                case 2: stage(std::integral_constant<int, 2>{}); break;
                case 3: stage(std::integral_constant<int, 3>{}); break;
                default: stage(std::integral_constant<int, 4>{}); break;
            }
        }
        advance(k);
        if (++cslot == D) {
            cslot = 0;
            cphase ^= 1u;
        }
    }
    // bulk copies issued but not consumed (only after a wait ran out): let them land before the CTA exits
    if (p.bulk)
        for (int st = consumed; st < issued; ++st)
            if (!warp_wait_bounded(bars + 8u * (uint32_t)(st % D), (uint32_t)((st / D) & 1), kDrainCycles) &&
                lane == 0)
                atomicOr(p.fault, kFaultCopyLost);
}

inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

template <int R, int W, int D, int UPL, bool PURE, bool SWIGLU, bool XG>
cudaError_t launch_kernel_cfg(const DeviceInfo& di, const MoEParams& p, uint32_t smem, cudaStream_t s) {
    auto kern = moe_q4_kernel<R, W, D, UPL, PURE, SWIGLU, XG>;
    static std::once_flag attr_once[64];
    cudaError_t err = cudaSuccess;
    std::call_once(attr_once[di.device & 63], [&] {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, di.sm_count, W * 32, smem, s, p);
}

template <int R, int W, int D, int UPL, bool PURE, bool SWIGLU>
cudaError_t launch_fixed(const DeviceInfo& di, MoEParams p, cudaStream_t s) {
    const uint32_t route = (uint32_t)round_up(route_ints(p.ms) * 4, 128);
    const uint32_t xsb = PURE ? 0u : (uint32_t)round_up(p.T * p.K / 32 * kXGRow * 4 + 512, 128);  // either layout
    const uint32_t axb = PURE ? 0u : (uint32_t)round_up(p.T * p.nblk * 8, 128);
    p.route_off = 0;
    p.xs_off = route;
    p.aux_off = route + xsb;
    p.bar_off = route + xsb + axb;
    p.slots_off = p.bar_off + (uint32_t)round_up(W * D * 8, 128);  // slot mbarriers
    const uint32_t smem = p.slots_off + (uint32_t)(W * D) * moe_slot_bytes(SWIGLU ? 2 * R : R, UPL);
    if (smem > (uint32_t)di.max_smem_optin) return cudaErrorNotSupported;
    p.S = (p.nblk + 32 * UPL - 1) / (32 * UPL);
    p.bulk = (p.dcopy && p.S == 1 && p.nblk == 32 * UPL) ? 1 : 0;
    // grouped staging whenever the blocks fill whole groups of 32 (no padding); the pure read stages nothing
    if constexpr (!PURE) {
        if (p.nblk % 32 == 0) return launch_kernel_cfg<R, W, D, UPL, PURE, SWIGLU, true>(di, p, smem, s);
    }
    return launch_kernel_cfg<R, W, D, UPL, PURE, SWIGLU, false>(di, p, smem, s);
}

// Ring depth 2 (depths 3 and 4 measured no faster with the bulk copies and are not compiled).
template <int R, int W, int UPL, bool PURE, bool SWIGLU>
cudaError_t launch_upl(const DeviceInfo& di, const MoEParams& p, int depth, cudaStream_t s) {
    (void)depth;
    return launch_fixed<R, W, 2, UPL, PURE, SWIGLU>(di, p, s);
}

// Whole rows in one chunk up to K = 4096 (UPL = 1, 2, 4), longer rows in 128-block chunks; the deepest ring
// of depth 2 beside the routing tables and the staged tokens.
template <int R, int W, bool PURE, bool SWIGLU = false>
cudaError_t launch(const DeviceInfo& di, const MoEParams& p, int depth, cudaStream_t s) {
    cudaError_t e = cudaErrorNotSupported;
    if (p.nblk <= 32) e = launch_upl<R, W, 1, PURE, SWIGLU>(di, p, depth, s);
    else if (p.nblk <= 64) e = launch_upl<R, W, 2, PURE, SWIGLU>(di, p, depth, s);
    if (e == cudaErrorNotSupported) e = launch_upl<R, W, 4, PURE, SWIGLU>(di, p, depth, s);
    if (e == cudaErrorNotSupported) e = launch_upl<R, W, 1, PURE, SWIGLU>(di, p, depth, s);
    return e;
}

}  // namespace

cudaError_t launch_moe_q4_gemv(float* y_gate, float* y_up, const uint8_t* qs_gate, const uint16_t* d_gate,
                               const uint8_t* qs_up, const uint16_t* d_up, const float* x, const int32_t* ids,
                               int T, int topk, int E, int N, int K, int32_t* dev_status, bool pure_read,
                               bool swiglu, cudaStream_t s) {
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
    p.ms = (T * topk + 31) / 32 * 32;
    p.dcopy = (p.nblk % 8 == 0) && ((reinterpret_cast<uintptr_t>(d_gate) & 15u) == 0) &&
              ((reinterpret_cast<uintptr_t>(d_up) & 15u) == 0);
    p.fault = device_fault_word(di.device);
    p.wait_cycles = wait_limit_cycles();
    if (!p.fault) return cudaErrorInvalidSymbol;
    // plans from sweeps over routing seeds and launch shapes: 8 warps x 8 rows per stage (a staged input quad
    // serves 8 rows; 16 warps x 4 rows needs more than the 128 registers a 512-thread CTA allows per thread),
    // ring depth 2, contiguous cost-balanced job ranges; the SwiGLU form (4 gate + 4 up rows per slot) 8 warps
    // with round-robin dealing
    const int depth = 2;
    p.cost_a = 9;
    p.cost_b = 5;
    p.deal = swiglu ? 1 : 0;
    // 8 warps x 8 rows when the ring fits beside the staged tokens, else 8 warps x 4 rows; the pure read
    // streams with the same plan
    if (swiglu) {  // R gate + R up rows per slot
        e = launch<4, 8, false, true>(di, p, depth, s);
        return e == cudaErrorNotSupported ? launch<2, 8, false, true>(di, p, depth, s) : e;
    }
    if (pure_read) {
        e = launch<8, 8, true>(di, p, depth, s);
        return e == cudaErrorNotSupported ? launch<4, 8, true>(di, p, depth, s) : e;
    }
    e = launch<8, 8, false>(di, p, depth, s);
    return e == cudaErrorNotSupported ? launch<4, 8, false>(di, p, depth, s) : e;
}


}  // namespace q4
