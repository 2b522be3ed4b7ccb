// MoE router for sm_103a: gate GEMV over the experts + top-K softmax, fused in one kernel.
//
// Problem (spark_model `gemm_quant.rs`, moe_gate_topk_fused): gate[e] = x . Wgate[e] for every expert, then the
// indices of the K largest logits and their softmax weights (optionally renormalised over the K). Here Wgate is
// planar Q4 (E rows of K weights, the library's format) and x is fp32; one token per CTA row of the grid.
//
// Kernel shape (one cluster of CS CTAs per token; the router matrix is small and stays in L2 after the first
// cluster reads it):
//  * every CTA stages the token's x block by block with the bias-free decode's per-block scaling
//    (device_common.cuh);
//  * CTA c of the cluster computes the logits of experts c, c + CS, ...: warp w takes experts c + CS*w,
//    c + CS*(w + W), ... two rows at a time; lane l takes units l, l + 32, ... with 16-byte loads (four issued
//    before use), one shift + eight ANDs per word and packed fp32x2 FMAs, folds each block with its scale, and
//    the warp sums the lanes; the logits go to the CTA's own shared memory;
//  * after a cluster barrier, CTA 0 gathers the other CTAs' logits through distributed shared memory; a second
//    barrier releases them; its warp 0 then takes the softmax over all E logits (max subtracted) and the top K
//    by a 64-bit key (the logit's order-preserving bits, a NaN below every other value, then the complement of
//    the index, so ties go to the lower index): up to 64 experts by each expert's rank among all keys (one
//    pass of shuffles), otherwise by K arg-max passes with taken experts marked in per-lane bit masks; it
//    writes ids and weights (the logits, when asked, come from every CTA).
#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

struct RouterParams {
    int32_t* ids;
    float* weights;
    float* logits;  // nullable
    const uint8_t* qs;
    const uint16_t* d;
    const float* x;
    int T, E, K, nblk, topk, normalize;
    uint32_t xs_off, aux_off, lg_off;
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster: writes before the barrier are visible to reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A float in CTA `rank`'s shared memory at this CTA's shared address `local`.
__device__ __forceinline__ float ld_cluster_f32(uint32_t local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <int W, int CS>
__global__ void __launch_bounds__(W * 32, 1) moe_router_kernel(const RouterParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int t = (int)blockIdx.x / CS;
    const int c = (int)cluster_ctarank();
    const uint32_t s_base = smem_addr(smem);
    const uint32_t xs = s_base + p.xs_off;
    const uint32_t aux = s_base + p.aux_off;
    float* lg = reinterpret_cast<float*>(smem + p.lg_off);

    // x belongs to the previous kernel in the stream when launches overlap.
    grid_dependency_wait();
    grid_launch_dependents();

    // stage x[t]: four lanes per 32-element block (whole warps take part in the group shuffles)
    {
        const float* xt = p.x + (size_t)t * p.K;
        const int t4 = lane & 3;
        const int nthr = (p.nblk * 4 + 31) & ~31;
        for (int thr = threadIdx.x; thr < nthr; thr += W * 32) {
            const int blk = thr >> 2;
            const bool in = blk < p.nblk;
            const float4* src = reinterpret_cast<const float4*>(xt) + (size_t)blk * 8 + 2 * t4;
            const float4 a = in ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 b = in ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            const Stage4 st = stage_block4(a, b, t4 >> 1);
            if (in) {
                const uint32_t a0 = xs + xs_chunk_offset(0u, (uint32_t)(2 * t4), (uint32_t)blk, 1u);
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "f"(st.a.x), "f"(st.a.y), "f"(st.a.z),
                             "f"(st.a.w)
                             : "memory");
                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + kXRow * 16u), "f"(st.b.x), "f"(st.b.y),
                             "f"(st.b.z), "f"(st.b.w)
                             : "memory");
                if (t4 == 0)
                    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(aux + aux_offset(0u, (uint32_t)blk, 1u)),
                                 "f"(block_factor(st.e)), "f"(0.0f)
                                 : "memory");
            }
        }
        __syncthreads();
        // each block's -8 offset term: the unit chain on codes of 8 over its staged quads
        for (int b = threadIdx.x; b < p.nblk; b += W * 32) {
            float4 xq[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) xq[q] = lds128f(xs + xs_chunk_offset(0u, (uint32_t)q, (uint32_t)b, 1u));
            const uint32_t a = aux + aux_offset(0u, (uint32_t)b, 1u);
            const float bias = q4_block_bias(xq, lds32f(a));
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(a + 4u), "f"(bias) : "memory");
        }
    }
    __syncthreads();

    // logits of this CTA's experts: warp w takes c + CS*w and c + CS*(w + W), then the next two ...; lane l
    // units l and l + 32, then l + 64 and l + 96, ...; the four (row, unit) loads of a step are issued before
    // any is used
    for (int e0 = c + CS * warp; e0 < p.E; e0 += 2 * CS * W) {
        const int ea = e0, eb = e0 + CS * W;
        const bool hb = eb < p.E;
        float ta = 0.f, tb = 0.f;
        for (int u0 = lane; u0 < p.nblk; u0 += 64) {
            const int u1 = u0 + 32;
            const bool h1 = u1 < p.nblk;
            uint4 w[4];
            uint32_t db[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = (j & 2) ? eb : ea;
                const int u = (j & 1) ? u1 : u0;
                const bool in = ((j & 2) ? hb : true) && ((j & 1) ? h1 : true);
                const size_t blk = (size_t)e * p.nblk + u;
                w[j] = in ? __ldg(reinterpret_cast<const uint4*>(p.qs) + blk) : make_uint4(0u, 0u, 0u, 0u);
                db[j] = in ? (uint32_t)__ldg(p.d + blk) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int u = (j & 1) ? u1 : u0;
                if ((j & 1) && !h1) continue;
                const uint32_t xa = xs + xs_chunk_offset(0u, 0u, (uint32_t)u, 1u);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const Word8s d8 = decode_word_sub(i == 0 ? w[j].x : i == 1 ? w[j].y : i == 2 ? w[j].z : w[j].w);
                    const float4 xl = lds128f(xa + (uint32_t)i * (kXRow * 16u));
                    const float4 xh = lds128f(xa + (uint32_t)(4 + i) * (kXRow * 16u));
                    acc = word_fma(d8, xl, xh, acc);
                }
                const float2 fa = lds64f(aux + aux_offset(0u, (uint32_t)u, 1u));
                const float v = f16_bits_to_f32(db[j]) * fmaf(acc.x + acc.y, fa.x, fa.y);
                if (j & 2) tb += v;
                else ta += v;
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            ta += __shfl_xor_sync(0xffffffffu, ta, off);
            tb += __shfl_xor_sync(0xffffffffu, tb, off);
        }
        if (lane == 0) {
            if (p.logits) p.logits[(size_t)t * p.E + ea] = ta;
            lg[ea] = ta;
            if (hb) {
                if (p.logits) p.logits[(size_t)t * p.E + eb] = tb;
                lg[eb] = tb;
            }
        }
    }
    // every CTA's logits are in its shared memory; CTA 0 gathers them, then the cluster may exit
    cluster_sync();
    if (c == 0) {
        const uint32_t lg_addr = smem_addr(lg);
        for (int e = threadIdx.x; e < p.E; e += W * 32)
            if (e % CS != 0) lg[e] = ld_cluster_f32(lg_addr + 4u * (uint32_t)e, (uint32_t)(e % CS));
    }
    cluster_sync();
    if (c != 0) return;
    __syncthreads();

    // softmax over all E logits and the top K (warp 0 of CTA 0)
    if (warp == 0) {
        float mx = -INFINITY;
        for (int e = lane; e < p.E; e += 32) mx = fmaxf(mx, lg[e]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float z = 0.f;
        for (int e = lane; e < p.E; e += 32) z += expf(lg[e] - mx);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        // The ranking key of expert e: the logit's order-preserving bits (-0 ranks with +0, a NaN below every
        // other value), then the complement of the index, so equal logits go to the lower index.
        auto key_of = [&](int e) {
            const float v = lg[e];
            const uint32_t u = v == 0.0f ? 0u : __float_as_uint(v);
            const uint32_t key = v != v ? 1u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
            return ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)e);
        };
        if (p.E <= 64) {
            // Up to 64 experts: lane l holds experts l and l + 32; each expert's rank is the number of larger keys
            // (all keys differ), and the experts of rank < K are the picks in order. The K weights are summed in
            // pick order, as the passes below do.
            const bool h0 = lane < p.E, h1 = lane + 32 < p.E;
            const unsigned long long k0 = h0 ? key_of(lane) : 0ull, k1 = h1 ? key_of(lane + 32) : 0ull;
            int r0 = 0, r1 = 0;
#pragma unroll 8
            for (int sl = 0; sl < 32; ++sl) {
                const unsigned long long a = __shfl_sync(0xffffffffu, k0, sl), b = __shfl_sync(0xffffffffu, k1, sl);
                r0 += (int)(a > k0) + (int)(b > k0);
                r1 += (int)(a > k1) + (int)(b > k1);
            }
            float* const pk = reinterpret_cast<float*>(smem + p.xs_off);  // the staged input is no longer needed
            const float pw0 = h0 ? expf(lg[lane] - mx) / z : 0.f;
            const float pw1 = h1 ? expf(lg[lane + 32] - mx) / z : 0.f;
            if (h0 && r0 < p.topk) {
                pk[r0] = pw0;
                p.ids[(size_t)t * p.topk + r0] = lane;
            }
            if (h1 && r1 < p.topk) {
                pk[r1] = pw1;
                p.ids[(size_t)t * p.topk + r1] = lane + 32;
            }
            __syncwarp();
            float wsum = 0.f;
            for (int i = 0; i < p.topk; ++i) wsum += pk[i];
            for (int i = lane; i < p.topk; i += 32)
                p.weights[(size_t)t * p.topk + i] = p.normalize ? pk[i] / wsum : pk[i];
            return;
        }
        // K arg-max passes over the untaken experts: lane l holds experts l + 32 j, taken ones marked in
        // tk[j / 32] bit j % 32 (E <= 4096); topk <= E, so a pass always finds an untaken expert
        uint32_t tk[4] = {0u, 0u, 0u, 0u};
        float wsum = 0.f;
        float wsel = 0.f;
        int isel = 0;
        for (int i = 0; i < p.topk; ++i) {
            unsigned long long best = 0ull;
            for (int e = lane, j = 0; e < p.E; e += 32, ++j) {
                if ((tk[j >> 5] >> (j & 31)) & 1u) continue;
                const unsigned long long c = key_of(e);
                best = c > best ? c : best;
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
                best = o > best ? o : best;
            }
            const int bi = best != 0ull ? (int)(0xFFFFFFFFu - (uint32_t)best) : -1;
            const bool found = bi >= 0 && bi < p.E;
            const float pw = found ? expf(lg[bi] - mx) / z : NAN;
            wsum += pw;
            if (lane == i % 32) {  // lane j holds pick j of the current group of 32 picks
                wsel = pw;
                isel = found ? bi : -1;
            }
            if (found && lane == (bi & 31)) tk[(bi >> 5) >> 5] |= 1u << ((bi >> 5) & 31);
            if (i % 32 == 31 || i == p.topk - 1) {
                const int base = i - (i % 32);
                if (lane <= i % 32) {
                    p.ids[(size_t)t * p.topk + base + lane] = isel;
                    p.weights[(size_t)t * p.topk + base + lane] = wsel;  // renormalised below when asked
                }
            }
        }
        if (p.normalize) {
            __syncwarp();
            for (int i = lane; i < p.topk; i += 32) p.weights[(size_t)t * p.topk + i] /= wsum;
        }
    }
}

}  // namespace

cudaError_t launch_moe_router(int32_t* ids, float* weights, float* logits, const uint8_t* qs, const uint16_t* d,
                              const float* x, int T, int E, int K, int topk, bool normalize, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    constexpr int W = 8, CS = 8;
    RouterParams p;
    p.ids = ids;
    p.weights = weights;
    p.logits = logits;
    p.qs = qs;
    p.d = d;
    p.x = x;
    p.T = T;
    p.E = E;
    p.K = K;
    p.nblk = K / 32;
    p.topk = topk;
    p.normalize = normalize ? 1 : 0;
    const uint32_t xsb = xs_chunk_bytes(1u, (uint32_t)p.nblk);
    const uint32_t axb = aux_bytes(1u, (uint32_t)p.nblk);
    p.xs_off = 0;
    p.aux_off = xsb;
    p.lg_off = xsb + axb;
    const uint32_t smem = p.lg_off + (uint32_t)E * 4u;
    if (smem > (uint32_t)di.max_smem_optin) return cudaErrorNotSupported;
    auto kern = moe_router_kernel<W, CS>;
    static std::once_flag attr_once[64];
    std::call_once(attr_once[di.device & 63], [&] {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
    });
    if (e != cudaSuccess) return e;
    // one cluster of CS CTAs per token (CS = 8 is the portable cluster size)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(T * CS));
    cfg.blockDim = dim3((unsigned)(W * 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_overlap() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace q4
