// Device-side building blocks shared by the decode-GEMV kernels (sm_103a).
//
// * Weight streaming: each warp owns a ring of shared-memory slots, filled by asynchronous bulk copies (TMA)
//   that complete on one mbarrier per slot; a warp waits only for its own copies, and every wait is bounded.
// * Nibble -> fp32 (bias-free decode): masking the 4-bit code that sits at bit p of a 32-bit word leaves the
//   float q * 2^(p-149) exactly (a subnormal). The matching input element is staged pre-scaled by
//   2^(127-p-e) (e bounds its 32-element block's exponent), so one packed fp32x2 FMA adds q * x * 2^(-22-e)
//   with one rounding.
// * The FMA chain of a 32-code unit (word_fma) is the one order every planar-format kernel uses, and the
//   format's -8 offset is removed with the same chain run on a unit of code 8 (q4_block_bias), so a block whose
//   codes are all 8 (zero weights) contributes exactly zero. The Q4_K kernels keep their own chains, with the
//   sub-block offsets folded from the same chain run on codes of 1.
// * Input staging (stage_blocks4): four lanes per 32-element block, the block's largest magnitude by two group
//   shuffles, each element scaled by two exact powers of two; a thread stages a batch of blocks together.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace q4 {

// Fault bits recorded by kernels (read back by the host through the ABI).
enum : unsigned {
    kFaultBadExpert = 4u,    // an MoE expert id was outside [0, E)
    kFaultWaitTimeout = 8u,  // a wait for a weight stage ran out of its cycle limit (the warp's later rows are NaN)
    kFaultCopyLost = 16u,    // even the final drain wait for a warp's issued copies ran out (should never happen)
};

// Bound of the drain wait a warp makes before exit for copies it issued but no longer consumes (about two
// seconds of SM clock); the per-stage limit is a kernel parameter (q4_set_wait_limit).
constexpr long long kDrainCycles = 4000000000LL;

// ------------------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Streaming-once policy: the weights are read exactly once per call, so let them leave L2 first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Warp-cooperative async copy global -> shared of `bytes` (a multiple of 16; both addresses 16-byte
// aligned): lane l moves bytes [16 l, 16 l + 16) of every 512-byte stretch.
__device__ __forceinline__ void warp_copy_async(uint32_t dst, const void* src, uint32_t bytes, int lane,
                                                uint64_t policy) {
    const char* s = static_cast<const char*>(src);
    for (uint32_t o = (uint32_t)lane * 16u; o < bytes; o += 512u)
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst + o), "l"(s + o),
                     "l"(policy)
                     : "memory");
}

// Programmatic dependent launch. grid_dependency_wait blocks until the grid that precedes this one in the
// stream has completed and its writes are visible; grid_launch_dependents lets the grid that follows be
// scheduled. Both are no-ops for a grid launched without a programmatic dependency.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// mbarrier with an arrival count and a transaction byte count (asynchronous bulk copies complete on it).
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred P;\n mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n selp.u32 %0, 1, 0, P;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}
// Wait for the completion of phase `parity` of an mbarrier, bounded by `max_cycles`; false if it ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long max_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > max_cycles) return false;
    return true;
}

// The same wait by every lane of a warp, made warp-uniform: true only if every lane saw the phase complete.
// A limit of 0 gives up at once without looking (it exercises the timeout path deterministically).
__device__ __forceinline__ bool warp_wait_bounded(uint32_t bar, uint32_t parity, long long max_cycles) {
    if (max_cycles <= 0) return false;
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, max_cycles)) != 0;
}

// Contiguous global -> shared bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned),
// completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's commit groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds32f(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}


__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// ------------------------------------------------------------------------------------------------
// Nibble decode of one packed 32-bit word
// ------------------------------------------------------------------------------------------------
//
// A 16-byte group holds 32 codes as four words. In word i, byte jj carries a "low" code (low nibble) and
// a "high" code (high nibble). For the Q4 block the low code is element 4i+jj and the high one element
// 16+4i+jj; for a Q4_K half-chunk the low code is element 4i+jj of sub-block 2c and the high one element
// 4i+jj of sub-block 2c+1 (offset by 16*h inside the sub-block). Either way the 8 codes of a word land at
// these bit positions p after the word and a copy shifted right by 12 are masked:
//   low  jj=0..3: p = 0, 8, 16, 12      high jj=0..3: p = 4, 12, 8, 16
//
// ------------------------------------------------------------------------------------------------
// Bias-free nibble decode (subnormal codes) and block-scaled staging
// ------------------------------------------------------------------------------------------------
//
// Masking a code that sits at bit p of a word leaves the float whose bit pattern is q << p, i.e. the exact
// value q * 2^(p-149) (p <= 16, so the pattern stays below 2^23: a subnormal, whose value is the pattern read
// as an integer times 2^-149). So one AND per code gives a float proportional to the unsigned code,
// with no bias to remove. The matching input element is staged as x * 2^(127-p-e), where e bounds the
// exponent of its 32-element block (every |x| of the block < 2^e); then each fp32x2 FMA adds exactly
// q * x * 2^(-22-e) up to one rounding, far from both overflow and the subnormal range. A block's sum
// A = sum q x * 2^(-22-e) is turned back with t = A * 2^(22+e) - 8 * sum(x), which also applies the
// format's -8 offset, and the row accumulates d * t.
// float4 loads each thread issues back to back while staging the input, before it uses any of them.
constexpr int kStageU = 8;

struct Word8s {
    float2 lo01, lo23, hi01, hi23;  // (lo jj0, lo jj1), (lo jj2, lo jj3), (hi jj0, hi jj1), (hi jj2, hi jj3)
};

__device__ __forceinline__ Word8s decode_word_sub(uint32_t w) {
    const uint32_t s = w >> 12;
    Word8s r;
    r.lo01 = make_float2(__uint_as_float(w & 0x0000000Fu), __uint_as_float(w & 0x00000F00u));
    r.lo23 = make_float2(__uint_as_float(w & 0x000F0000u), __uint_as_float(s & 0x0000F000u));
    r.hi01 = make_float2(__uint_as_float(w & 0x000000F0u), __uint_as_float(w & 0x0000F000u));
    r.hi23 = make_float2(__uint_as_float(s & 0x00000F00u), __uint_as_float(s & 0x000F0000u));
    return r;
}

// One 32-bit word of a unit against its staged quads: the low pairs (jj 0,1), (jj 2,3) then the high pairs, each
// one packed FMA into the running (even, odd) pair. Every kernel accumulates a unit's four words in this order
// (word 0 first, starting from zero), so equal codes and inputs give equal sums whatever the kernel.
__device__ __forceinline__ float2 word_fma(const Word8s& d8, float4 xl, float4 xh, float2 a) {
    a = ffma2(d8.lo01, make_float2(xl.x, xl.y), a);
    a = ffma2(d8.lo23, make_float2(xl.z, xl.w), a);
    a = ffma2(d8.hi01, make_float2(xh.x, xh.y), a);
    a = ffma2(d8.hi23, make_float2(xh.z, xh.w), a);
    return a;
}

// The block term of the planar format's -8 offset: -(A8 * 2^(22+e)) with A8 the unit chain of a block whose 32
// codes are all 8, on the block's staged quads xq[8] (quad i: low codes of word i, quad 4+i: high codes) and
// factor f = 2^(22+e). A block is then folded as t = fma(A, f, bias), which is exactly zero when its codes are
// all 8 (A equals A8 bit for bit, and A8 * f is exact), and otherwise equals A * f - 8 * sum(x) up to rounding.
__device__ __forceinline__ float q4_block_bias(const float4 (&xq)[8], float f) {
    const Word8s c8 = decode_word_sub(0x88888888u);
    float2 a = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) a = word_fma(c8, xq[i], xq[4 + i], a);
    return -((a.x + a.y) * f);
}

// (n / d, n % d) for n = n0, n0 + step, n0 + 2 * step, ... (all >= 0, d > 0) with two divisions at the start and
// none per step: the staging loops walk their block indices this way, since a 32-bit division per item costs more
// than the item's own staging arithmetic.
struct DivWalk {
    int q, r;
    int dq, dr, d;
    __device__ __forceinline__ DivWalk(int n0, int step, int d_) : d(d_) {
        q = n0 / d;
        r = n0 - q * d;
        dq = step / d;
        dr = step - dq * d;
    }
    __device__ __forceinline__ void next() {
        q += dq;
        r += dr;
        if (r >= d) {
            r -= d;
            ++q;
        }
    }
};

// 2^k for -126 <= k <= 127.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// Exponent bound e of a block from its largest magnitude m: m < 2^e, clamped to [-100, 128]. Blocks whose
// largest magnitude is below 2^-101 stage with e = -100 (their elements are still represented exactly);
// a non-finite element gives e = 128 and propagates.
__device__ __forceinline__ int block_exponent(float m) {
    const int ef = (int)((__float_as_uint(m) >> 23) & 0xFFu);
    if (ef == 255) return 128;
    return max(ef - 126, -100);
}

// Block factor 2^(22+e); +inf once that passes the float range (blocks with an element of magnitude 2^105
// or more are outside the supported range and yield a non-finite result).
__device__ __forceinline__ float block_factor(int e) { return 22 + e <= 127 ? pow2i(22 + e) : INFINITY; }

// Four lanes stage one 32-element block: lane t of an aligned group of 4 holds float4 2t and 2t+1 (both in
// the same half: elements 8t .. 8t+7). The group's largest magnitude (fixed tree), then every lane scales its
// eight elements with the block's exponent bound e for code positions (hi, jj): the staged value is
// x * 2^(127-p-e), applied as two exact power-of-two factors per position. stage_blocks4 stages NB blocks per
// group at once, in place: each block takes the same operations in the same order as alone, with the steps of the
// NB blocks interleaved so that their group shuffles overlap instead of running one block after another.
template <int NB>
__device__ __forceinline__ void stage_blocks4(float4 (&a)[NB], float4 (&b)[NB], int hi, int (&e)[NB]) {
    float m[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
        m[j] = fmaxf(fmaxf(fmaxf(fabsf(a[j].x), fabsf(a[j].y)), fmaxf(fabsf(a[j].z), fabsf(a[j].w))),
                     fmaxf(fmaxf(fabsf(b[j].x), fabsf(b[j].y)), fmaxf(fabsf(b[j].z), fabsf(b[j].w))));
#pragma unroll
    for (int j = 0; j < NB; ++j) m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], 1));
#pragma unroll
    for (int j = 0; j < NB; ++j) m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], 2));
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        e[j] = block_exponent(m[j]);
        float f1[4], f2[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int p = hi ? (jj == 0 ? 4 : jj == 1 ? 12 : jj == 2 ? 8 : 16) : (jj == 0 ? 0 : jj == 1 ? 8 : jj == 2 ? 16 : 12);
            const int k = 127 - p - e[j];
            const int k1 = k >> 1;
            f1[jj] = pow2i(k1);
            f2[jj] = pow2i(k - k1);
        }
        a[j] = make_float4((a[j].x * f1[0]) * f2[0], (a[j].y * f1[1]) * f2[1], (a[j].z * f1[2]) * f2[2],
                           (a[j].w * f1[3]) * f2[3]);
        b[j] = make_float4((b[j].x * f1[0]) * f2[0], (b[j].y * f1[1]) * f2[1], (b[j].z * f1[2]) * f2[2],
                           (b[j].w * f1[3]) * f2[3]);
    }
}
struct Stage4 {
    int e;        // exponent bound
    float4 a, b;  // the lane's two float4, scaled
};
__device__ __forceinline__ Stage4 stage_block4(float4 a, float4 b, int hi) {
    float4 aa[1] = {a}, bb[1] = {b};
    int e[1];
    stage_blocks4<1>(aa, bb, hi, e);
    Stage4 st;
    st.e = e[0];
    st.a = aa[0];
    st.b = bb[0];
    return st;
}


// Chunk-major staged input: float[ceil(U/32)][V][8 quads][32 unit lanes + 1 pad][4] for V vectors of U units. A
// lane that always works on units u = 32c + lane finds every quad of every vector at one base register plus
// compile-time offsets, and a warp's 32 lanes read 512 consecutive bytes. The 16-byte pad after each quad row
// puts the staging stores of a unit's four lanes (quads 2t and 2t+1) into distinct bank groups.
constexpr uint32_t kXRow = 33;  // float4 per quad row
__host__ __device__ __forceinline__ uint32_t xs_chunk_offset(uint32_t v, uint32_t q, uint32_t u, uint32_t V) {
    return (((u >> 5) * V + v) * 8u + q) * (kXRow * 16u) + (u & 31u) * 16u;
}
__host__ __device__ __forceinline__ uint32_t xs_chunk_bytes(uint32_t V, uint32_t U) {
    return ((U + 31u) / 32u) * V * 8u * kXRow * 16u;
}
// Per-block (2^(22+e), -8 offset term) pairs in the same order: float2[ceil(U/32)][V][32].
__host__ __device__ __forceinline__ uint32_t aux_offset(uint32_t v, uint32_t u, uint32_t V) {
    return ((u >> 5) * V + v) * 256u + (u & 31u) * 8u;
}
__host__ __device__ __forceinline__ uint32_t aux_bytes(uint32_t V, uint32_t U) {
    return ((U + 31u) / 32u) * V * 256u;
}

// ------------------------------------------------------------------------------------------------
// Staged-input layout
// ------------------------------------------------------------------------------------------------
//
// For V input vectors of length K the staged copy is float[V][8][U][4] with U = K/32 sixteen-byte units
// per row. Quad q = half*4 + i of unit u holds the four elements that word i's low (half 0) or high
// (half 1) nibbles multiply, each pre-scaled for its code position (stage_block4). Lanes that work on
// consecutive units read consecutive 16-byte quads, so these loads are free of bank conflicts.
__host__ __device__ __forceinline__ uint32_t xs_index(uint32_t v, uint32_t q, uint32_t u, uint32_t U) {
    return ((v * 8u + q) * U + u) * 4u;
}

// ------------------------------------------------------------------------------------------------
// Warp reductions
// ------------------------------------------------------------------------------------------------

// Sum V (a power of two, <= 32) per-lane values over the warp. Afterwards every lane holds in v[0] the
// total of value index (lane >> (5 - log2 V)).
template <int V>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[V], int lane) {
    static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
    int off = 16;
#pragma unroll
    for (int n = V; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
}

template <int V>
__device__ __forceinline__ constexpr int log2_const() {
    return V <= 1 ? 0 : 1 + log2_const<V / 2>();
}

template <int X>
struct NextPow2 {
    static constexpr int value = X <= 1 ? 1 : X <= 2 ? 2 : X <= 4 ? 4 : X <= 8 ? 8 : X <= 16 ? 16 : 32;
};

// silu(g) = g / (1 + e^-g), the gate of the SwiGLU epilogue.
__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xFFFFu)));
}

}  // namespace q4
