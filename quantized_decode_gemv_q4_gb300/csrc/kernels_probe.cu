// FMA-ceiling instrument: the fp32 FMA work of a GEMV call with no loads at all, so that a call whose
// arithmetic may bind (the batched forms at M = 8 and up: 8 FMAs per weight) can be placed against the FMA
// roof as well as the HBM one. One persistent CTA of 512 threads per SM; every thread runs eight independent
// chains of packed fp32x2 FMAs (a <- a * mul + add), enough chains per scheduler to keep the FMA pipe issuing
// every cycle; the chains' end values are summed per CTA in a fixed order into the sink, so nothing is
// optimised away.
#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

constexpr int kProbeThreads = 512;
constexpr int kChains = 8;

__global__ void __launch_bounds__(kProbeThreads, 1) fma_ceiling_kernel(float* sink, long long iters, float2 mul,
                                                                         float2 add) {
    float2 a[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j)
        a[j] = make_float2((float)((int)(threadIdx.x % 7u) + j), (float)((int)(threadIdx.x % 5u) + j));
#pragma unroll 4
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) a[j] = ffma2(a[j], mul, add);
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += a[j].x + a[j].y;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    __shared__ float part[kProbeThreads / 32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < kProbeThreads / 32; ++w) t += part[w];
        sink[blockIdx.x] = t;
    }
}

}  // namespace

long long fma_ceiling_fmas_per_iter(int sm_count) { return (long long)sm_count * kProbeThreads * kChains * 2; }

cudaError_t launch_fma_ceiling(float* sink, long long iters, float mul, float add, int sm_count, cudaStream_t s) {
    fma_ceiling_kernel<<<sm_count, kProbeThreads, 0, s>>>(sink, iters, make_float2(mul, mul), make_float2(add, add));
    return cudaGetLastError();
}

}  // namespace q4
