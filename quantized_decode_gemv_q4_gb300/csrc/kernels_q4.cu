// Planar Q4 decode GEMV for sm_103a: the single-vector launch plans, the dispatch over batch widths, the
// pure-read ceiling instrument and the bit-exact dequant dump. The kernel itself is in q4_dense.cuh.
#include <cstdio>
#include <cstdlib>

#include "q4_dense.cuh"

namespace q4 {
namespace dense {

// One vector: 16 warps x 2 rows per lane, whole rows per stage up to K = 4096 (4 units per lane; longer rows in
// 128-block chunks), ring depth 2 (3 on request through Q4GEMV_Q4_DEPTH). Measured slower at 14336x4096:
// 16 warps x 1 row, 24 warps x 1 row, 10-14 warps x 2 rows, 8 warps x 4 rows with the input in registers,
// two accumulation chains per row, rings of depth 3 to 8.
cudaError_t gemv_v1(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int N,
                    int K, cudaStream_t s) {
    return launch<1, 2, 16, 3, false>(di, Y, qs, d, X, N, K, 2, 4, s);
}

}  // namespace dense

cudaError_t launch_q4_gemv(float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V, int N, int K,
                           cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    if (V == 1) return dense::gemv_v1(di, Y, qs, d, X, N, K, s);
    if (V >= 2 && V <= 4) return dense::gemv_v2_4(di, Y, qs, d, X, V, N, K, s);
    if (V >= 5 && V <= 8) return dense::gemv_v5_8(di, Y, qs, d, X, V, N, K, s);
    if (V >= 9 && V <= 16) return dense::gemv_v9_16(di, Y, qs, d, X, V, N, K, s);
    return cudaErrorInvalidValue;
}

// The same streaming as the single-vector plan (16 warps x 2 rows, whole rows per stage, ring depth 2), no
// math.
cudaError_t launch_q4_pure_read(float* sink, const uint8_t* qs, const uint16_t* d, int N, int K, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    return dense::launch<1, 2, 16, 3, true>(di, sink, qs, d, nullptr, N, K, 2, 4, s);
}

namespace {

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

}  // namespace

cudaError_t launch_q4_dequant(float* W, const uint8_t* qs, const uint16_t* d, int N, int K, cudaStream_t s) {
    const long long nunits = (long long)N * (K / 32);
    const int threads = 256;
    const long long blocks = (nunits + threads - 1) / threads;
    q4_dequant_kernel<<<(unsigned)blocks, threads, 0, s>>>(W, qs, d, nunits);
    return cudaGetLastError();
}

}  // namespace q4
