// Planar Q4 decode GEMV for sm_103a: the single-vector launch plans, the dispatch over batch widths, the
// pure-read ceiling instrument and the bit-exact dequant dump. The kernels are in q4_xr.cuh (one vector, input
// in registers) and q4_dense.cuh (the general and batched kernel).
#include <cstdio>
#include <cstdlib>

#include "q4_dense.cuh"
#include "q4_xr.cuh"

namespace q4 {
namespace dense {

// The register-input plan for one vector: 8 warps x 4 rows per job, ring depth 2 (one stage requested before the
// dependency wait), for K/32 a multiple of 8 up to 128 blocks with 16-byte aligned scales. Measured on the
// 14336x4096 workload against 3 rows at depth 3, 5 rows, 2 rows at depth 4, 6 to 12 warps and the shared-memory
// input plan (16 warps x 2 rows); requesting the whole ring before the wait was slower (the copies delay the
// input's staging and the release of the dependent launch).
template <bool PURE>
cudaError_t launch_xr_plan(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X,
                           int N, int K, cudaStream_t s) {
    const int nblk = K / 32;
    if (nblk > 96) return xr::launch_xr<4, 8, 2, 4, 1, PURE>(di, Y, qs, d, X, N, K, s);
    if (nblk > 64) return xr::launch_xr<4, 8, 2, 3, 1, PURE>(di, Y, qs, d, X, N, K, s);
    if (nblk > 32) return xr::launch_xr<4, 8, 2, 2, 1, PURE>(di, Y, qs, d, X, N, K, s);
    return xr::launch_xr<4, 8, 2, 1, 1, PURE>(di, Y, qs, d, X, N, K, s);
}

// One vector: the register-input plan where it applies, else 16 warps x 2 rows per lane, whole rows per stage
// up to K = 4096 (longer rows in 128-block chunks), ring depth 2.
cudaError_t gemv_v1(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int N,
                    int K, cudaStream_t s) {
    cudaError_t e = launch_xr_plan<false>(di, Y, qs, d, X, N, K, s);
    if (e != cudaErrorNotSupported) return e;
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

// The same streaming as the single-vector plan (the register-input plan where it applies, else 16 warps x 2
// rows, whole rows per stage, ring depth 2), no math.
cudaError_t launch_q4_pure_read(float* sink, const uint8_t* qs, const uint16_t* d, int N, int K, cudaStream_t s) {
    DeviceInfo di;
    cudaError_t e = current_device_info(&di);
    if (e != cudaSuccess) return e;
    e = dense::launch_xr_plan<true>(di, sink, qs, d, nullptr, N, K, s);
    if (e != cudaErrorNotSupported) return e;
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
