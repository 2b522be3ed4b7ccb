// Q4_K entry points for sm_103a: the fused RMSNorm + GEMV and gate+up GEMVs and the pure-read instrument run
// the row-per-lane kernel (kernels_q4k_rows.cu); this file holds the bit-exact dequant dump.
//
// Format (trueno-gpu `fused.rs`, FusedRmsNormQ4KGemvKernel phase 3): a row is K/256 super-blocks of 144
// bytes: f16 d, f16 dmin, 12 bytes of packed 6-bit scales/mins, 128 quant bytes. Weight e of a super-block
// lives in chunk c = e/64: low nibbles of the chunk's 32 bytes are sub-block 2c, high nibbles sub-block 2c+1;
// its value is d*sc_j*q - dmin*m_j for its sub-block j.
#include "device_common.cuh"
#include "launch.h"

namespace q4 {

namespace {

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

}  // namespace

cudaError_t launch_q4k_gemv(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x,
                            const float* gamma, float eps, int N, int K, bool swiglu, cudaStream_t s) {
    return launch_q4k_rows_gemv(y0, y1, w0, w1, x, gamma, eps, N, K, swiglu, s);
}

cudaError_t launch_q4k_pure_read(float* sink, const uint8_t* w, int N, int K, cudaStream_t s) {
    return launch_q4k_rows_pure_read(sink, w, N, K, s);
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
