// Planar Q4 batched decode GEMV, 9 to 16 vectors (kernel in q4_dense.cuh): 8 warps x 2 rows per lane, ring
// depth 2. The 9..16 staged vectors must fit in shared memory beside the rings (M*K*4 bytes: K <= 2048 at
// M = 16); larger inputs are refused as unsupported rather than streamed twice.
#include "q4_dense.cuh"

namespace q4 {
namespace dense {

cudaError_t gemv_v9_16(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V,
                       int N, int K, cudaStream_t s) {
    switch (V) {
        case 9: return launch<9, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 10: return launch<10, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 11: return launch<11, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 12: return launch<12, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 13: return launch<13, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 14: return launch<14, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 15: return launch<15, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 16: return launch<16, 2, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dense
}  // namespace q4
