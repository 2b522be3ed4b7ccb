// Planar Q4 batched decode GEMV, 5 to 8 vectors (kernel in q4_dense.cuh): 12 warps x 3 rows per lane, ring
// depth 2; with the staged vectors taking up to 132 KB, the rows stream in 64-block chunks when whole
// 128-block rows do not fit.
#include "q4_dense.cuh"

namespace q4 {
namespace dense {

cudaError_t gemv_v5_8(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V,
                      int N, int K, cudaStream_t s) {
    switch (V) {
        case 5: return launch<5, 3, 12, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 6: return launch<6, 3, 12, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 7: return launch<7, 3, 12, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 8: return launch<8, 3, 12, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dense
}  // namespace q4
