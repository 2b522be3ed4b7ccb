// Planar Q4 batched decode GEMV, 2 to 4 vectors (kernel in q4_dense.cuh): 8 warps x 4 rows per lane, so
// each staged-input load feeds four rows; ring depth 2 beside the staged vectors.
#include "q4_dense.cuh"

namespace q4 {
namespace dense {

cudaError_t gemv_v2_4(const DeviceInfo& di, float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V,
                      int N, int K, cudaStream_t s) {
    switch (V) {
        case 2: return launch<2, 4, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 3: return launch<3, 4, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        case 4: return launch<4, 4, 8, 2, false>(di, Y, qs, d, X, N, K, 2, 4, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dense
}  // namespace q4
