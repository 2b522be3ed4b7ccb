// Internal host-side interface between the C ABI (abi.cu) and the kernel translation units.
// Arguments reaching these functions have already been validated by the ABI layer.
#pragma once

#include <cuda.h>  // tensor-map types (the encoder is reached through the runtime's driver entry point)
#include <cuda_runtime.h>
#include <stdint.h>

namespace q4 {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;  // bytes of dynamic shared memory a CTA may opt into
    int major = 0, minor = 0;
};

// Cached per-device properties of the current device (thread-safe after first call).
cudaError_t current_device_info(DeviceInfo* out);

// Process-wide launch-overlap setting (programmatic dependent launch), set through the C ABI.
bool launch_overlap();

// Process-wide limit, in SM cycles, of one kernel wait for a weight stage (q4_set_wait_limit); default 4e9.
long long wait_limit_cycles();

// Device address of the fault word of `device` (the current device), which kernels OR kFault* bits into; nullptr
// when it cannot be resolved. The word is read and cleared by q4_device_faults.
unsigned* device_fault_word(int device);

// A 2-D tensor map of a byte matrix [rows][row_bytes] (row_bytes a multiple of 16, base 16-byte aligned), box
// box_bytes x box_rows, rows past the end read as zero; swizzle128 selects the 128-byte swizzle (box_bytes must
// then be 128, and the shared-memory destination 1024-byte aligned). Maps are cached per (base, shape, box,
// swizzle), since encoding one costs host time. False when the driver's encoder is unavailable or refuses.
bool cached_tensor_map_2d(CUtensorMap* out, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                          uint32_t box_rows, bool swizzle128);

// Launch a GEMV kernel; with launch overlap on, it may start while the previous kernel in the stream is
// still running (the kernel waits for it before touching inputs or outputs, see grid_dependency_wait).
template <typename Kernel, typename Params>
cudaError_t launch_kernel(Kernel kern, int grid, int block, uint32_t smem, cudaStream_t s, const Params& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = launch_overlap() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// ---- planar Q4 (32-weight blocks, f16 scale per block) -------------------------------------------
// Y[v][n] = sum_k W[n][k] * X[v][k] for v < V; V in 1..16. Returns cudaErrorNotSupported when the
// staged input does not fit in shared memory.
cudaError_t launch_q4_gemv(float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int V, int N, int K,
                           cudaStream_t s);
// Same bytes, same addressing, no math: sink[n] = XOR of row n's quant words and (zero-extended) scales.
cudaError_t launch_q4_pure_read(float* sink, const uint8_t* qs, const uint16_t* d, int N, int K, cudaStream_t s);
// FMA-ceiling instrument (kernels_probe.cu): `iters` rounds of 16 fp32 FMAs per thread on one 512-thread CTA per
// SM; fma_ceiling_fmas_per_iter(sm_count) FMAs per round in all.
long long fma_ceiling_fmas_per_iter(int sm_count);
cudaError_t launch_fma_ceiling(float* sink, long long iters, float mul, float add, int sm_count, cudaStream_t s);
cudaError_t launch_q4_dequant(float* W, const uint8_t* qs, const uint16_t* d, int N, int K, cudaStream_t s);

// ---- Q4_K (144-byte super-blocks of 256 weights) ------------------------------------------------------
// One or two weight streams against one input; gamma == nullptr skips RMSNorm. With swiglu (two streams)
// y0 = silu(W0 xhat) * (W1 xhat) and y1 is not written.
cudaError_t launch_q4k_gemv(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x,
                            const float* gamma, float eps, int N, int K, bool swiglu, cudaStream_t s);
// Row-per-lane forms of launch_q4k_gemv and launch_q4k_pure_read (kernels_q4k_rows.cu).
cudaError_t launch_q4k_rows_gemv(float* y0, float* y1, const uint8_t* w0, const uint8_t* w1, const float* x,
                                 const float* gamma, float eps, int N, int K, bool swiglu, cudaStream_t s);
cudaError_t launch_q4k_rows_pure_read(float* sink, const uint8_t* w, int N, int K, cudaStream_t s);
// Y[v][n] = sum_k W[n][k] * X[v][k], V in 1..8, no normalisation.
cudaError_t launch_q4k_gemv_batched(float* Y, const uint8_t* w, const float* X, int V, int N, int K, cudaStream_t s);
cudaError_t launch_q4k_pure_read(float* sink, const uint8_t* w, int N, int K, cudaStream_t s);
cudaError_t launch_q4k_dequant(float* W, const uint8_t* w, int N, int K, cudaStream_t s);

// ---- MoE expert-gathered planar Q4 gate+up ---------------------------------------------------------
// swiglu: y_gate = silu(gate) * up per routed row, y_up unused.
cudaError_t launch_moe_q4_gemv(float* y_gate, float* y_up, const uint8_t* qs_gate, const uint16_t* d_gate,
                               const uint8_t* qs_up, const uint16_t* d_up, const float* x, const int32_t* ids,
                               int T, int topk, int E, int N, int K, int32_t* dev_status, bool pure_read,
                               bool swiglu, cudaStream_t s);

// ---- MoE router: gate GEMV over E planar-Q4 rows + top-K softmax per token ---------------------------
cudaError_t launch_moe_router(int32_t* ids, float* weights, float* logits, const uint8_t* qs, const uint16_t* d,
                              const float* x, int T, int E, int K, int topk, bool normalize, cudaStream_t s);


}  // namespace q4
