// The C ABI: argument validation (before any CUDA call, so refusals need no GPU), the device check,
// error reporting and dispatch to the kernel families.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/q4gemv.h"
#include "launch.h"

namespace q4 {

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int cuda_fail(const char* what, cudaError_t e) {
    if (e == cudaErrorNotSupported)
        return fail(Q4_EUNSUPPORTED, "%s: the staged input does not fit in shared memory next to the weight rings",
                    what);
    return fail(Q4_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The device check: the library carries sm_103a code only.
int check_device(const char* what, DeviceInfo* di) {
    cudaError_t e = current_device_info(di);
    if (e != cudaSuccess) return cuda_fail(what, e);
    if (di->major != 10 || di->minor != 3)
        return fail(Q4_EUNSUPPORTED, "%s: device is sm_%d%d, this library is built for sm_103a", what, di->major,
                    di->minor);
    return Q4_OK;
}

int check_eps(const char* what, float eps) {
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return fail(Q4_EINVAL, "%s: eps must be finite and >= 0", what);
    return Q4_OK;
}

int check_q4_weights(const char* what, const uint8_t* qs, const uint16_t* d, int N, int K) {
    if (!qs || !d) return fail(Q4_EINVAL, "%s: null weight pointer", what);
    if (N <= 0) return fail(Q4_EINVAL, "%s: N must be >= 1 (got %d)", what, N);
    if (K <= 0 || K % 32 != 0) return fail(Q4_EINVAL, "%s: K must be a positive multiple of 32 (got %d)", what, K);
    if (!aligned(qs, 16)) return fail(Q4_EALIGN, "%s: qs must be 16-byte aligned", what);
    if (!aligned(d, 2)) return fail(Q4_EALIGN, "%s: d must be 2-byte aligned", what);
    return Q4_OK;
}

int check_q4k_weights(const char* what, const uint8_t* w, int N, int K) {
    if (!w) return fail(Q4_EINVAL, "%s: null weight pointer", what);
    if (N <= 0) return fail(Q4_EINVAL, "%s: N must be >= 1 (got %d)", what, N);
    if (K <= 0 || K % 256 != 0) return fail(Q4_EINVAL, "%s: K must be a positive multiple of 256 (got %d)", what, K);
    if (!aligned(w, 16)) return fail(Q4_EALIGN, "%s: weights must be 16-byte aligned", what);
    return Q4_OK;
}

int check_out(const char* what, const float* y, uintptr_t a = 4) {
    if (!y) return fail(Q4_EINVAL, "%s: null output pointer", what);
    if (!aligned(y, a)) return fail(Q4_EALIGN, "%s: output must be %d-byte aligned", what, (int)a);
    return Q4_OK;
}

int check_vec(const char* what, const char* name, const float* v) {
    if (!v) return fail(Q4_EINVAL, "%s: null %s", what, name);
    if (!aligned(v, 16)) return fail(Q4_EALIGN, "%s: %s must be 16-byte aligned", what, name);
    return Q4_OK;
}

#define Q4_TRY(expr)            \
    do {                        \
        int rc_ = (expr);       \
        if (rc_ != Q4_OK) return rc_; \
    } while (0)

int finish(const char* what, cudaError_t e) {
    if (e != cudaSuccess) return cuda_fail(what, e);
    g_last_error.clear();
    return Q4_OK;
}

}  // namespace

namespace {
std::atomic<int> g_launch_overlap{0};
std::atomic<long long> g_wait_limit{4000000000LL};
}  // namespace

bool launch_overlap() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }

long long wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

// The fault word every kernel family ORs its kFault* bits into (one per device that loads the library).
static __device__ unsigned g_faults;

unsigned* device_fault_word(int device) {
    static unsigned* ptrs[64] = {};
    static std::mutex mu;
    if (device < 0 || device >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[device]) {
        unsigned* p = nullptr;
        if (cudaGetSymbolAddress((void**)&p, g_faults) != cudaSuccess) return nullptr;
        ptrs[device] = p;
    }
    return ptrs[device];
}

static cudaError_t read_and_clear_faults(unsigned* out) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_faults, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_faults, &zero, sizeof(unsigned));
    return e;
}

cudaError_t current_device_info(DeviceInfo* out) {
    static DeviceInfo cache[64];
    static std::mutex mu;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].device != dev) {
        DeviceInfo di;
        di.device = dev;
        if ((e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
        cache[dev] = di;
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace q4

using namespace q4;

extern "C" {

int q4_gemv(float* y, const uint8_t* qs, const uint16_t* d, const float* x, int N, int K, q4_stream_t stream) {
    const char* what = "q4_gemv";
    Q4_TRY(check_out(what, y));
    Q4_TRY(check_q4_weights(what, qs, d, N, K));
    Q4_TRY(check_vec(what, "x", x));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4_gemv(y, qs, d, x, 1, N, K, (cudaStream_t)stream));
}

int q4_gemv_batched(float* Y, const uint8_t* qs, const uint16_t* d, const float* X, int M, int N, int K,
                    q4_stream_t stream) {
    const char* what = "q4_gemv_batched";
    Q4_TRY(check_out(what, Y));
    Q4_TRY(check_q4_weights(what, qs, d, N, K));
    Q4_TRY(check_vec(what, "X", X));
    if (M < 1 || M > 16) return fail(Q4_EINVAL, "%s: M=%d outside 1..16 (refused, not clamped)", what, M);
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4_gemv(Y, qs, d, X, M, N, K, (cudaStream_t)stream));
}

int fused_rmsnorm_q4k_gemv(float* y, const uint8_t* w, const float* x, const float* gamma, float eps, int N, int K,
                           q4_stream_t stream) {
    const char* what = "fused_rmsnorm_q4k_gemv";
    Q4_TRY(check_out(what, y));
    Q4_TRY(check_q4k_weights(what, w, N, K));
    Q4_TRY(check_vec(what, "x", x));
    Q4_TRY(check_vec(what, "gamma", gamma));
    Q4_TRY(check_eps(what, eps));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4k_gemv(y, nullptr, w, nullptr, x, gamma, eps, N, K, false, (cudaStream_t)stream));
}

int q4k_gemv_batched(float* Y, const uint8_t* w, const float* X, int M, int N, int K, q4_stream_t stream) {
    const char* what = "q4k_gemv_batched";
    Q4_TRY(check_out(what, Y));
    Q4_TRY(check_q4k_weights(what, w, N, K));
    Q4_TRY(check_vec(what, "X", X));
    if (M < 1 || M > 8) return fail(Q4_EINVAL, "%s: M=%d outside 1..8 (refused, not clamped)", what, M);
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4k_gemv_batched(Y, w, X, M, N, K, (cudaStream_t)stream));
}

int fused_gateup_q4k_gemv(float* y_gate, float* y_up, const uint8_t* w_gate, const uint8_t* w_up, const float* x,
                          const float* gamma, float eps, int N, int K, q4_stream_t stream) {
    const char* what = "fused_gateup_q4k_gemv";
    Q4_TRY(check_out(what, y_gate));
    Q4_TRY(check_out(what, y_up));
    Q4_TRY(check_q4k_weights(what, w_gate, N, K));
    Q4_TRY(check_q4k_weights(what, w_up, N, K));
    Q4_TRY(check_vec(what, "x", x));
    if (gamma) Q4_TRY(check_vec(what, "gamma", gamma));
    Q4_TRY(check_eps(what, eps));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4k_gemv(y_gate, y_up, w_gate, w_up, x, gamma, eps, N, K, false, (cudaStream_t)stream));
}

static int check_moe(const char* what, const float* y_gate, const float* y_up, const uint8_t* qs_gate,
                     const uint16_t* d_gate, const uint8_t* qs_up, const uint16_t* d_up, const int32_t* ids, int T,
                     int topk, int E, int N, int K) {
    Q4_TRY(check_out(what, y_gate));
    Q4_TRY(check_out(what, y_up));
    if (E <= 0) return fail(Q4_EINVAL, "%s: E must be >= 1 (got %d)", what, E);
    if ((long long)E * N > 0x7fffffffLL) return fail(Q4_EINVAL, "%s: E*N exceeds 2^31-1 rows", what);
    Q4_TRY(check_q4_weights(what, qs_gate, d_gate, N, K));
    Q4_TRY(check_q4_weights(what, qs_up, d_up, N, K));
    if (!ids) return fail(Q4_EINVAL, "%s: null expert_ids", what);
    if (!aligned(ids, 4)) return fail(Q4_EALIGN, "%s: expert_ids must be 4-byte aligned", what);
    if (T <= 0 || topk <= 0) return fail(Q4_EINVAL, "%s: T and topk must be >= 1", what);
    if (topk > E) return fail(Q4_EINVAL, "%s: topk=%d exceeds E=%d", what, topk, E);
    if ((long long)T * topk > 512) return fail(Q4_EINVAL, "%s: T*topk=%lld exceeds 512", what, (long long)T * topk);
    return Q4_OK;
}

int moe_q4_gemv(float* y_gate, float* y_up, const uint8_t* qs_gate, const uint16_t* d_gate, const uint8_t* qs_up,
                const uint16_t* d_up, const float* x, const int32_t* expert_ids, int T, int topk, int E, int N, int K,
                int32_t* dev_status, q4_stream_t stream) {
    const char* what = "moe_q4_gemv";
    Q4_TRY(check_moe(what, y_gate, y_up, qs_gate, d_gate, qs_up, d_up, expert_ids, T, topk, E, N, K));
    Q4_TRY(check_vec(what, "x", x));
    if (dev_status && !aligned(dev_status, 4)) return fail(Q4_EALIGN, "%s: dev_status must be 4-byte aligned", what);
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_moe_q4_gemv(y_gate, y_up, qs_gate, d_gate, qs_up, d_up, x, expert_ids, T, topk, E, N,
                                           K, dev_status, false, false, (cudaStream_t)stream));
}

int fused_gateup_swiglu_q4k_gemv(float* y, const uint8_t* w_gate, const uint8_t* w_up, const float* x,
                                 const float* gamma, float eps, int N, int K, q4_stream_t stream) {
    const char* what = "fused_gateup_swiglu_q4k_gemv";
    Q4_TRY(check_out(what, y));
    Q4_TRY(check_q4k_weights(what, w_gate, N, K));
    Q4_TRY(check_q4k_weights(what, w_up, N, K));
    Q4_TRY(check_vec(what, "x", x));
    if (gamma) Q4_TRY(check_vec(what, "gamma", gamma));
    Q4_TRY(check_eps(what, eps));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4k_gemv(y, nullptr, w_gate, w_up, x, gamma, eps, N, K, true, (cudaStream_t)stream));
}

int moe_q4_swiglu_gemv(float* y, const uint8_t* qs_gate, const uint16_t* d_gate, const uint8_t* qs_up,
                       const uint16_t* d_up, const float* x, const int32_t* expert_ids, int T, int topk, int E, int N,
                       int K, int32_t* dev_status, q4_stream_t stream) {
    const char* what = "moe_q4_swiglu_gemv";
    Q4_TRY(check_moe(what, y, y, qs_gate, d_gate, qs_up, d_up, expert_ids, T, topk, E, N, K));
    Q4_TRY(check_vec(what, "x", x));
    if (dev_status && !aligned(dev_status, 4)) return fail(Q4_EALIGN, "%s: dev_status must be 4-byte aligned", what);
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_moe_q4_gemv(y, nullptr, qs_gate, d_gate, qs_up, d_up, x, expert_ids, T, topk, E, N, K,
                                           dev_status, false, true, (cudaStream_t)stream));
}

int moe_router_q4(int32_t* expert_ids, float* expert_weights, float* logits, const uint8_t* qs, const uint16_t* d,
                  const float* x, int T, int E, int K, int topk, int normalize, q4_stream_t stream) {
    const char* what = "moe_router_q4";
    if (!expert_ids || !expert_weights) return fail(Q4_EINVAL, "%s: null output pointer", what);
    if (!aligned(expert_ids, 4) || !aligned(expert_weights, 4) || (logits && !aligned(logits, 4)))
        return fail(Q4_EALIGN, "%s: outputs must be 4-byte aligned", what);
    if (E <= 0 || E > 4096) return fail(Q4_EINVAL, "%s: E must be in 1..4096 (got %d)", what, E);
    Q4_TRY(check_q4_weights(what, qs, d, E, K));
    Q4_TRY(check_vec(what, "x", x));
    if (T <= 0) return fail(Q4_EINVAL, "%s: T must be >= 1 (got %d)", what, T);
    if (topk <= 0 || topk > E) return fail(Q4_EINVAL, "%s: topk must be in 1..E (got %d, E=%d)", what, topk, E);
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_moe_router(expert_ids, expert_weights, logits, qs, d, x, T, E, K, topk, normalize != 0,
                                          (cudaStream_t)stream));
}

int q4_pure_read(float* sink, const uint8_t* qs, const uint16_t* d, int N, int K, q4_stream_t stream) {
    const char* what = "q4_pure_read";
    Q4_TRY(check_out(what, sink));
    Q4_TRY(check_q4_weights(what, qs, d, N, K));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4_pure_read(sink, qs, d, N, K, (cudaStream_t)stream));
}

int q4k_pure_read(float* sink, const uint8_t* w, int N, int K, q4_stream_t stream) {
    const char* what = "q4k_pure_read";
    Q4_TRY(check_out(what, sink));
    Q4_TRY(check_q4k_weights(what, w, N, K));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4k_pure_read(sink, w, N, K, (cudaStream_t)stream));
}

int moe_q4_pure_read(float* sink_gate, float* sink_up, const uint8_t* qs_gate, const uint16_t* d_gate,
                     const uint8_t* qs_up, const uint16_t* d_up, const int32_t* expert_ids, int T, int topk, int E,
                     int N, int K, int32_t* dev_status, q4_stream_t stream) {
    const char* what = "moe_q4_pure_read";
    Q4_TRY(check_moe(what, sink_gate, sink_up, qs_gate, d_gate, qs_up, d_up, expert_ids, T, topk, E, N, K));
    if (dev_status && !aligned(dev_status, 4)) return fail(Q4_EALIGN, "%s: dev_status must be 4-byte aligned", what);
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_moe_q4_gemv(sink_gate, sink_up, qs_gate, d_gate, qs_up, d_up, nullptr, expert_ids, T,
                                           topk, E, N, K, dev_status, true, false, (cudaStream_t)stream));
}

int q4_fma_ceiling(float* sink, int sink_len, long long fmas, float mul, float add, long long* fmas_done,
                   q4_stream_t stream) {
    const char* what = "q4_fma_ceiling";
    Q4_TRY(check_out(what, sink));
    if (fmas <= 0) return fail(Q4_EINVAL, "%s: fmas must be >= 1 (got %lld)", what, fmas);
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    if (sink_len < di.sm_count)
        return fail(Q4_EINVAL, "%s: sink holds %d floats, the launch writes one per SM (%d)", what, sink_len,
                    di.sm_count);
    const long long per = fma_ceiling_fmas_per_iter(di.sm_count);
    const long long iters = (fmas + per - 1) / per;
    if (fmas_done) *fmas_done = iters * per;
    return finish(what, launch_fma_ceiling(sink, iters, mul, add, di.sm_count, (cudaStream_t)stream));
}

int q4_dequant(float* W, const uint8_t* qs, const uint16_t* d, int N, int K, q4_stream_t stream) {
    const char* what = "q4_dequant";
    Q4_TRY(check_out(what, W, 16));
    Q4_TRY(check_q4_weights(what, qs, d, N, K));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4_dequant(W, qs, d, N, K, (cudaStream_t)stream));
}

int q4k_dequant(float* W, const uint8_t* w, int N, int K, q4_stream_t stream) {
    const char* what = "q4k_dequant";
    Q4_TRY(check_out(what, W, 16));
    Q4_TRY(check_q4k_weights(what, w, N, K));
    DeviceInfo di;
    Q4_TRY(check_device(what, &di));
    return finish(what, launch_q4k_dequant(W, w, N, K, (cudaStream_t)stream));
}

const char* q4_last_error(void) { return g_last_error.c_str(); }

int q4_set_launch_overlap(int enable) {
    g_launch_overlap.store(enable ? 1 : 0, std::memory_order_relaxed);
    return Q4_OK;
}

int q4_get_launch_overlap(void) { return g_launch_overlap.load(std::memory_order_relaxed); }

int q4_device_faults(unsigned* faults) {
    const char* what = "q4_device_faults";
    if (!faults) return fail(Q4_EINVAL, "%s: null output pointer", what);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(what, e);
    unsigned f = 0;
    if ((e = read_and_clear_faults(&f)) != cudaSuccess) return cuda_fail(what, e);
    *faults |= f;
    return finish(what, cudaSuccess);
}

int q4_set_wait_limit(long long cycles) {
    if (cycles < 0) return fail(Q4_EINVAL, "q4_set_wait_limit: the limit must be >= 0 (got %lld)", cycles);
    g_wait_limit.store(cycles, std::memory_order_relaxed);
    g_last_error.clear();
    return Q4_OK;
}

long long q4_get_wait_limit(void) { return g_wait_limit.load(std::memory_order_relaxed); }

}  // extern "C"
