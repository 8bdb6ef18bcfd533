// fp8_linear for callers that cannot allocate device memory.
//
// fp8_linear needs a workspace for the quantized activations and their
// per-token scales.  Some callers have no way to provide one: a plugin
// running inside a host application that owns every device allocation and
// allows no side allocations, or a latency-critical loop where cudaMalloc /
// cudaFree (which can synchronize the device) must not be called.  For them
// this file keeps that scratch in a fixed array that lives inside the library
// itself, so the call needs no workspace argument and allocates nothing.
//
// Cost and limits:
//   * every GPU that loads the library holds FP8_STATIC_SCRATCH_BYTES of
//     device memory for this array until the process exits;
//   * a layer fits when round_up(M*K, 256) + round_up(4*M, 256) <=
//     FP8_STATIC_SCRATCH_BYTES (for example all decode batches of the Llama
//     8B / 70B layers); larger calls are rejected with FP8_ERR_WORKSPACE;
//   * all calls on a device share the one array, which keeps whatever the
//     last call left in it: two calls that overlap on the GPU (for example on
//     two streams at once) race on it and give wrong results.  Nothing in it
//     has to start at zero: the quantizer writes every byte the GEMM reads.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8w8a8.h"
#include "launch.h"

namespace {

static __device__ __align__(256) uint8_t g_static_scratch[FP8_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of the array on the current device.  In host code the
// array's name only stands for it, so the address is looked up once per
// device (with that device current) and cached.
fp8_status_t scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();  // leave no pending error behind
            return FP8_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FP8_OK;
}

}  // namespace

extern "C" fp8_status_t fp8_linear_static_scratch(const void* x_bf16, const uint8_t* wq,
                                                  const float* s_w, void* y_bf16, int64_t M,
                                                  int64_t N, int64_t K, void* stream) {
    // The same argument and device checks as fp8_linear, before anything
    // touches the array: a device the library does not support answers
    // FP8_ERR_UNSUPPORTED here, as it would from fp8_linear.
    fp8_status_t st = fp8k::linear_checks(x_bf16, wq, s_w, y_bf16, M, N, K);
    if (st != FP8_OK || M == 0 || N == 0) return st;
    const size_t need = fp8_linear_workspace_size(M, N, K);
    if (need == 0) return FP8_ERR_INVALID_ARG;
    if (need > static_cast<size_t>(FP8_STATIC_SCRATCH_BYTES)) return FP8_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = scratch_on_current_device(&scratch);
    if (st != FP8_OK) return st;
    return fp8_linear(x_bf16, wq, s_w, y_bf16, M, N, K, scratch, FP8_STATIC_SCRATCH_BYTES,
                      stream);
}
