// C-ABI entry points of the FP8_DYNAMIC W8A8 linear layer (fp8w8a8.h).
//
// This file only validates arguments on the host, keeps a little per-device
// state (SM count, the device status word, kernel attributes) and launches
// the kernels of quant.cu, quant_variants.cu, norm_quant.cu, gemm_pair.cu,
// gemm_decode.cu and gemm_blockwise.cu.  It never
// allocates device memory and never synchronizes, except in
// fp8_device_status().
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8w8a8.h"
#include "launch.h"

namespace {

// Device status word: kernels OR error bits into it (bounded waits that ran
// out).  One copy per device, located with cudaGetSymbolAddress.
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    fp8_status_t verdict = FP8_ERR_UNSUPPORTED;
    int num_sms = 0;
    int pair_clusters = 0;  // co-resident clusters of the paired-SM GEMM
    // co-resident clusters of S decode-GEMM CTAs (S = 1..8) at the footprint
    // of c = 1..3 CTAs per SM: [(c - 1) * 9 + S]
    int decode_clusters[27] = {};
    unsigned* status = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Per-device setup on first use: capability check (10.3 = GB300), SM count,
// status word address, dynamic shared memory limits of the GEMM kernels.
fp8_status_t current_device(DeviceState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8_ERR_CUDA;
        if (major != 10 || minor != 3) {
            d.verdict = FP8_ERR_UNSUPPORTED;
        } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word) !=
                       cudaSuccess ||
                   fp8k::prepare_gemm_decode() != cudaSuccess ||
                   fp8k::prepare_gemm_blockwise() != cudaSuccess ||
                   fp8k::prepare_gemm_pair() != cudaSuccess) {
            d.verdict = FP8_ERR_CUDA;
        } else {
            d.pair_clusters = fp8k::gemm_pair_resident_clusters(d.num_sms);
            for (int per_sm = 1; per_sm <= 3; ++per_sm)
                for (int c = 1; c <= 8; ++c)
                    d.decode_clusters[(per_sm - 1) * 9 + c] =
                        fp8k::gemm_decode_resident_clusters(c, per_sm);
            d.verdict = FP8_OK;
        }
        d.ready = true;
    }
    *out = &d;
    return d.verdict;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Validation shared by the two quantizing entry points.
fp8_status_t check_quant(const void* x, int64_t R, int64_t K, int64_t ldx, const uint8_t* q,
                         int64_t ldq, const float* s) {
    if (R < 0 || K < 0 || R > kMaxDim || K > kMaxDim) return FP8_ERR_INVALID_ARG;
    if (R == 0) return FP8_OK;
    if (!s || (K > 0 && (!x || !q))) return FP8_ERR_INVALID_ARG;
    if (K > 0 && (ldx < K || ldq < K)) return FP8_ERR_INVALID_ARG;
    if (K % 16 != 0) return FP8_ERR_UNSUPPORTED;
    if (K > 0 && (ldx % 8 != 0 || ldq % 16 != 0 || !aligned(x, 16) || !aligned(q, 16)))
        return FP8_ERR_UNSUPPORTED;
    if (!aligned(s, 4)) return FP8_ERR_UNSUPPORTED;
    return FP8_OK;
}

fp8_status_t quant_rows(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                        float* s, void* stream) {
    fp8_status_t st = check_quant(x, R, K, ldx, q, ldq, s);
    if (st != FP8_OK || R == 0) return st;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_quant_rows(x, R, K, ldx, q, ldq, s,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t check_gemm(const uint8_t* xq, const float* s_tok, const uint8_t* wq, const float* s_w,
                        const void* y, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (!xq || !s_tok || !wq || !s_w || !y) return FP8_ERR_INVALID_ARG;
    if (K <= 0 || K % 16 != 0) return FP8_ERR_UNSUPPORTED;
    if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(s_tok, 4) ||
        !aligned(s_w, 4))
        return FP8_ERR_UNSUPPORTED;
    return FP8_OK;
}

fp8_status_t run_gemm(const uint8_t* xq, const float* s_tok, const uint8_t* wq, const float* s_w,
                      void* y, int64_t M, int64_t N, int64_t K, void* stream, DeviceState* d,
                      bool blockwise = false) {
    fp8k::GemmArgs a;
    a.xq = xq;
    a.s_tok = s_tok;
    a.wq = wq;
    a.s_w = s_w;
    a.y = y;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.status = d->status;
    a.num_sms = d->num_sms;
    a.pdl = true;
    a.pair_clusters = d->pair_clusters;
    a.decode_clusters = d->decode_clusters;
    a.stream = static_cast<cudaStream_t>(stream);
    cudaError_t e = blockwise                 ? fp8k::launch_gemm_blockwise(a)
                    : M <= fp8k::kDecodeMaxM ? fp8k::launch_gemm_decode(a)
                                             : fp8k::launch_gemm_pair(a);
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

constexpr int64_t kScaleBlock = 128;

int64_t blocks_of(int64_t n) { return (n + kScaleBlock - 1) / kScaleBlock; }

}  // namespace

namespace fp8k {

fp8_status_t linear_checks(const void* x, const uint8_t* wq, const float* s_w, const void* y,
                           int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (!x || !wq || !s_w || !y) return FP8_ERR_INVALID_ARG;
    if (K % 16 != 0) return FP8_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(s_w, 4))
        return FP8_ERR_UNSUPPORTED;
    DeviceState* d = nullptr;
    return current_device(&d);
}

bool encode_tmap_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t ld_bytes, uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace fp8k

extern "C" {

fp8_status_t fp8_quant_per_token(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                 uint8_t* xq, int64_t ldq, float* s_tok, void* stream) {
    return quant_rows(x_bf16, M, K, ldx, xq, ldq, s_tok, stream);
}

fp8_status_t fp8_quant_per_channel_weights(const void* w_bf16, int64_t N, int64_t K, int64_t ldw,
                                           uint8_t* wq, int64_t ldwq, float* s_w, void* stream) {
    return quant_rows(w_bf16, N, K, ldw, wq, ldwq, s_w, stream);
}

fp8_status_t fp8_scaled_gemm(const uint8_t* xq, const float* s_tok, const uint8_t* wq,
                             const float* s_w, void* y_bf16, int64_t M, int64_t N, int64_t K,
                             void* workspace, size_t ws_bytes, void* stream) {
    (void)workspace;
    (void)ws_bytes;
    fp8_status_t st = check_gemm(xq, s_tok, wq, s_w, y_bf16, M, N, K);
    if (st != FP8_OK || M == 0 || N == 0) return st;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    // A programmatic dependent of the previous kernel on the stream, which may
    // be anything (even the kernel writing wq): before its griddepcontrol.wait
    // the GEMM only prefetches weights into L2, the point of coherence, so an
    // early start cannot read stale inputs.
    return run_gemm(xq, s_tok, wq, s_w, y_bf16, M, N, K, stream, d);
}

size_t fp8_linear_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)N;
    if (M < 0 || K < 0 || M > kMaxDim || K > kMaxDim) return 0;
    return round_up(static_cast<size_t>(M) * static_cast<size_t>(K), 256) +
           round_up(4 * static_cast<size_t>(M), 256);
}

size_t fp8_scaled_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)M;
    (void)N;
    (void)K;
    return 0;
}

fp8_status_t fp8_linear(const void* x_bf16, const uint8_t* wq, const float* s_w, void* y_bf16,
                        int64_t M, int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                        void* stream) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (!x_bf16 || !wq || !s_w || !y_bf16) return FP8_ERR_INVALID_ARG;
    if (K <= 0 || K % 16 != 0) return FP8_ERR_UNSUPPORTED;
    if (!aligned(x_bf16, 16)) return FP8_ERR_UNSUPPORTED;
    const size_t need = fp8_linear_workspace_size(M, N, K);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return FP8_ERR_WORKSPACE;
    uint8_t* xq = static_cast<uint8_t*>(workspace);
    float* s_tok = reinterpret_cast<float*>(xq + round_up(static_cast<size_t>(M) * K, 256));
    fp8_status_t st = check_gemm(xq, s_tok, wq, s_w, y_bf16, M, N, K);
    if (st != FP8_OK) return st;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_quant_rows(x_bf16, M, K, K, xq, K, s_tok,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return FP8_ERR_CUDA;
    // Both launches are programmatic dependents of their predecessor and
    // release their own dependents at their start.  Before its
    // griddepcontrol.wait the GEMM only prefetches weights into L2; the wait
    // returns once the quantizer has completed, and the quantizer completes
    // only after its own wait (every earlier kernel, any writer of wq or x,
    // has finished).
    return run_gemm(xq, s_tok, wq, s_w, y_bf16, M, N, K, stream, d);
}

fp8_status_t fp8_quant_static(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                              const float* s, uint8_t* xq, int64_t ldq, float* s_rows,
                              void* stream) {
    fp8_status_t st = check_quant(x_bf16, M, K, ldx, xq, ldq, s);
    if (st != FP8_OK || M == 0) return st;
    if (s_rows && !aligned(s_rows, 4)) return FP8_ERR_UNSUPPORTED;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_quant_given_scale(x_bf16, M, K, ldx, s, xq, ldq, s_rows,
                                                   d->num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

size_t fp8_quant_per_tensor_workspace_size(int64_t M, int64_t K) {
    (void)M;
    (void)K;
    return sizeof(float) * fp8k::kMaxTensorPartials;
}

fp8_status_t fp8_quant_per_tensor(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* xq, int64_t ldq, float* s_out, float* s_rows,
                                  void* workspace, size_t ws_bytes, void* stream) {
    fp8_status_t st = check_quant(x_bf16, M, K, ldx, xq, ldq, s_out);
    if (st != FP8_OK || M == 0) return st;
    if (s_rows && !aligned(s_rows, 4)) return FP8_ERR_UNSUPPORTED;
    if (!workspace || ws_bytes < fp8_quant_per_tensor_workspace_size(M, K) ||
        !aligned(workspace, 16))
        return FP8_ERR_WORKSPACE;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_quant_per_tensor(x_bf16, M, K, ldx, xq, ldq, s_out, s_rows,
                                                  static_cast<float*>(workspace), d->num_sms,
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

namespace {
// Shared by the one-tensor and the keys-and-values entry points; x1, scale1
// and cache1 are null for the first.
fp8_status_t kv_cache_write(const void* x0, const void* x1, int64_t T, int64_t H, int64_t D,
                            const float* scale0, const float* scale1, int64_t scale_stride,
                            const int64_t* slot_mapping, uint8_t* cache0, uint8_t* cache1,
                            int64_t n_slots, bool pair, void* stream) {
    if (T < 0 || H < 0 || D < 0 || n_slots < 0 || scale_stride < 0 || T > kMaxDim ||
        H > kMaxDim || D > kMaxDim || n_slots > kMaxDim)
        return FP8_ERR_INVALID_ARG;
    if (T == 0 || H == 0 || D == 0 || n_slots == 0) return FP8_OK;
    if (!x0 || !scale0 || !cache0 || (pair && (!x1 || !scale1 || !cache1)))
        return FP8_ERR_INVALID_ARG;
    if (D % 16 != 0) return FP8_ERR_UNSUPPORTED;
    if (!aligned(x0, 16) || !aligned(cache0, 16) || !aligned(scale0, 4) ||
        (pair && (!aligned(x1, 16) || !aligned(cache1, 16) || !aligned(scale1, 4))) ||
        (slot_mapping && !aligned(slot_mapping, 8)))
        return FP8_ERR_UNSUPPORTED;
    DeviceState* d = nullptr;
    fp8_status_t st = current_device(&d);
    if (st != FP8_OK) return st;
    cudaError_t e = fp8k::launch_kv_cache_quant(x0, x1, T, H, D, scale0, scale1, scale_stride,
                                                slot_mapping, cache0, cache1, n_slots,
                                                d->num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}
}  // namespace

fp8_status_t fp8_kv_cache_quant(const void* kv_bf16, int64_t T, int64_t H, int64_t D,
                                const float* scale, int64_t scale_stride,
                                const int64_t* slot_mapping, uint8_t* cache, int64_t n_slots,
                                void* stream) {
    return kv_cache_write(kv_bf16, nullptr, T, H, D, scale, nullptr, scale_stride, slot_mapping,
                          cache, nullptr, n_slots, false, stream);
}

fp8_status_t fp8_kv_cache_quant_kv(const void* k_bf16, const void* v_bf16, int64_t T, int64_t H,
                                   int64_t D, const float* k_scale, const float* v_scale,
                                   int64_t scale_stride, const int64_t* slot_mapping,
                                   uint8_t* k_cache, uint8_t* v_cache, int64_t n_slots,
                                   void* stream) {
    return kv_cache_write(k_bf16, v_bf16, T, H, D, k_scale, v_scale, scale_stride, slot_mapping,
                          k_cache, v_cache, n_slots, true, stream);
}

fp8_status_t fp8_quant_per_token_group(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                       uint8_t* xq, int64_t ldq, float* s_x, void* stream) {
    fp8_status_t st = check_quant(x_bf16, M, K, ldx, xq, ldq, s_x);
    if (st != FP8_OK || M == 0 || K == 0) return st;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_quant_groups(x_bf16, M, K, ldx, xq, ldq, s_x, d->num_sms,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t fp8_quant_weight_blocks(const void* w_bf16, int64_t N, int64_t K, int64_t ldw,
                                     uint8_t* wq, int64_t ldwq, float* s_w, void* stream) {
    fp8_status_t st = check_quant(w_bf16, N, K, ldw, wq, ldwq, s_w);
    if (st != FP8_OK || N == 0 || K == 0) return st;
    if (blocks_of(N) > 65535) return FP8_ERR_UNSUPPORTED;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_quant_weight_blocks(w_bf16, N, K, ldw, wq, ldwq, s_w,
                                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t fp8_scaled_gemm_blockwise(const uint8_t* xq, const float* s_x, const uint8_t* wq,
                                       const float* s_w, void* y_bf16, int64_t M, int64_t N,
                                       int64_t K, void* workspace, size_t ws_bytes,
                                       void* stream) {
    (void)workspace;
    (void)ws_bytes;
    fp8_status_t st = check_gemm(xq, s_x, wq, s_w, y_bf16, M, N, K);
    if (st != FP8_OK || M == 0 || N == 0) return st;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    return run_gemm(xq, s_x, wq, s_w, y_bf16, M, N, K, stream, d, true);
}

size_t fp8_linear_blockwise_workspace_size(int64_t M, int64_t N, int64_t K) {
    (void)N;
    if (M < 0 || K < 0 || M > kMaxDim || K > kMaxDim) return 0;
    return round_up(static_cast<size_t>(M) * static_cast<size_t>(K), 256) +
           round_up(4 * static_cast<size_t>(M) * static_cast<size_t>(blocks_of(K)), 256);
}

fp8_status_t fp8_linear_blockwise(const void* x_bf16, const uint8_t* wq, const float* s_w,
                                  void* y_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                                  size_t ws_bytes, void* stream) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (!x_bf16 || !wq || !s_w || !y_bf16) return FP8_ERR_INVALID_ARG;
    if (K <= 0 || K % 16 != 0) return FP8_ERR_UNSUPPORTED;
    if (!aligned(x_bf16, 16)) return FP8_ERR_UNSUPPORTED;
    const size_t need = fp8_linear_blockwise_workspace_size(M, N, K);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return FP8_ERR_WORKSPACE;
    uint8_t* xq = static_cast<uint8_t*>(workspace);
    float* s_x = reinterpret_cast<float*>(xq + round_up(static_cast<size_t>(M) * K, 256));
    fp8_status_t st = check_gemm(xq, s_x, wq, s_w, y_bf16, M, N, K);
    if (st != FP8_OK) return st;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_quant_groups(x_bf16, M, K, K, xq, K, s_x, d->num_sms,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return FP8_ERR_CUDA;
    // as in fp8_linear: the GEMM reads nothing but L2 prefetches before its
    // griddepcontrol.wait, which returns once the quantizer has completed
    return run_gemm(xq, s_x, wq, s_w, y_bf16, M, N, K, stream, d, true);
}

fp8_status_t fp8_rmsnorm_quant(const void* x_bf16, const void* gamma_bf16, float eps, int64_t M,
                               int64_t K, int64_t ldx, uint8_t* xq, int64_t ldq, float* s_tok,
                               void* y_bf16, void* stream) {
    fp8_status_t st = check_quant(x_bf16, M, K, ldx, xq, ldq, s_tok);
    if (st != FP8_OK || M == 0) return st;
    if (K == 0 || K > 65536) return FP8_ERR_UNSUPPORTED;
    if (!gamma_bf16) return FP8_ERR_INVALID_ARG;
    if (!aligned(gamma_bf16, 16) || (y_bf16 && !aligned(y_bf16, 16))) return FP8_ERR_UNSUPPORTED;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return FP8_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_rmsnorm_quant(x_bf16, gamma_bf16, eps, M, K, ldx, xq, ldq, s_tok,
                                               y_bf16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t fp8_linear_rmsnorm(const void* x_bf16, const void* gamma_bf16, float eps,
                                const uint8_t* wq, const float* s_w, void* y_bf16, int64_t M,
                                int64_t N, int64_t K, void* workspace, size_t ws_bytes,
                                void* stream) {
    if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return FP8_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8_OK;
    if (!x_bf16 || !gamma_bf16 || !wq || !s_w || !y_bf16) return FP8_ERR_INVALID_ARG;
    if (K <= 0 || K % 16 != 0 || K > 65536) return FP8_ERR_UNSUPPORTED;
    if (!aligned(x_bf16, 16) || !aligned(gamma_bf16, 16)) return FP8_ERR_UNSUPPORTED;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return FP8_ERR_INVALID_ARG;
    const size_t need = fp8_linear_workspace_size(M, N, K);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return FP8_ERR_WORKSPACE;
    uint8_t* xq = static_cast<uint8_t*>(workspace);
    float* s_tok = reinterpret_cast<float*>(xq + round_up(static_cast<size_t>(M) * K, 256));
    fp8_status_t st = check_gemm(xq, s_tok, wq, s_w, y_bf16, M, N, K);
    if (st != FP8_OK) return st;
    DeviceState* d = nullptr;
    if ((st = current_device(&d)) != FP8_OK) return st;
    cudaError_t e = fp8k::launch_rmsnorm_quant(x_bf16, gamma_bf16, eps, M, K, K, xq, K, s_tok,
                                               nullptr, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return FP8_ERR_CUDA;
    // as in fp8_linear: the GEMM reads nothing but L2 prefetches before its
    // griddepcontrol.wait, which returns once the producer of the codes has
    // completed
    return run_gemm(xq, s_tok, wq, s_w, y_bf16, M, N, K, stream, d);
}

const char* fp8_status_string(fp8_status_t status) {
    switch (status) {
        case FP8_OK: return "FP8_OK";
        case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
        case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED";
        case FP8_ERR_WORKSPACE: return "FP8_ERR_WORKSPACE";
        case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
        case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
    }
    return "FP8_ERR_UNKNOWN";
}

fp8_status_t fp8_selftest_wait_timeout(int64_t limit_ns, uint64_t* report, void* stream) {
    if (limit_ns < 1000 || limit_ns > 100000000 || !report) return FP8_ERR_INVALID_ARG;
    if (!aligned(report, 8)) return FP8_ERR_UNSUPPORTED;
    DeviceState* d = nullptr;
    fp8_status_t st = current_device(&d);
    if (st != FP8_OK) return st;
    cudaError_t e = fp8k::launch_wait_timeout_selftest(
        static_cast<uint64_t>(limit_ns), d->status,
        reinterpret_cast<unsigned long long*>(report), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

fp8_status_t fp8_device_status(int clear) {
    DeviceState* d = nullptr;
    fp8_status_t st = current_device(&d);
    if (st != FP8_OK) return st;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess) return FP8_ERR_CUDA;
    if (clear) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess)
            return FP8_ERR_CUDA;
    }
    return v ? FP8_ERR_TIMEOUT : FP8_OK;
}

}  // extern "C"
