// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Nothing here is exported from the shared library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fp8w8a8.h"

namespace fp8k {

// Per-row dynamic E4M3 quantization (quant.cu).  R > 0, K % 16 == 0.
cudaError_t launch_quant_rows(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                              int64_t ldq, float* s, cudaStream_t st);
// The same row layout with the scale *s_given for every row (static scale);
// K > 0; s_rows (optional) receives the scale per row.  Rows longer than
// the register path holds: cudaErrorNotSupported.
cudaError_t launch_quant_rows_given(const void* x, int64_t R, int64_t K, int64_t ldx,
                                    uint8_t* q, int64_t ldq, const float* s_given, float* s_rows,
                                    cudaStream_t st);

// Everything a scaled-GEMM launch needs.  xq [M, K] and wq [N, K] are
// contiguous E4M3, y [M, N] contiguous bf16.
struct GemmArgs {
    const uint8_t* xq;
    const float* s_tok;
    const uint8_t* wq;
    const float* s_w;
    void* y;
    int M, N, K;
    unsigned* status;     // device status word
    int num_sms;
    bool pdl;             // launch as a programmatic dependent of the previous kernel
    int pair_clusters;    // co-resident clusters of the paired-SM kernel (0: unknown)
    // decode_clusters[(c - 1) * 9 + S]: clusters of S decode-GEMM CTAs that
    // can be resident at once with the footprint of c CTAs per SM (c = 1..3,
    // S = 1..8; null or 0: unknown)
    const int* decode_clusters = nullptr;
    cudaStream_t stream;
};

// 2-D row-major uint8 tensor [rows, cols] (leading dimension ld_bytes) as a
// TMA tensor map with a {box_cols, box_rows} box and 128-byte swizzle.
// Returns false if the driver rejects it.  (api.cu)
bool encode_tmap_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t ld_bytes, uint32_t box_cols, uint32_t box_rows);

// Weight-streaming split-K tcgen05 GEMM for M <= kDecodeMaxM (gemm_decode.cu);
// the block-scaled variant (gemm_blockwise.cu) up to kBlockwiseDecodeMaxM.
constexpr int kDecodeMaxM = 256;
constexpr int kBlockwiseDecodeMaxM = 64;

// Persistent 256x256-tile GEMM on pairs of SMs (tcgen05 cta_group::2) for
// every larger M (gemm_pair.cu).
cudaError_t launch_gemm_pair(const GemmArgs& a);
int gemm_pair_resident_clusters(int num_sms);

cudaError_t launch_gemm_decode(const GemmArgs& a);
// How many clusters of `size` decode-GEMM CTAs can be resident at once (a
// cluster must fit on the SMs of one GPC); 0 if unknown.
int gemm_decode_resident_clusters(int size, int ctas_per_sm);

// Quantization with other scale granularities (quant_variants.cu).
// Every row quantized with the scale *s; s_rows (optional) gets s per row.
cudaError_t launch_quant_given_scale(const void* x, int64_t R, int64_t K, int64_t ldx,
                                     const float* s, uint8_t* q, int64_t ldq, float* s_rows,
                                     int num_sms, cudaStream_t st);
// One dynamic scale for the whole tensor; `partial` holds kMaxTensorPartials floats.
constexpr int kMaxTensorPartials = 2048;
cudaError_t launch_quant_per_tensor(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                                    int64_t ldq, float* s_out, float* s_rows, float* partial,
                                    int num_sms, cudaStream_t st);
// KV-cache write: x0 [T, H, D] -> cache0[slot[t] (or t), h, :] with scale
// scale0[h * scale_stride]; tokens whose slot is negative or >= n_slots are
// skipped.  x1 non-null: the same for x1 / scale1 / cache1 in the same launch.
cudaError_t launch_kv_cache_quant(const void* x0, const void* x1, int64_t T, int64_t H,
                                  int64_t D, const float* scale0, const float* scale1,
                                  int64_t scale_stride, const int64_t* slot, uint8_t* cache0,
                                  uint8_t* cache1, int64_t n_slots, int num_sms,
                                  cudaStream_t st);

// RMSNorm fused with the per-token quantizer (norm_quant.cu); K <= 65536.
// y (optional) receives the bf16 normalised rows, [R, K] contiguous.
cudaError_t launch_rmsnorm_quant(const void* x, const void* gamma, float eps, int64_t R,
                                 int64_t K, int64_t ldx, uint8_t* q, int64_t ldq, float* s,
                                 void* y, cudaStream_t st);

// Block-wise scales (quant_variants.cu): activations one scale per token per
// 128 inputs, s [R, ceil(K/128)]; weights one scale per 128 x 128 block,
// s [ceil(N/128), ceil(K/128)].
cudaError_t launch_quant_groups(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                                int64_t ldq, float* s, int num_sms, cudaStream_t st);
cudaError_t launch_quant_weight_blocks(const void* w, int64_t N, int64_t K, int64_t ldw,
                                       uint8_t* q, int64_t ldq, float* s, cudaStream_t st);

// Block-scaled GEMM (gemm_blockwise.cu): GemmArgs with s_tok = s_x
// [M, ceil(K/128)] and s_w [ceil(N/128), ceil(K/128)].
cudaError_t launch_gemm_blockwise(const GemmArgs& a);

// Self-test of the bounded waits (selftest.cu): one CTA whose waits run out
// after limit_ns; report[0..3] as fp8_selftest_wait_timeout documents.
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned* status,
                                         unsigned long long* report, cudaStream_t st);

// The checks fp8_linear makes on everything but its workspace (sizes,
// pointers, alignment), then the device check (api.cu).  FP8_OK for an
// empty layer too.
fp8_status_t linear_checks(const void* x, const uint8_t* wq, const float* s_w, const void* y,
                           int64_t M, int64_t N, int64_t K);

// One-time per-device kernel attribute setup (dynamic shared memory limits).
cudaError_t prepare_gemm_decode();
cudaError_t prepare_gemm_blockwise();
cudaError_t prepare_gemm_pair();

}  // namespace fp8k
