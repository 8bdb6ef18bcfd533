/*
 * fp8w8a8.h -- C ABI of the GB300 (sm_103a) FP8_DYNAMIC W8A8 linear layer.
 *
 * The layer (page titles and sections of the sources it follows):
 *   "FP8 Inference Explained, in depth", "Inside a quantized linear layer":
 *     weights are stored offline as E4M3 with one FP32 scale per output
 *     channel; at run time a small kernel finds each token's amax, divides
 *     and casts the activations to E4M3; the tensor cores multiply E4M3 by
 *     E4M3 and accumulate in FP32; both scales are constant along K, so
 *     y[m,n] = s_tok[m] * s_w[n] * sum_k q_x[m,k] * q_w[n,k].
 *   "FP8 Inference Explained, in depth", "Scales and their granularity":
 *     x_fp8 = round(x / s) with s = amax / 448.
 *   "FP8 Quantization", "How FP8 Matmul Works at the Hardware Level":
 *     FP8 x FP8 -> FP32 accumulate -> BF16 output.
 *
 * Numerics of every quantizing entry point (bit-exact, deterministic):
 *   amax = max_k |x[k]| in fp32 (bf16 inputs widen exactly);
 *   s    = amax / 448 as an IEEE fp32 division (round to nearest even),
 *          or s = 1 when amax == 0;
 *   q[k] = E4M3(x[k] / s): IEEE fp32 quotient, then round to nearest even
 *          onto the float8_e4m3fn grid, saturating at +-448 (0x7E / 0xFE),
 *          subnormals down to 2^-9, the sign of zero kept.
 *   NaN or Inf inputs are outside the contract.
 *
 * Conventions shared by every entry point:
 *   - Pointers marked "device" are CUDA device pointers owned by the caller
 *     (for example PyTorch-allocated).  The library never allocates, frees or
 *     keeps them after the call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream and never
 *     synchronizes the host.
 *   - Kernels are launched with programmatic stream serialization: one may
 *     start while the previous work on the stream drains, but reads no
 *     global memory except L2 prefetches of weights before all of that work
 *     has completed, so stream order holds for the caller's data.  Each
 *     kernel also lets its successor on the stream launch early; a caller's
 *     kernel launched with programmatic stream serialization after one of
 *     these calls must execute griddepcontrol.wait (cudaGridDependencySynchronize)
 *     before reading the call's outputs, as any such kernel must.
 *   - Layouts are row-major.  Activations X are [M, K] (tokens x in-features),
 *     weights W are [N, K] (out-features x in-features, the nn.Linear layout,
 *     K contiguous), outputs Y are [M, N] bf16 with leading dimension N.
 *   - Host-side argument checks run before any launch; a rejected call
 *     launches nothing and returns FP8_ERR_INVALID_ARG or FP8_ERR_UNSUPPORTED.
 *     M == 0 or N == 0 is a valid no-op and returns FP8_OK.
 *   - The current CUDA device must be the one that owns the pointers; it must
 *     be a compute capability 10.3 (GB300) device, else FP8_ERR_UNSUPPORTED.
 *   - A launch failure returns FP8_ERR_CUDA.  Device-side waits are bounded:
 *     a kernel whose wait runs out records it in a device status word and
 *     exits; fp8_device_status() reports it as FP8_ERR_TIMEOUT.
 */
#ifndef FP8W8A8_H
#define FP8W8A8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8_API __attribute__((visibility("default")))
#else
#define FP8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8_OK = 0,
    FP8_ERR_INVALID_ARG = 1,  /* null pointer, negative size, ld < K, ...    */
    FP8_ERR_UNSUPPORTED = 2,  /* alignment/size outside what the kernels take,
                                 or not a GB300 device                        */
    FP8_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small   */
    FP8_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed            */
    FP8_ERR_TIMEOUT = 5       /* a device-side wait ran out (see
                                 fp8_device_status)                           */
} fp8_status_t;

/*
 * Dynamic per-token activation quantization.
 * Source: "FP8 Inference Explained, in depth", "Scales and their
 * granularity" (s = amax / 448, x_fp8 = round(x / s)); "Quantization: FP8
 * inference and KV-cache quantization", "Dynamic scales or static scales"
 * (one scale per token, recomputed on every forward pass).
 *
 *   x_bf16 [device, in]  bf16 [M, K], leading dimension ldx (elements)
 *   M, K                 tokens, in-features; M >= 0, K >= 0
 *   ldx                  >= K, multiple of 8 (16-byte rows)
 *   xq     [device, out] E4M3 codes [M, K], leading dimension ldq (bytes)
 *   ldq                  >= K, multiple of 16
 *   s_tok  [device, out] fp32 [M], the dequant scale of each token
 * Requirements: K % 16 == 0; x_bf16 and xq 16-byte aligned; s_tok 4-byte
 * aligned.  K == 0 writes s_tok = 1.
 */
FP8_API fp8_status_t fp8_quant_per_token(const void* x_bf16, int64_t M, int64_t K,
                                         int64_t ldx, uint8_t* xq, int64_t ldq, float* s_tok,
                                         void* stream);

/*
 * Static per-output-channel weight quantization (run once, offline): the
 * same rule as fp8_quant_per_token applied to each row of W [N, K].
 * Source: "FP8 Quantization", "Granularity" (per-channel: one scale per
 * output row) and "Implementation" (FP8_DYNAMIC: weights quantized
 * statically per channel offline).
 *
 *   w_bf16 [device, in]  bf16 [N, K], leading dimension ldw (elements)
 *   wq     [device, out] E4M3 codes [N, K], leading dimension ldwq (bytes)
 *   s_w    [device, out] fp32 [N]
 * Requirements as for fp8_quant_per_token (with N for M).
 */
FP8_API fp8_status_t fp8_quant_per_channel_weights(const void* w_bf16, int64_t N, int64_t K,
                                                   int64_t ldw, uint8_t* wq, int64_t ldwq,
                                                   float* s_w, void* stream);

/*
 * Scaled FP8 GEMM with the dequant epilogue fused:
 *   y[m, n] = bf16_rn( (acc[m, n] * s_tok[m]) * s_w[n] ),
 *   acc[m, n] = sum_k e4m3(xq[m, k]) * e4m3(wq[n, k])   (fp32 accumulation)
 * Source: "FP8 Inference Explained, in depth", "Inside a quantized linear
 * layer"; "FP8 Quantization", "How FP8 Matmul Works at the Hardware Level".
 *
 *   xq     [device, in]  E4M3 [M, K], contiguous (leading dimension K)
 *   s_tok  [device, in]  fp32 [M]
 *   wq     [device, in]  E4M3 [N, K], contiguous (leading dimension K)
 *   s_w    [device, in]  fp32 [N]
 *   y_bf16 [device, out] bf16 [M, N], contiguous
 *   workspace, ws_bytes  unused by the current kernels (may be NULL / 0);
 *                        fp8_scaled_gemm_workspace_size() returns 0.
 * Requirements: K % 16 == 0, K > 0; xq, wq, y_bf16 16-byte aligned;
 * M, N, K < 2^31.  The fp32 summation order is fixed for a given shape, so
 * repeated calls give identical bits.
 * Kernel choice: M <= 256 uses the weight-streaming split-K kernel (weights on
 * the 128-row MMA side, tokens on the other, in tiles of 16, 32, 64, 128 or
 * 256), larger M the persistent 256x256-tile kernel that runs each MMA on a
 * pair of SMs (cta_group::2).
 */
FP8_API fp8_status_t fp8_scaled_gemm(const uint8_t* xq, const float* s_tok, const uint8_t* wq,
                                     const float* s_w, void* y_bf16, int64_t M, int64_t N,
                                     int64_t K, void* workspace, size_t ws_bytes, void* stream);

/*
 * The whole W8A8 linear layer: fp8_quant_per_token on X into the workspace,
 * then fp8_scaled_gemm, on `stream`, as two launches (the second may start
 * its prologue and weight prefetch while the first finishes).
 *
 *   x_bf16 [device, in]  bf16 [M, K], contiguous
 *   wq, s_w              as for fp8_scaled_gemm (offline-quantized weights)
 *   y_bf16 [device, out] bf16 [M, N], contiguous
 *   workspace [device]   at least fp8_linear_workspace_size(M, N, K) bytes,
 *                        256-byte aligned; holds xq [M, K] then s_tok [M].
 *                        Its contents after the call are the quantized
 *                        activations and their scales.  It must not be in
 *                        use by another call in flight.
 * Requirements: as for the two calls it makes.
 */
FP8_API fp8_status_t fp8_linear(const void* x_bf16, const uint8_t* wq, const float* s_w,
                                void* y_bf16, int64_t M, int64_t N, int64_t K, void* workspace,
                                size_t ws_bytes, void* stream);

/*
 * fp8_linear for callers that cannot allocate device memory (no workspace
 * argument; the call allocates nothing).  The pages have no counterpart:
 * this is a convenience of this library.
 *
 * Who needs it: code that may not create device allocations of its own, such
 * as a plugin inside a host application that owns all device memory, or a
 * latency-critical loop in which cudaMalloc / cudaFree (which can synchronize
 * the device) must not run.  The quantized activations and scales go to a
 * fixed array of FP8_STATIC_SCRATCH_BYTES inside the library instead; every
 * GPU that loads the library holds that array until the process exits.
 *
 *   x_bf16, wq, s_w, y_bf16, M, N, K, stream   as for fp8_linear.
 * Limit: round_up(M*K, 256) + round_up(4*M, 256) <= FP8_STATIC_SCRATCH_BYTES,
 * else FP8_ERR_WORKSPACE and nothing is launched.
 * The first call on each device does a one-time set-up (it looks up the
 * array's device address with that device current); make that first call
 * before any stream capture.  All calls on a device share the array and it
 * keeps the last call's contents: calls that overlap on the GPU (two streams
 * at once) race on it.  Nothing in it needs to start at zero.
 */
#define FP8_STATIC_SCRATCH_BYTES (8u << 20)
FP8_API fp8_status_t fp8_linear_static_scratch(const void* x_bf16, const uint8_t* wq,
                                               const float* s_w, void* y_bf16, int64_t M,
                                               int64_t N, int64_t K, void* stream);

/*
 * Quantization with a given (static, calibrated) per-tensor scale:
 *   q[m,k] = E4M3_rn_satfinite(x[m,k] / s)   (IEEE fp32 quotient)
 * Source: "Quantization: FP8 inference and KV-cache quantization", "Dynamic
 * scales or static scales" (a scale fixed from calibration costs nothing at
 * run time; values beyond 448 s clip to +-448 in saturating mode).
 *
 *   x_bf16, M, K, ldx, xq, ldq   as for fp8_quant_per_token
 *   s       [device, in]  fp32 [1], the scale
 *   s_rows  [device, out] fp32 [M] or NULL: s written for every row, so the
 *                         codes can go straight to fp8_scaled_gemm
 * Requirements as for fp8_quant_per_token; s 4-byte aligned, s > 0 finite.
 */
FP8_API fp8_status_t fp8_quant_static(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                      const float* s, uint8_t* xq, int64_t ldq, float* s_rows,
                                      void* stream);

/*
 * Dynamic per-tensor quantization: one scale for the whole [M, K] tensor,
 *   s = amax_{m,k} |x| / 448 (IEEE fp32 division; 1 if the tensor is zero),
 *   q[m,k] = E4M3_rn_satfinite(x[m,k] / s).
 * Source: "FP8 Quantization", "Choose Scaling Strategy" (dynamic scaling from
 * max |X| on the fly) and "Granularity" (per-tensor: one scale for the entire
 * matrix).  Two launches; bit-identical results on every call.
 *
 *   x_bf16, M, K, ldx, xq, ldq   as for fp8_quant_per_token
 *   s_out   [device, out] fp32 [1]
 *   s_rows  [device, out] fp32 [M] or NULL (s for every row, as above)
 *   workspace [device]    fp8_quant_per_tensor_workspace_size() bytes,
 *                         16-byte aligned (per-CTA maxima)
 */
FP8_API fp8_status_t fp8_quant_per_tensor(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                          uint8_t* xq, int64_t ldq, float* s_out, float* s_rows,
                                          void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes of fp8_quant_per_tensor (a fixed 8 KB). */
FP8_API size_t fp8_quant_per_tensor_workspace_size(int64_t M, int64_t K);

/*
 * FP8 KV-cache write (quantize on write): for every token t, head h, and
 * d < D,
 *   cache[slot[t], h, d] = E4M3_rn_satfinite(kv[t, h, d] / scale[h * scale_stride])
 * Source: "Quantization: FP8 inference and KV-cache quantization", "Turning
 * it on in an engine" (one scale per tensor or per attention head, 1.0 when
 * uncalibrated; values beyond 448 are clipped) and "FP8 Inference Explained,
 * in depth", "FP8 KV cache".
 *
 *   kv_bf16 [device, in]  bf16 [T, H, D], contiguous (keys or values)
 *   scale   [device, in]  fp32: [H] with scale_stride 1 (per head) or [1]
 *                         with scale_stride 0 (per tensor)
 *   slot_mapping [device, in] int64 [T] or NULL (token t -> row t); a token
 *                         whose slot is negative or >= n_slots is skipped;
 *                         slots must be distinct (two tokens writing one
 *                         slot leave an unspecified mix of their codes)
 *   cache   [device, out] E4M3 [n_slots, H, D], contiguous
 * Requirements: D % 16 == 0; kv_bf16 and cache 16-byte aligned.
 */
FP8_API fp8_status_t fp8_kv_cache_quant(const void* kv_bf16, int64_t T, int64_t H, int64_t D,
                                        const float* scale, int64_t scale_stride,
                                        const int64_t* slot_mapping, uint8_t* cache,
                                        int64_t n_slots, void* stream);

/*
 * A layer's keys and values written in one launch: exactly
 *   fp8_kv_cache_quant(k_bf16, T, H, D, k_scale, scale_stride, slot_mapping,
 *                      k_cache, n_slots, stream) and
 *   fp8_kv_cache_quant(v_bf16, T, H, D, v_scale, scale_stride, slot_mapping,
 *                      v_cache, n_slots, stream)
 * with the same slots (the cache holds keys and values per layer, "FP8
 * Inference Explained, in depth", "FP8 KV cache"; an engine writes both at
 * once, "Quantization: FP8 inference and KV-cache quantization", "Turning it
 * on in an engine").  Arguments and requirements as above, for each of the
 * two tensors; k_cache and v_cache must not overlap.
 */
FP8_API fp8_status_t fp8_kv_cache_quant_kv(const void* k_bf16, const void* v_bf16, int64_t T,
                                           int64_t H, int64_t D, const float* k_scale,
                                           const float* v_scale, int64_t scale_stride,
                                           const int64_t* slot_mapping, uint8_t* k_cache,
                                           uint8_t* v_cache, int64_t n_slots, void* stream);

/*
 * Block-wise scales.  Source: "FP8 Quantization", "Granularity" (per-block:
 * one scale per 128 x 128 weight tile) and "FP8 Inference Explained, in
 * depth", "Inside a quantized linear layer" (block-wise scales vary along k,
 * so each block's partial sum is multiplied by its scales before the partial
 * sums are added).  Reading: activations take one scale per token per 128
 * inputs (the 128-element promotion interval of "Quantization: FP8 inference
 * and KV-cache quantization", "Training in FP8 or lower"); every block uses
 * the per-token rule, s = fl32(amax / 448) (1 if the block is all zero) and
 * q = E4M3_rn_satfinite(fl32(x / s)).  KB = ceil(K / 128), NB = ceil(N / 128);
 * the last block of each dimension may be partial.
 *
 * fp8_quant_per_token_group:  x_bf16 [M, K] (ld ldx) -> xq [M, K] (ld ldq),
 *   s_x [M, KB] fp32 row-major.  Requirements as for fp8_quant_per_token.
 * fp8_quant_weight_blocks:    w_bf16 [N, K] (ld ldw) -> wq [N, K] (ld ldwq),
 *   s_w [NB, KB] fp32 row-major (offline, once per checkpoint).  Same
 *   requirements; NB <= 65535.
 */
FP8_API fp8_status_t fp8_quant_per_token_group(const void* x_bf16, int64_t M, int64_t K,
                                               int64_t ldx, uint8_t* xq, int64_t ldq, float* s_x,
                                               void* stream);
FP8_API fp8_status_t fp8_quant_weight_blocks(const void* w_bf16, int64_t N, int64_t K,
                                             int64_t ldw, uint8_t* wq, int64_t ldwq, float* s_w,
                                             void* stream);

/*
 * Block-scaled GEMM:
 *   y[m,n] = bf16_rn( sum_kb s_x[m,kb] * s_w[n/128,kb] *
 *                     sum_{k in block kb} e4m3(xq[m,k]) * e4m3(wq[n,k]) )
 * with each block's partial sum accumulated in fp32.
 *
 *   xq [device] E4M3 [M, K] contiguous; s_x fp32 [M, KB]
 *   wq [device] E4M3 [N, K] contiguous; s_w fp32 [NB, KB]
 *   y  [device, out] bf16 [M, N] contiguous
 *   workspace  unused (may be NULL)
 * Requirements as for fp8_scaled_gemm.
 */
FP8_API fp8_status_t fp8_scaled_gemm_blockwise(const uint8_t* xq, const float* s_x,
                                               const uint8_t* wq, const float* s_w, void* y_bf16,
                                               int64_t M, int64_t N, int64_t K, void* workspace,
                                               size_t ws_bytes, void* stream);

/*
 * The block-scaled layer: group quantization of x (into the workspace: codes
 * [M, K] at offset 0, s_x [M, KB] at round_up(M*K, 256)) followed by the
 * block-scaled GEMM.  wq / s_w come from fp8_quant_weight_blocks.
 * Requirements as for fp8_linear, with
 * fp8_linear_blockwise_workspace_size(M, N, K) workspace bytes.
 */
FP8_API fp8_status_t fp8_linear_blockwise(const void* x_bf16, const uint8_t* wq, const float* s_w,
                                          void* y_bf16, int64_t M, int64_t N, int64_t K,
                                          void* workspace, size_t ws_bytes, void* stream);

/* round_up(M*K, 256) + round_up(4*M*KB, 256) bytes. */
FP8_API size_t fp8_linear_blockwise_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * RMSNorm with the per-token quantizer fused into it (the amax reduction done
 * by the kernel that produces the activations).  Source: "FP8 Inference
 * Explained, in depth", "Scales and their granularity" (engines fuse the
 * per-token amax into the preceding kernel) and "What stays in higher
 * precision" (normalisation stays in 16/32-bit).  The pages do not define the
 * normalisation; this is RMSNorm with every step an IEEE fp32 operation:
 *   ss = sum_k x_k^2 (fp32, within 2^-17 relative of the exact sum),
 *   inv = fl32(1 / fl32(sqrt(fl32(fl32(ss / K) + eps)))),
 *   y_k = bf16_rn(fl32(fl32(x_k * inv) * gamma_k)),
 * followed by the per-token rule of fp8_quant_per_token on the bf16 row y.
 *
 *   x_bf16     [device, in]  bf16 [M, K], leading dimension ldx
 *   gamma_bf16 [device, in]  bf16 [K], 16-byte aligned
 *   eps                      >= 0, finite
 *   xq, ldq, s_tok           as for fp8_quant_per_token (codes of y, scales)
 *   y_bf16     [device, out] bf16 [M, K] contiguous, or NULL: the normalised
 *                            rows the codes were taken from
 * Requirements as for fp8_quant_per_token, and 0 < K <= 65536.
 */
FP8_API fp8_status_t fp8_rmsnorm_quant(const void* x_bf16, const void* gamma_bf16, float eps,
                                       int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                                       int64_t ldq, float* s_tok, void* y_bf16, void* stream);

/*
 * The layer fed by RMSNorm: fp8_rmsnorm_quant of x into the workspace (the
 * same layout and size as fp8_linear's) followed by the scaled GEMM.
 * x contiguous [M, K]; requirements as for fp8_linear and K <= 65536.
 */
FP8_API fp8_status_t fp8_linear_rmsnorm(const void* x_bf16, const void* gamma_bf16, float eps,
                                        const uint8_t* wq, const float* s_w, void* y_bf16,
                                        int64_t M, int64_t N, int64_t K, void* workspace,
                                        size_t ws_bytes, void* stream);

/* Workspace bytes fp8_linear needs for an [M, K] x [N, K]^T layer:
 * round_up(M*K, 256) + round_up(4*M, 256).  0 for invalid sizes. */
FP8_API size_t fp8_linear_workspace_size(int64_t M, int64_t N, int64_t K);

/* Workspace bytes fp8_scaled_gemm needs (currently always 0). */
FP8_API size_t fp8_scaled_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* Static, NUL-terminated name of a status code; never NULL. */
FP8_API const char* fp8_status_string(fp8_status_t status);

/* Device status word of the current device: FP8_OK, or FP8_ERR_TIMEOUT if a
 * kernel of this library gave up a bounded wait since the last clear.  Reads
 * the word with a synchronous copy (it waits for the device); clear != 0
 * resets it.  Returns FP8_ERR_CUDA if the copy fails. */
FP8_API fp8_status_t fp8_device_status(int clear);

/*
 * Self-test of the bounded device waits (failure detection).  The pages have
 * no counterpart: it exercises this library's own safeguard.  Every wait of
 * the GEMM kernels has a time limit; when one runs out the kernel raises a
 * CTA-wide abort flag (the CTA's other waits give up too), drains the tensor
 * core operations it issued, frees its tensor memory, records the timeout in
 * the device status word and returns.  This call launches one small kernel
 * that goes through exactly that sequence on purpose: a wait on a barrier
 * that nothing arrives on gives up after limit_ns, and a second role waiting
 * with the kernels' own (long) limit must return on the abort flag.
 *
 *   limit_ns  [in]           1e3 .. 1e8 (1 us .. 100 ms), else INVALID_ARG
 *   report    [device, out]  4 x uint64, 8-byte aligned:
 *                            [0] 1 if the short wait gave up (expected),
 *                            [1] 1 if the second role returned without its
 *                                barrier completing (expected),
 *                            [2] ns from the start of the waits until the
 *                                first one gave up (expected >= limit_ns),
 *                            [3] ns until the second role returned.
 * Afterwards fp8_device_status() returns FP8_ERR_TIMEOUT until cleared with
 * fp8_device_status(1).  Nothing faults; the context stays usable.
 */
FP8_API fp8_status_t fp8_selftest_wait_timeout(int64_t limit_ns, uint64_t* report, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8W8A8_H */
