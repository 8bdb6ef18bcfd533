// Quantization with scales other than one per token:
//   * a given (static, calibrated) scale: q = E4M3_rn_sat(x / s)
//     ("Quantization: FP8 inference and KV-cache quantization", "Dynamic
//     scales or static scales": no run-time reduction; values beyond 448 s
//     clip to +-448);
//   * one dynamic scale for the whole tensor, s = amax(all) / 448
//     ("FP8 Quantization", "Choose Scaling Strategy" and "Granularity");
//   * FP8 KV-cache writes with a per-tensor or per-head scale, scattered to
//     cache slots ("Quantization: FP8 inference and KV-cache quantization",
//     "Turning it on in an engine").
// The arithmetic is that of the per-token quantizer (quant_math.cuh).  The
// static scale runs in the per-token quantizer's row layout (quant.cu) and
// falls back to the grid-stride loop here for empty or very long rows; the
// others are grid-stride loops over 16-element chunks (one 32-byte load, one
// 16-byte store), memory-bound; contiguous tensors take a flat loop with no
// row arithmetic and two chunks in flight per thread.  The per-tensor amax is two
// launches (per-CTA maxima, then every CTA reduces them), which needs no
// atomics and no zeroed memory; the first pass reads x with an L2
// evict-last hint and the second reads it back from the end, so that much of
// it comes from L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8k {
namespace {

constexpr int kThreads = 256;
constexpr int64_t kGroup = 128;  // block edge of the block-wise scales

template <bool kBounded = false>
__device__ __forceinline__ uint4 quant16(const uint4* src, const Divisor& d) {
    const uint4 a = __ldg(src), b = __ldg(src + 1);
    const uint2 qa = quant8<kBounded>(a, d), qb = quant8<kBounded>(b, d);
    return make_uint4(qa.x, qa.y, qb.x, qb.y);
}

template <bool kBounded = false>
__device__ __forceinline__ uint4 quant16v(const uint4& a, const uint4& b, const Divisor& d) {
    const uint2 qa = quant8<kBounded>(a, d), qb = quant8<kBounded>(b, d);
    return make_uint4(qa.x, qa.y, qb.x, qb.y);
}

// 16-byte load that does not allocate in L1, with an L2 eviction-priority
// hint (a createpolicy result), and the matching store.
__device__ __forceinline__ uint4 ld_hint(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ void st_hint(uint4* p, const uint4& v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

constexpr int kUnroll = 2;  // chunks in flight per thread and loop trip

// Contiguous x [R, K] / s -> contiguous q: chunk i is the 16 elements at
// offset 16 i of both, so the grid-stride loop needs no row arithmetic and
// keeps kUnroll chunks of loads in flight per thread.  `reverse` walks the
// chunks from the end (the per-tensor second pass: the chunks the first pass
// read last are the likeliest still in L2; measured faster than each thread
// revisiting its own chunks backwards).
template <bool kBounded>
__device__ __forceinline__ void quant_flat(const uint16_t* __restrict__ x, uint8_t* __restrict__ q,
                                           int64_t total, const Divisor& dv, uint64_t ld_pol,
                                           uint64_t st_pol, bool reverse) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    for (; j + (kUnroll - 1) * stride < total; j += kUnroll * stride) {
        uint4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t ch = j + u * stride;
            const int64_t i = reverse ? total - 1 - ch : ch;
            const uint4* src = reinterpret_cast<const uint4*>(x + i * 16);
            a[u] = ld_hint(src, ld_pol);
            b[u] = ld_hint(src + 1, ld_pol);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t ch = j + u * stride;
            const int64_t i = reverse ? total - 1 - ch : ch;
            st_hint(reinterpret_cast<uint4*>(q + i * 16), quant16v<kBounded>(a[u], b[u], dv),
                    st_pol);
        }
    }
    for (; j < total; j += stride) {
        const int64_t i = reverse ? total - 1 - j : j;
        const uint4* src = reinterpret_cast<const uint4*>(x + i * 16);
        const uint4 a = ld_hint(src, ld_pol), b = ld_hint(src + 1, ld_pol);
        st_hint(reinterpret_cast<uint4*>(q + i * 16), quant16v<kBounded>(a, b, dv), st_pol);
    }
}

// x [R, K] (ld ldx elements) / s -> q [R, K] (ld ldq bytes), grid-stride
// over 16-element chunks.  kBounded: s = amax / 448 of x itself.
template <bool kBounded = false>
__device__ __forceinline__ void quant_chunks(const uint16_t* __restrict__ x, int64_t R, int64_t K,
                                             int64_t ldx, float s, uint8_t* __restrict__ q,
                                             int64_t ldq, uint64_t ld_pol, uint64_t st_pol,
                                             bool reverse = false) {
    const int64_t C = K >> 4;
    const int64_t total = R * C;
    const Divisor dv = divisor_of(s);
    if (ldx == K && ldq == K) {
        quant_flat<kBounded>(x, q, total, dv, ld_pol, st_pol, reverse);
        return;
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t r = i / C, c = i - r * C;
        const uint4* src = reinterpret_cast<const uint4*>(x + r * ldx + c * 16);
        *reinterpret_cast<uint4*>(q + r * ldq + c * 16) = quant16<kBounded>(src, dv);
    }
}

// s for every row (the per-row scale vector the scaled GEMM consumes).
__device__ __forceinline__ void fill_rows(float* __restrict__ s_rows, int64_t R, float s) {
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; r < R;
         r += static_cast<int64_t>(gridDim.x) * kThreads)
        s_rows[r] = s;
}

// Static scale: every row divided by *s_ptr.
__global__ void __launch_bounds__(kThreads)
    quant_given_scale(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ldx,
                      const float* __restrict__ s_ptr, uint8_t* __restrict__ q, int64_t ldq,
                      float* __restrict__ s_rows) {
    pdl_launch_dependents();
    pdl_wait_primary();
    const float s = __ldg(s_ptr);
    const uint64_t pol = policy_evict_first();
    quant_chunks(x, R, K, ldx, s, q, ldq, pol, pol);
    if (s_rows) fill_rows(s_rows, R, s);
}

__device__ __forceinline__ float block_max(float m, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane_id() == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
    __syncthreads();
    return r;
}

// Pass 1 of the per-tensor scale: partial[b] = max |x| over this CTA's chunks.
// Held to 32 registers (no spill) so that all eight CTAs per SM of the grid
// are resident: more loads in flight (measured +2% on the per-tensor pair).
__global__ void __launch_bounds__(kThreads, 8)
    tensor_amax_partial(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ldx,
                        float* __restrict__ partial) {
    __shared__ float red[kThreads / 32];
    pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t C = K >> 4;
    const int64_t total = R * C;
    float m = 0.0f;
    if (ldx == K) {
        // contiguous: flat chunks, four in flight per thread; the lines stay
        // in L2 (evict_last) for the second pass
        const uint64_t pol = policy_evict_last();
        const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
        int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
        constexpr int U = 4;
        for (; i + (U - 1) * stride < total; i += U * stride) {
            uint4 a[U], b[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint4* src = reinterpret_cast<const uint4*>(x + (i + u * stride) * 16);
                a[u] = ld_hint(src, pol);
                b[u] = ld_hint(src + 1, pol);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) m = amax8(b[u], amax8(a[u], m));
        }
        for (; i < total; i += stride) {
            const uint4* src = reinterpret_cast<const uint4*>(x + i * 16);
            m = amax8(ld_hint(src + 1, pol), amax8(ld_hint(src, pol), m));
        }
    } else {
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
             i += static_cast<int64_t>(gridDim.x) * kThreads) {
            const int64_t r = i / C, c = i - r * C;
            const uint4* src = reinterpret_cast<const uint4*>(x + r * ldx + c * 16);
            m = amax8(__ldg(src + 1), amax8(__ldg(src), m));
        }
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) partial[blockIdx.x] = m;
}

// Pass 2: every CTA reduces the partial maxima (a fixed, order-independent
// max), forms s = amax / 448 (1 if zero) and quantizes its chunks.
__global__ void __launch_bounds__(kThreads)
    tensor_quant(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ldx,
                 const float* __restrict__ partial, int n_partial, uint8_t* __restrict__ q,
                 int64_t ldq, float* __restrict__ s_out, float* __restrict__ s_rows) {
    __shared__ float red[kThreads / 32];
    pdl_launch_dependents();
    pdl_wait_primary();
    float m = 0.0f;
    for (int i = threadIdx.x; i < n_partial; i += kThreads) m = fmaxf(m, partial[i]);
    const float s = scale_of(block_max(m, red));
    if (blockIdx.x == 0 && threadIdx.x == 0) *s_out = s;
    // last use of x: read it back from the end (the lines the first pass
    // touched last first), evict-first, and write the codes evict-first
    const uint64_t pol = policy_evict_first();
    quant_chunks<true>(x, R, K, ldx, s, q, ldq, pol, pol, true);
    if (s_rows) fill_rows(s_rows, R, s);
}

// KV-cache write: x [T, H, D] bf16 -> cache[slot[t], h, :] E4M3 with scale
// scale[h * scale_stride]; slot < 0 skips the token.
__global__ void __launch_bounds__(kThreads)
    kv_cache_quant(const uint16_t* __restrict__ x, int64_t T, int64_t H, int64_t D,
                   const float* __restrict__ scale, int64_t scale_stride,
                   const int64_t* __restrict__ slot, uint8_t* __restrict__ cache,
                   int64_t n_slots) {
    pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t C = D >> 4;  // chunks per head
    const int64_t total = T * H * C;
    const uint32_t C32 = static_cast<uint32_t>(C), H32 = static_cast<uint32_t>(H);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        // x is contiguous [T, H, D]: chunk i starts at element 16 i.  The
        // source is loaded before the slot is known (the slot only decides
        // where, or whether, the codes go), and the index arithmetic is
        // 32-bit whenever the chunk count allows.
        const uint4* src = reinterpret_cast<const uint4*>(x + i * 16);
        const uint4 a = __ldg(src), b = __ldg(src + 1);
        uint32_t c, h;
        int64_t t;
        if (total <= 0xFFFFFFFFll) {
            const uint32_t i32 = static_cast<uint32_t>(i);
            const uint32_t th = i32 / C32;  // token * H + head
            c = i32 - th * C32;
            const uint32_t t32 = th / H32;
            h = th - t32 * H32;
            t = t32;
        } else {
            const int64_t th = i / C;
            c = static_cast<uint32_t>(i - th * C);
            t = th / H;
            h = static_cast<uint32_t>(th - t * H);
        }
        const int64_t row = slot ? __ldg(slot + t) : t;
        if (row < 0 || row >= n_slots) continue;
        const float s = __ldg(scale + h * scale_stride);
        *reinterpret_cast<uint4*>(cache + (row * H + h) * D + c * 16) =
            quant16v(a, b, divisor_of(s));
    }
}

// A layer's keys and values in one launch: x0 -> cache0 with scale0 and x1
// -> cache1 with scale1, the same slots.  Each thread takes chunk i of both
// tensors, so one index computation and one slot load serve two chunks and
// four 16-byte loads are in flight per thread (measured 20% faster than two
// launches of the kernel above).
__global__ void __launch_bounds__(kThreads)
    kv_cache_quant_pair(const uint16_t* __restrict__ x0, const uint16_t* __restrict__ x1,
                        int64_t T, int64_t H, int64_t D, const float* __restrict__ scale0,
                        const float* __restrict__ scale1, int64_t scale_stride,
                        const int64_t* __restrict__ slot, uint8_t* __restrict__ cache0,
                        uint8_t* __restrict__ cache1, int64_t n_slots) {
    pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t C = D >> 4;  // chunks per head
    const int64_t total = T * H * C;
    const uint32_t C32 = static_cast<uint32_t>(C), H32 = static_cast<uint32_t>(H);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
        const uint4* src0 = reinterpret_cast<const uint4*>(x0 + i * 16);
        const uint4* src1 = reinterpret_cast<const uint4*>(x1 + i * 16);
        const uint4 a0 = __ldg(src0), b0 = __ldg(src0 + 1), a1 = __ldg(src1), b1 = __ldg(src1 + 1);
        uint32_t c, h;
        int64_t t;
        if (total <= 0xFFFFFFFFll) {
            const uint32_t i32 = static_cast<uint32_t>(i);
            const uint32_t th = i32 / C32;  // token * H + head
            c = i32 - th * C32;
            const uint32_t t32 = th / H32;
            h = th - t32 * H32;
            t = t32;
        } else {
            const int64_t th = i / C;
            c = static_cast<uint32_t>(i - th * C);
            t = th / H;
            h = static_cast<uint32_t>(th - t * H);
        }
        const int64_t row = slot ? __ldg(slot + t) : t;
        if (row < 0 || row >= n_slots) continue;
        const int64_t off = (row * H + h) * D + c * 16;
        *reinterpret_cast<uint4*>(cache0 + off) =
            quant16v(a0, b0, divisor_of(__ldg(scale0 + h * scale_stride)));
        *reinterpret_cast<uint4*>(cache1 + off) =
            quant16v(a1, b1, divisor_of(__ldg(scale1 + h * scale_stride)));
    }
}

// Block-wise activation scales: one scale per token per 128 inputs.  Eight
// consecutive lanes own a group (one 16-element chunk each), so a warp covers
// four groups; the loop runs per warp (uniform trip count) and the group
// maximum is a three-step butterfly within the eight lanes.
__global__ void __launch_bounds__(kThreads)
    quant_groups(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ldx,
                 uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s, int64_t KB) {
    pdl_launch_dependents();
    pdl_wait_primary();
    const int lane = lane_id();
    const int sub = lane & 7;
    const int64_t groups = R * KB;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t base = (static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5)) * 4;
         base < groups; base += warps * 4) {
        const int64_t g = base + (lane >> 3);
        const int64_t r = g < groups ? g / KB : 0, kb = g - r * KB;
        const int64_t k = kb * kGroup + sub * 16;
        const bool live = g < groups && k < K;
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        const uint4* src = reinterpret_cast<const uint4*>(x + r * ldx + k);
        if (live) {
            a = __ldg(src);
            b = __ldg(src + 1);
        }
        float m = amax8(b, amax8(a, 0.0f));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const float sc = scale_of(m);
        if (live) {
            const Divisor dv = divisor_of(sc);
            const uint2 qa = quant8<true>(a, dv), qb = quant8<true>(b, dv);
            *reinterpret_cast<uint4*>(q + r * ldq + k) = make_uint4(qa.x, qa.y, qb.x, qb.y);
            if (sub == 0) s[r * KB + kb] = sc;
        }
    }
}

// Block-wise weight scales: one CTA per 128 x 128 block (partial at the
// edges); each thread holds four 16-element chunks (rows t/8 + 32 i, chunk
// t % 8) in registers between the block maximum and the quantization.
__global__ void __launch_bounds__(kThreads)
    quant_weight_blocks(const uint16_t* __restrict__ w, int64_t N, int64_t K, int64_t ldw,
                        uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s) {
    __shared__ float red[kThreads / 32];
    pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t kb = blockIdx.x, nb = blockIdx.y, KB = gridDim.x;
    const int64_t k = kb * kGroup + (threadIdx.x & 7) * 16;
    uint4 v[4][2];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t n = nb * kGroup + (threadIdx.x >> 3) + 32 * i;
        v[i][0] = v[i][1] = make_uint4(0, 0, 0, 0);
        if (n < N && k < K) {
            const uint4* src = reinterpret_cast<const uint4*>(w + n * ldw + k);
            v[i][0] = __ldg(src);
            v[i][1] = __ldg(src + 1);
        }
        m = amax8(v[i][1], amax8(v[i][0], m));
    }
    const float sc = scale_of(block_max(m, red));
    const Divisor dv = divisor_of(sc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t n = nb * kGroup + (threadIdx.x >> 3) + 32 * i;
        if (n < N && k < K) {
            const uint2 qa = quant8<true>(v[i][0], dv), qb = quant8<true>(v[i][1], dv);
            *reinterpret_cast<uint4*>(q + n * ldq + k) = make_uint4(qa.x, qa.y, qb.x, qb.y);
        }
    }
    if (threadIdx.x == 0) s[nb * KB + kb] = sc;
}

template <typename... Params, typename... Args>
cudaError_t launch(void (*kernel)(Params...), int64_t grid, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

int64_t grid_for(int64_t chunks, int num_sms) {
    const int64_t want = (chunks + kThreads - 1) / kThreads;
    int64_t cap = static_cast<int64_t>(num_sms) * 8;  // 8 x 256 threads per SM
    if (cap > kMaxTensorPartials) cap = kMaxTensorPartials;
    return want < 1 ? 1 : (want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_quant_given_scale(const void* x, int64_t R, int64_t K, int64_t ldx,
                                     const float* s, uint8_t* q, int64_t ldq, float* s_rows,
                                     int num_sms, cudaStream_t st) {
    // rows held in registers, as the per-token quantizer (measured faster than
    // the grid-stride loop); the loop takes empty and very long rows
    if (K > 0) {
        const cudaError_t e = launch_quant_rows_given(x, R, K, ldx, q, ldq, s, s_rows, st);
        if (e != cudaErrorNotSupported) return e;
    }
    return launch(quant_given_scale, grid_for(R * (K >> 4), num_sms), st,
                  static_cast<const uint16_t*>(x), R, K, ldx, s, q, ldq, s_rows);
}

cudaError_t launch_quant_per_tensor(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                                    int64_t ldq, float* s_out, float* s_rows, float* partial,
                                    int num_sms, cudaStream_t st) {
    const int64_t grid = grid_for(R * (K >> 4), num_sms);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    cudaError_t e = launch(tensor_amax_partial, grid, st, xb, R, K, ldx, partial);
    if (e != cudaSuccess) return e;
    return launch(tensor_quant, grid, st, xb, R, K, ldx, static_cast<const float*>(partial),
                  static_cast<int>(grid), q, ldq, s_out, s_rows);
}

cudaError_t launch_kv_cache_quant(const void* x0, const void* x1, int64_t T, int64_t H,
                                  int64_t D, const float* scale0, const float* scale1,
                                  int64_t scale_stride, const int64_t* slot, uint8_t* cache0,
                                  uint8_t* cache1, int64_t n_slots, int num_sms,
                                  cudaStream_t st) {
    const int64_t grid = grid_for(T * H * (D >> 4), num_sms);
    const uint16_t *p0 = static_cast<const uint16_t*>(x0), *p1 = static_cast<const uint16_t*>(x1);
    if (x1)
        return launch(kv_cache_quant_pair, grid, st, p0, p1, T, H, D, scale0, scale1,
                      scale_stride, slot, cache0, cache1, n_slots);
    return launch(kv_cache_quant, grid, st, p0, T, H, D, scale0, scale_stride, slot, cache0,
                  n_slots);
}

cudaError_t launch_quant_groups(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                                int64_t ldq, float* s, int num_sms, cudaStream_t st) {
    const int64_t KB = (K + kGroup - 1) / kGroup;
    const int64_t grid = grid_for(R * KB * 8, num_sms);  // eight threads per group
    return launch(quant_groups, grid, st, static_cast<const uint16_t*>(x), R, K, ldx, q, ldq, s,
                  KB);
}

cudaError_t launch_quant_weight_blocks(const void* w, int64_t N, int64_t K, int64_t ldw,
                                       uint8_t* q, int64_t ldq, float* s, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>((K + kGroup - 1) / kGroup),
                       static_cast<unsigned>((N + kGroup - 1) / kGroup));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quant_weight_blocks, static_cast<const uint16_t*>(w), N, K,
                              ldw, q, ldq, s);
}

}  // namespace fp8k
