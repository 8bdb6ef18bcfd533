// RMSNorm with the per-token quantizer fused into it: the amax reduction of
// the dynamic activation scale done by the kernel that produces the
// activations ("FP8 Inference Explained, in depth", "Scales and their
// granularity": engines typically fuse it into the preceding kernel; "What
// stays in higher precision": normalisation stays in 16/32-bit).
//
// For every row r of x [R, K] (bf16) and the weights g [K] (bf16):
//   ss   = sum_k x_k^2                         (fp32, see below)
//   inv  = fl32(1 / fl32(sqrt(fl32(fl32(ss / K) + eps))))
//   y_k  = bf16_rn(fl32(fl32(x_k * inv) * g_k))   -- the normalised row
//   s    = fl32(amax_k |y_k| / 448) (1 if zero), q_k = E4M3(fl32(y_k / s))
// i.e. the per-token quantizer applied to the bf16 row an unfused RMSNorm
// would have written; y can also be written out.
//
// Same work layout as quant.cu (G threads per row, VPT 16-element chunks per
// thread held in registers; x is read once).  The sum of squares is each
// thread's chunks in order into two running sums (even and odd elements,
// one packed FMA per pair) added at the end, then a butterfly over the warp,
// then the warps' partial sums in order: at most 8 VPT + 1 + 5 + 31 < 128
// roundings of non-negative terms on any path, so the fp32 sum is within
// 128 * 2^-24 = 2^-17 of the exact one (relative); every later step is an
// IEEE operation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8k {
namespace {

constexpr int kBlock = 256;
constexpr int kVPT = 2;
constexpr int64_t kLatencyChunks = 152 * 1024;

template <int G, int B, bool kMax>
__device__ __forceinline__ float group_reduce(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = kMax ? fmaxf(v, w) : __fadd_rn(v, w);
    }
    if constexpr (G > 32) {
        constexpr int WPG = G / 32;
        const int warp = threadIdx.x >> 5;
        if (lane_id() == 0) red[warp] = v;
        __syncthreads();
        const int first = (warp / WPG) * WPG;
        v = red[first];
#pragma unroll
        for (int w = 1; w < WPG; ++w) v = kMax ? fmaxf(v, red[first + w]) : __fadd_rn(v, red[first + w]);
        __syncthreads();  // red is reused by the next reduction
    }
    return v;
}

// Sum of squares of a bf16 pair into two running sums (the low and the
// high lanes), one packed f32x2 FMA; a * a is exact for a bf16 value.
__device__ __forceinline__ void sumsq2(uint32_t w, float& s0, float& s1) {
    const float a = bf16lo(w), b = bf16hi(w);
    fma2(s0, s1, a, b, a, b);
}

__device__ __forceinline__ void sumsq8(const uint4& v, float& s0, float& s1) {
    sumsq2(v.x, s0, s1);
    sumsq2(v.y, s0, s1);
    sumsq2(v.z, s0, s1);
    sumsq2(v.w, s0, s1);
}

// Two fp32 values -> a bf16 pair (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// One bf16 pair normalised (x * inv * g, each product rounded to fp32, then
// bf16), the products as packed f32x2 multiplies.
__device__ __forceinline__ uint32_t norm2(uint32_t xw, uint32_t gw, float inv) {
    float lo, hi;
    mul2(lo, hi, bf16lo(xw), bf16hi(xw), inv, inv);
    float ylo, yhi;
    mul2(ylo, yhi, lo, hi, bf16lo(gw), bf16hi(gw));
    return bf16x2_rn(ylo, yhi);
}

// Normalise 8 values in place; returns the running max |y|.
__device__ __forceinline__ float norm8(uint4& v, const uint4& g, float inv, float m) {
    v.x = norm2(v.x, g.x, inv);
    v.y = norm2(v.y, g.y, inv);
    v.z = norm2(v.z, g.z, inv);
    v.w = norm2(v.w, g.w, inv);
    return amax8(v, m);
}

// CTAs of kBlock threads are held to six per SM worth of registers (40 a
// thread, no spill): the kernel is bound by issue and latency, and more
// resident warps hide more of it (8192 x 4096: 4240 GB/s at four CTAs per
// SM, 4600 at five, 4770 at six with gamma loaded after the sum of squares).
template <int G, int VPT>
__global__ void __launch_bounds__(G > kBlock ? G : kBlock, G > kBlock ? 1 : 6)
    rmsnorm_quant_rows(const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps,
                       int64_t R, int64_t K, int64_t ldx, uint8_t* __restrict__ q, int64_t ldq,
                       float* __restrict__ s, uint16_t* __restrict__ y_out) {
    constexpr int B = G > kBlock ? G : kBlock;
    constexpr int ROWS = B / G;
    __shared__ float red[B / 32];
    pdl_launch_dependents();
    pdl_wait_primary();

    const int64_t row = static_cast<int64_t>(blockIdx.x) * ROWS + threadIdx.x / G;
    const int t = threadIdx.x % G;
    const bool live = row < R;
    const int64_t C = K >> 4;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (live ? row : 0) * ldx);
    const uint4* gr = reinterpret_cast<const uint4*>(gamma);

    // The matching gamma chunks are loaded together with x where registers
    // allow (one chunk per thread, or two in the large CTAs), so no load
    // sits between the two reductions; the register-bounded two-chunk CTAs
    // load gamma after the sum of squares instead (an L1 hit: every row
    // reads the same gamma).
    constexpr bool kPreG = VPT == 1 || (G > kBlock && VPT <= 2);
    uint4 v[VPT][2], gv[kPreG ? VPT : 1][2];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t c = t + static_cast<int64_t>(i) * G;
        if (live && c < C) {
            v[i][0] = __ldg(xr + 2 * c);
            v[i][1] = __ldg(xr + 2 * c + 1);
            if constexpr (kPreG) {
                gv[i][0] = __ldg(gr + 2 * c);
                gv[i][1] = __ldg(gr + 2 * c + 1);
            }
        }
    }
    float s1 = 0.0f;  // ss collects the low lanes, s1 the high lanes
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t c = t + static_cast<int64_t>(i) * G;
        if (live && c < C) {
            sumsq8(v[i][0], ss, s1);
            sumsq8(v[i][1], ss, s1);
        }
    }
    ss = __fadd_rn(ss, s1);
    ss = group_reduce<G, B, false>(ss, red);
    const float mean = __fdiv_rn(ss, static_cast<float>(K));
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));

    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t c = t + static_cast<int64_t>(i) * G;
        if (live && c < C) {
            if constexpr (kPreG) {
                m = norm8(v[i][0], gv[i][0], inv, m);
                m = norm8(v[i][1], gv[i][1], inv, m);
            } else {
                m = norm8(v[i][0], __ldg(gr + 2 * c), inv, m);
                m = norm8(v[i][1], __ldg(gr + 2 * c + 1), inv, m);
            }
        }
    }
    m = group_reduce<G, B, true>(m, red);
    const float sc = scale_of(m);
    const Divisor dv = divisor_of(sc);
    if (!live) return;
    uint4* qr = reinterpret_cast<uint4*>(q + row * ldq);
    uint4* yr = y_out ? reinterpret_cast<uint4*>(y_out + row * K) : nullptr;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t c = t + static_cast<int64_t>(i) * G;
        if (c < C) {
            const uint2 a = quant8<true>(v[i][0], dv);
            const uint2 b = quant8<true>(v[i][1], dv);
            qr[c] = make_uint4(a.x, a.y, b.x, b.y);
            if (yr) {
                yr[2 * c] = v[i][0];
                yr[2 * c + 1] = v[i][1];
            }
        }
    }
    if (t == 0) s[row] = sc;
}

template <int G, int VPT>
cudaError_t launch_rows(const uint16_t* x, const uint16_t* g, float eps, int64_t R, int64_t K,
                        int64_t ldx, uint8_t* q, int64_t ldq, float* s, uint16_t* y,
                        cudaStream_t st) {
    constexpr int B = G > kBlock ? G : kBlock;
    constexpr int ROWS = B / G;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>((R + ROWS - 1) / ROWS));
    cfg.blockDim = dim3(B);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rmsnorm_quant_rows<G, VPT>, x, g, eps, R, K, ldx, q, ldq, s,
                              y);
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const void* x, const void* gamma, float eps, int64_t R,
                                 int64_t K, int64_t ldx, uint8_t* q, int64_t ldq, float* s,
                                 void* y, cudaStream_t st) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    const uint16_t* gb = static_cast<const uint16_t*>(gamma);
    uint16_t* yb = static_cast<uint16_t*>(y);
    const int64_t C = K / 16;
    if (R * C <= kLatencyChunks) {
        if (C <= 32) return launch_rows<32, 1>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
        if (C <= 64) return launch_rows<64, 1>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
        if (C <= 128) return launch_rows<128, 1>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
        if (C <= 256) return launch_rows<256, 1>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
        if (C <= 512) return launch_rows<512, 1>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
        if (C <= 1024) return launch_rows<1024, 1>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
        if (C <= 2048) return launch_rows<1024, 2>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    }
    if (C <= 32 * kVPT) return launch_rows<32, kVPT>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    if (C <= 64 * kVPT) return launch_rows<64, kVPT>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    if (C <= 128 * kVPT) return launch_rows<128, kVPT>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    if (C <= 256 * kVPT) return launch_rows<256, kVPT>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    if (C <= 512 * kVPT) return launch_rows<512, kVPT>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    if (C <= 1024 * kVPT)
        return launch_rows<1024, kVPT>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    if (C <= 1024 * 4) return launch_rows<1024, 4>(xb, gb, eps, R, K, ldx, q, ldq, s, yb, st);
    return cudaErrorInvalidValue;  // K > 65536: rejected by the caller
}

}  // namespace fp8k
