// Dynamic per-row E4M3 quantization: one scale per row (a token of X, or an
// output channel of W).
//
// Computes, for every row r of a bf16 matrix [R, K]:
//   amax_r = max_k |x[r,k]|                      (exact, fp32)
//   s_r    = amax_r / 448  (IEEE fp32 division), or 1 if amax_r == 0
//   q[r,k] = E4M3_rn_satfinite(x[r,k] / s_r)     (IEEE fp32 quotient)
// following "FP8 Inference Explained, in depth", "Scales and their
// granularity" (s = amax / 448, x_fp8 = round(x / s)) and "Quantization: FP8
// inference and KV-cache quantization", "Dynamic scales or static scales"
// (per-token scales; saturating conversion).
//
// Layout of the work: a group of G threads owns a row; each thread keeps up
// to VPT 16-element chunks (two 16-byte loads each) of the row in registers
// between the amax pass and the quantize pass, so X is read from HBM once.
// The amax reduction is a butterfly of warp shuffles, then (G > 32) a pass
// through shared memory.  Codes leave as one 16-byte store per chunk.
// Small problems (decode batches) use one chunk per thread, so each
// thread's serial work -- the latency of the call -- is as short as
// possible; large ones use two (four for rows longer than 32768), the
// measured optimum between occupancy and bytes in flight per thread.  Very
// long rows (K > 65536) take a variant that streams the row twice.
//
// Memory-bound: 2 bytes in + 1 byte out per element (+4 bytes per row).
// The scale is an IEEE division; each quotient x / s is the correctly rounded
// fp32 value, from one reciprocal per row and a multiply and two fused
// multiply-adds per element (quant_math.cuh).  Nothing here is compiled with
// fast-math or flush-to-zero, so results are bit-identical to the fp32
// definition above.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8k {
namespace {

constexpr int kBlock = 256;  // threads per CTA for G <= 256
constexpr int kVPT = 2;      // 16-element chunks per thread, large problems (measured best)
// Total 16-element chunks up to which the one-chunk-per-thread (latency)
// layout is used: about one wave of 1024 threads per SM on 152 SMs.
constexpr int64_t kLatencyChunks = 152 * 1024;

// Read-once 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Max over the G threads of a row group.  `red` holds one float per warp.
template <int G, int B>
__device__ __forceinline__ float group_max(float m, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if constexpr (G > 32) {
        constexpr int WPG = G / 32;  // warps per group
        const int warp = threadIdx.x >> 5;
        if (lane_id() == 0) red[warp] = m;
        __syncthreads();
        // every lane reads one warp maximum of its group; a shuffle tree over
        // WPG lanes combines them (max is exact in any order)
        const int first = (warp / WPG) * WPG;
        m = red[first + (lane_id() & (WPG - 1))];
#pragma unroll
        for (int o = WPG / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    }
    return m;
}

// kGiven: the scale is *s_given for every row (a static, calibrated scale:
// no maximum is taken, and quotients beyond 448 saturate); s (optional, may
// be null) receives it per row.
template <int G, int VPT, bool kGiven = false>
__global__ void __launch_bounds__(G > kBlock ? G : kBlock)
    quant_rows_regs(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ldx,
                    uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s,
                    const float* __restrict__ s_given = nullptr) {
    constexpr int B = G > kBlock ? G : kBlock;
    constexpr int ROWS = B / G;
    __shared__ float red[B / 32];
    // Launched as a programmatic dependent: the next kernel may start at
    // once (it reads nothing but L2 prefetches before its own wait, which
    // returns after this grid has completed); this one waits for its
    // predecessor before touching memory.
    pdl_launch_dependents();
    pdl_wait_primary();

    const int64_t row = static_cast<int64_t>(blockIdx.x) * ROWS + threadIdx.x / G;
    const int t = threadIdx.x % G;
    const bool live = row < R;
    const int64_t C = K >> 4;  // 16-element chunks per row

    const uint4* xr = reinterpret_cast<const uint4*>(x + (live ? row : 0) * ldx);
    uint4 v[VPT][2];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t c = t + static_cast<int64_t>(i) * G;
        if (live && c < C) {
            v[i][0] = ld_stream(xr + 2 * c);
            v[i][1] = ld_stream(xr + 2 * c + 1);
            if constexpr (!kGiven) m = amax8(v[i][1], amax8(v[i][0], m));
        }
    }
    float sc;
    if constexpr (kGiven) {
        sc = __ldg(s_given);
    } else {
        m = group_max<G, B>(m, red);
        sc = scale_of(m);
    }
    if (!live) return;
    const Divisor dv = divisor_of(sc);
    uint4* qr = reinterpret_cast<uint4*>(q + row * ldq);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t c = t + static_cast<int64_t>(i) * G;
        if (c < C) {
            const uint2 a = quant8<!kGiven>(v[i][0], dv);
            const uint2 b = quant8<!kGiven>(v[i][1], dv);
            qr[c] = make_uint4(a.x, a.y, b.x, b.y);
        }
    }
    if (t == 0 && s) s[row] = sc;
}

// Rows longer than the register path holds: stream the row twice (the
// second pass mostly hits L2).
__global__ void __launch_bounds__(1024)
    quant_rows_stream(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ldx,
                      uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s) {
    __shared__ float red[32];
    pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t row = blockIdx.x;
    const int64_t C = K >> 4;
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * ldx);
    float m = 0.0f;
    for (int64_t c = threadIdx.x; c < C; c += 1024) {
        const uint4 a = __ldg(xr + 2 * c), b = __ldg(xr + 2 * c + 1);
        m = amax8(b, amax8(a, m));
    }
    m = group_max<1024, 1024>(m, red);
    const float sc = scale_of(m);
    const Divisor dv = divisor_of(sc);
    uint4* qr = reinterpret_cast<uint4*>(q + row * ldq);
    for (int64_t c = threadIdx.x; c < C; c += 1024) {
        const uint2 a = quant8<true>(ld_stream(xr + 2 * c), dv);
        const uint2 b = quant8<true>(ld_stream(xr + 2 * c + 1), dv);
        qr[c] = make_uint4(a.x, a.y, b.x, b.y);
    }
    if (threadIdx.x == 0) s[row] = sc;
}

// K == 0: an empty row has amax 0, so its scale is 1.
__global__ void fill_ones(float* s, int64_t R) {
    pdl_launch_dependents();
    pdl_wait_primary();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < R) s[i] = 1.0f;
}

// Every kernel here waits (griddepcontrol.wait) before reading or writing
// global memory, so it is always launched as a programmatic dependent of the
// previous kernel on the stream: its launch overlaps that kernel's tail.  It
// releases its own dependents at its start: they too touch nothing but L2
// before their own wait, which returns once this grid has completed.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), int64_t grid, int block, cudaStream_t st,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int G, int VPT, bool kGiven = false>
cudaError_t launch_regs(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                        int64_t ldq, float* s, cudaStream_t st, const float* s_given = nullptr) {
    constexpr int B = G > kBlock ? G : kBlock;
    constexpr int ROWS = B / G;
    const int64_t grid = (R + ROWS - 1) / ROWS;
    return launch_pdl(quant_rows_regs<G, VPT, kGiven>, grid, B, st, x, R, K, ldx, q, ldq, s,
                      s_given);
}

// The launch for rows of K = 16 C values: small problems (decode batches)
// one chunk per thread, large ones kVPT (four for rows longer than 32768).
// Returns cudaErrorNotSupported for rows longer than the register path holds.
template <bool kGiven>
cudaError_t dispatch_regs(const uint16_t* xb, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                          int64_t ldq, float* s, const float* s_given, cudaStream_t st) {
    const int64_t C = K / 16;
    if (R * C <= kLatencyChunks) {
        if (C <= 32) return launch_regs<32, 1, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
        if (C <= 64) return launch_regs<64, 1, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
        if (C <= 128) return launch_regs<128, 1, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
        if (C <= 256) return launch_regs<256, 1, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
        if (C <= 512) return launch_regs<512, 1, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
        if (C <= 1024) return launch_regs<1024, 1, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
        if (C <= 2048) return launch_regs<1024, 2, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    }
    if (C <= 32 * kVPT) return launch_regs<32, kVPT, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    if (C <= 64 * kVPT) return launch_regs<64, kVPT, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    if (C <= 128 * kVPT)
        return launch_regs<128, kVPT, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    if (C <= 256 * kVPT)
        return launch_regs<256, kVPT, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    if (C <= 512 * kVPT)
        return launch_regs<512, kVPT, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    if (C <= 1024 * kVPT)
        return launch_regs<1024, kVPT, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    if (C <= 1024 * 4) return launch_regs<1024, 4, kGiven>(xb, R, K, ldx, q, ldq, s, st, s_given);
    return cudaErrorNotSupported;
}

}  // namespace

// Rows with a given scale (the static quantizer): the row layout of the
// per-token quantizer without its maximum.  Rows longer than the register
// path holds return cudaErrorNotSupported (the caller's grid-stride kernel
// takes them).  Preconditions as below, and K > 0; s_rows may be null.
cudaError_t launch_quant_rows_given(const void* x, int64_t R, int64_t K, int64_t ldx,
                                    uint8_t* q, int64_t ldq, const float* s_given, float* s_rows,
                                    cudaStream_t st) {
    return dispatch_regs<true>(static_cast<const uint16_t*>(x), R, K, ldx, q, ldq, s_rows,
                               s_given, st);
}

// Host launcher.  Preconditions (checked by the caller): R > 0, K % 16 == 0,
// 16-byte aligned rows, R < 2^31.
cudaError_t launch_quant_rows(const void* x, int64_t R, int64_t K, int64_t ldx, uint8_t* q,
                              int64_t ldq, float* s, cudaStream_t st) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    if (K == 0) return launch_pdl(fill_ones, (R + 255) / 256, 256, st, s, R);
    const cudaError_t e = dispatch_regs<false>(xb, R, K, ldx, q, ldq, s, nullptr, st);
    if (e != cudaErrorNotSupported) return e;
    return launch_pdl(quant_rows_stream, R, 1024, st, xb, R, K, ldx, q, ldq, s);
}

}  // namespace fp8k
