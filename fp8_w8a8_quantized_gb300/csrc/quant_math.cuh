// E4M3 quantization arithmetic shared by the per-token quantizer (quant.cu)
// and the quantizers with other scale granularities (quant_variants.cu), so
// all produce the same bytes:
//   amax = max |x| (exact in fp32), s = amax / 448 (IEEE fp32 division) or 1,
//   q = E4M3_rn_satfinite(x / s) (IEEE fp32 quotient).
// "FP8 Inference Explained, in depth", "Scales and their granularity";
// "Quantization: FP8 inference and KV-cache quantization", "Dynamic scales or
// static scales".
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8k {

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ float amax2(uint32_t u, float m) {
    return fmaxf(fmaxf(m, fabsf(bf16lo(u))), fabsf(bf16hi(u)));
}

__device__ __forceinline__ float amax8(const uint4& v, float m) {
    return amax2(v.w, amax2(v.z, amax2(v.y, amax2(v.x, m))));
}

// Two fp32 values -> two E4M3 codes (RN, saturating to +-448); `lo` lands in
// the low byte (lower address).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// One bf16 pair -> two codes in the low 16 bits.
__device__ __forceinline__ uint32_t quant2(uint32_t u, float s) {
    return cvt_e4m3x2(__fdiv_rn(bf16lo(u), s), __fdiv_rn(bf16hi(u), s));
}

// Four bf16 values (8 bytes) -> four codes packed in one 32-bit word.
__device__ __forceinline__ uint32_t quant4(const uint2& v, float s) {
    return quant2(v.x, s) | (quant2(v.y, s) << 16);
}

// Eight bf16 values (16 bytes) -> eight codes packed in two 32-bit words.
__device__ __forceinline__ uint2 quant8(const uint4& v, float s) {
    return make_uint2(quant2(v.x, s) | (quant2(v.y, s) << 16),
                      quant2(v.z, s) | (quant2(v.w, s) << 16));
}

__device__ __forceinline__ float scale_of(float amax) {
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

}  // namespace fp8k
