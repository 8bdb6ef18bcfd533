// E4M3 quantization arithmetic shared by the per-token quantizer (quant.cu)
// and the quantizers with other scale granularities (quant_variants.cu), so
// all produce the same bytes:
//   amax = max |x| (exact in fp32), s = amax / 448 (IEEE fp32 division) or 1,
//   q = E4M3_rn_satfinite(x / s) (the correctly rounded fp32 quotient).
// "FP8 Inference Explained, in depth", "Scales and their granularity";
// "Quantization: FP8 inference and KV-cache quantization", "Dynamic scales or
// static scales".
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace fp8k {

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// max(|a|, |b|) per bf16 lane (exact); the sign bits of the result are
// the XOR of the inputs' and carry no meaning.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// max(m, |x_0|, ..., |x_7|) over eight bf16 values, exact: the maxima are
// taken on bf16 pairs, then the two lanes are widened (exactly) to fp32.
__device__ __forceinline__ float amax8(const uint4& v, float m) {
    const uint32_t a = absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w)) & 0x7FFF7FFFu;
    return fmaxf(m, fmaxf(bf16lo(a), bf16hi(a)));
}

// Two fp32 values -> two E4M3 codes (RN, saturating to +-448); `lo` lands in
// the low byte (lower address).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// x / s rounded to nearest fp32, for a scale s > 0 shared by many x,
// without a division per element.  Markstein's division theorem (P.
// Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990; also "IA-64 and
// Elementary Functions", 2000): with r = RN(1/s) and a quotient q0 within
// one ulp of x/s (here q0 = RN(x * r)), the residual e = x - s * q0 is exact
// in one fused multiply-add and RN(q0 + e * r) = RN(x / s) whenever the
// quotient is a normal number.  Quotients below the normal range can only
// become an E4M3 zero, where an ulp does not matter; the sign of zero is
// that of x (s > 0), as for the IEEE quotient.  A quotient that overflows
// (a small static scale) stays infinite and saturates like the IEEE one.  A
// scale whose reciprocal is not a normal number (s below the normal range or
// above 2^126), or that is not finite, takes the IEEE division.
struct Divisor {
    float s, ns, r, nr;  // s, -s, RN(1/s), -RN(1/s)
    bool ieee;
};

__device__ __forceinline__ Divisor divisor_of(float s) {
    Divisor d;
    d.s = s;
    d.ns = -s;
    d.r = __frcp_rn(s);
    d.nr = -d.r;
    d.ieee = !(s >= 1.17549435e-38f && s <= 8.50705917e37f);  // [2^-126, 2^126]
    return d;
}

// RN(x / s) for a scale on the fast path (d.ieee false): the method for one
// value; quant2 below runs it on two values per instruction.
__device__ __forceinline__ float div_rn(float x, const Divisor& d) {
    const float q0 = __fmul_rn(x, d.r);
    const float e = __fmaf_rn(-q0, d.s, x);
    const float q = copysignf(__fmaf_rn(e, d.r, q0), x);
    return isinf(q0) ? q0 : q;
}

// One bf16 pair -> two codes in the low 16 bits: div_rn on both values in
// packed f32x2 fused multiply-adds (each lane an IEEE fp32 FMA, so the same
// bits).  The pair is unpacked negated, z = -x (one integer multiply-add and
// one logic op: z_lo = (u << 16) + 2^31, z_hi = (u & 0xffff0000) ^ 2^31), and
// the steps run on z with -r:
//   q0 = RN(z * (-r))         = RN(x * r)       (the same product)
//   e' = RN(q0 * s + z)       = -(x - s * q0)   (exact)
//   y  = RN(e' * (-r) + q0)   = RN(q0 + e * r)  (the same fused sum)
// so every nonzero result has the bits of div_rn.  The sign of a zero
// result comes out right without a copysign: x = -0 gives q0 = -0,
// e' = +0 and y = (+0)(-r) + (-0) = -0; x = +0 gives +0; a nonzero x whose
// quotient underflows gives RN(x * r) = zero with the sign of x.  kBounded:
// the scale comes from these values' own maximum (s = amax / 448), so |q0|
// stays near 448 and cannot overflow; otherwise an infinite q0 is kept, as
// in div_rn.
template <bool kBounded>
__device__ __forceinline__ uint32_t quant2(uint32_t u, const Divisor& d) {
    const float z0 = __uint_as_float(u * 0x10000u + 0x80000000u);
    const float z1 = __uint_as_float((u & 0xFFFF0000u) ^ 0x80000000u);
    float q0, q1;
    mul2(q0, q1, z0, z1, d.nr, d.nr);
    float e0 = z0, e1 = z1;
    fma2(e0, e1, q0, q1, d.s, d.s);  // s * q0 - x, exact
    float y0 = q0, y1 = q1;
    fma2(y0, y1, e0, e1, d.nr, d.nr);
    if (!kBounded) {
        y0 = isinf(q0) ? q0 : y0;
        y1 = isinf(q1) ? q1 : y1;
    }
    return cvt_e4m3x2(y0, y1);
}

__device__ __forceinline__ uint32_t quant2_ieee(uint32_t u, float s) {
    return cvt_e4m3x2(__fdiv_rn(bf16lo(u), s), __fdiv_rn(bf16hi(u), s));
}

// Scales outside the fast path's range: out of line, so that the common
// path keeps its registers.
static __device__ __noinline__ uint2 quant8_ieee(uint4 v, float s) {
    return make_uint2(quant2_ieee(v.x, s) | (quant2_ieee(v.y, s) << 16),
                      quant2_ieee(v.z, s) | (quant2_ieee(v.w, s) << 16));
}

// Eight bf16 values (16 bytes) -> eight codes packed in two 32-bit words.
// kBounded as for quant2: true where s = amax / 448 of a set holding v.
template <bool kBounded = false>
__device__ __forceinline__ uint2 quant8(const uint4& v, const Divisor& d) {
    if (d.ieee) return quant8_ieee(v, d.s);
    return make_uint2(quant2<kBounded>(v.x, d) | (quant2<kBounded>(v.y, d) << 16),
                      quant2<kBounded>(v.z, d) | (quant2<kBounded>(v.w, d) << 16));
}

__device__ __forceinline__ float scale_of(float amax) {
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

}  // namespace fp8k
