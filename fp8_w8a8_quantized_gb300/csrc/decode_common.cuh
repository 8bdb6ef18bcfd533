// Shape constants and helpers shared by the decode-sized (weight-streaming)
// GEMMs: per-token x per-channel scales (gemm_decode.cu) and block-wise
// scales (gemm_blockwise.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace fp8k {
namespace decode {

constexpr int BNW = 128;  // weight rows per slab (tcgen05 M)
constexpr int BK = 128;   // bytes (= E4M3 elements) of K per stage
constexpr int KSTEP = 32; // K of one tcgen05.mma kind::f8f6f4
constexpr int kThreads = 192;
constexpr uint32_t W_TILE = BNW * BK;
constexpr int kMaxSplits = 8;
// CTAs per SM the shared-memory footprint is sized for.  Several small CTAs
// per SM keep more independent TMA producers busy than one deep ring does
// (measured on GB300: 3 per SM streams weights fastest).
constexpr int kCtasPerSm = 3;
constexpr uint32_t kSmemPerSm = 228 * 1024;
constexpr uint32_t kCtaSmem = kSmemPerSm / kCtasPerSm - 1024;  // 1 KB reserved per CTA
constexpr int kL2PrefetchBlocks = 8;  // k-blocks of W prefetched into L2 before the wait

// Accumulator columns of one warp's 32 TMEM lanes -> registers.
template <int MT>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* out) {
    if constexpr (MT == 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) out[j] = __uint_as_float(r[j]);
    } else {
#pragma unroll
        for (int h = 0; h < MT / 32; ++h) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + h * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) out[h * 32 + j] = __uint_as_float(r[j]);
        }
    }
}

// k-blocks [kb0, kb0 + nkb) of split `rank` out of `splits` over nk blocks:
// the first nk % splits splits take one block more.
__host__ __device__ __forceinline__ void split_range(int rank, int nk, int splits, int* kb0,
                                                     int* nkb) {
    const int per = nk / splits, rem = nk % splits;
    *kb0 = rank * per + (rank < rem ? rank : rem);
    *nkb = per + (rank < rem ? 1 : 0);
}

// K-split count S (cluster size): as many clusters x splits as fill the GPU
// with kCtasPerSm CTAs per SM in whole waves, at least 2 k-blocks per split,
// at most kMaxSplits.
inline int choose_splits(int n_tiles, int nk, int num_sms) {
    const int slots = kCtasPerSm * num_sms;
    int best = 1;
    double best_eff = -1.0;
    for (int s = 1; s <= kMaxSplits; ++s) {
        if (s > 1 && nk < 2 * s) break;
        const int ctas = n_tiles * s;
        const int waves = (ctas + slots - 1) / slots;
        const double eff = static_cast<double>(ctas) / (static_cast<double>(waves) * slots);
        if (eff > best_eff + 0.02) {
            best_eff = eff;
            best = s;
        }
    }
    return best;
}

}  // namespace decode
}  // namespace fp8k
