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
constexpr uint32_t kCtaSmem2 = kSmemPerSm / 2 - 1024;           // two CTAs per SM
constexpr uint32_t kCtaSmem1 = kSmemPerSm - 1024;               // one CTA per SM
constexpr int kL2PrefetchBlocks = 4;  // k-blocks of W prefetched into L2 before the wait (measured)

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

// K-split count S (cluster size): the one whose grid (n_tiles clusters of S
// CTAs) keeps the largest share of the kCtasPerSm x num_sms CTA slots busy
// over its waves, with at least 2 k-blocks per split and S <= kMaxSplits.
// A cluster must fit on the SMs of one GPC, so fewer than slots / S clusters
// of S may be resident at once: clusters[S], when known, is that number and
// sets the waves (measured on GB300: 64 clusters of 7 do not fit, 74 of 6
// do).
inline int choose_splits(int n_tiles, int nk, int num_sms, const int* clusters = nullptr,
                         int ctas_per_sm = kCtasPerSm) {
    const int slots = ctas_per_sm * num_sms;
    int best = 1;
    double best_eff = -1.0;
    for (int s = 1; s <= kMaxSplits; ++s) {
        if (s > 1 && nk < 2 * s) break;
        const int per_wave = (clusters && clusters[s] > 0) ? clusters[s] : slots / s;
        if (per_wave < 1) break;
        const int waves = (n_tiles + per_wave - 1) / per_wave;
        const double eff = static_cast<double>(n_tiles) * s / (static_cast<double>(waves) * slots);
        if (eff > best_eff + 0.02) {
            best_eff = eff;
            best = s;
        }
    }
    return best;
}

// Split count for the 32- and 64-token tiles, whose partials are pulled
// across the cluster after a barrier (the tail grows with S and waits for
// the slowest CTA): about kPullTargetCtas CTAs per layer, S = the nearest
// integer to kPullTargetCtas / n_tiles, lowered until every cluster of S is
// resident at once (clusters[S] when known) and each split has at least 2
// k-blocks.  Against the busy-slot rule: 70B decode layers at 32 tokens
// +3.1% (S = 3 / 4 / 1 / 4 instead of 5 / 6 / 1 / 6), the 8B decode step
// unchanged; targets of 192 and 224 CTAs were slower on the 8B step.
constexpr int kPullTargetCtas = 256;
inline int choose_splits_pull(int n_tiles, int nk, const int* clusters) {
    int s = (kPullTargetCtas + n_tiles / 2) / n_tiles;
    s = s < 1 ? 1 : (s > kMaxSplits ? kMaxSplits : s);
    while (s > 1 && (nk < 2 * s || (clusters && clusters[s] > 0 && clusters[s] < n_tiles))) --s;
    return s;
}

// Split count for the wide token tiles (128 and 256 tokens: two CTAs or one
// per SM, slots = ctas_per_sm x num_sms), whose per-CTA overhead (ring fill,
// a 64-128 KB partial pulled across the cluster) makes every extra wave
// expensive: the fewest waves, counted with the clusters of S that can be
// resident at once (clusters[S] when known, else slots / S), and among
// those the largest S (at least 2 k-blocks per split).  Measured on the 8B
// layers at 128 and 256 tokens it picks the fastest S of a 1..8 sweep on
// every layer, where the busy-slot rule above lost up to 1.7x.
inline int choose_splits_min_waves(int n_tiles, int nk, int slots, const int* clusters) {
    int best = 1, best_waves = 1 << 30;
    for (int s = 1; s <= kMaxSplits; ++s) {
        if (s > 1 && nk < 2 * s) break;
        const int per_wave = (clusters && clusters[s] > 0) ? clusters[s] : slots / s;
        if (per_wave < 1) break;
        const int waves = (n_tiles + per_wave - 1) / per_wave;
        if (waves <= best_waves) {
            best_waves = waves;
            best = s;
        }
    }
    return best;
}

// ---------------------------------------------------------------------------
// Split-K reduction.  Each CTA of a cluster of S owns output rows
// [lo, lo + width) of the 128-row slab, lo = rank * rows_per with rows_per =
// owner_rows(S) (ceil(128 / S) rounded up to a multiple of 4), and sums the
// S partials of those rows in rank order
// (deterministic).  `out(m, r, sum)` writes the output of token m, slab row
// r.  Outputs are visited token-major (item i = token i / width, row lo +
// i % width), so a warp writes consecutive outputs of one token.
// ---------------------------------------------------------------------------

// Output rows owned by each CTA of a cluster of S: ceil(128 / S) rounded
// up to a multiple of 4, so every owner's rows start on a 16-byte boundary
// of a token's partial row (the last owner takes what is left: 8 to 128
// rows, never none).
__host__ __device__ constexpr int owner_rows(int splits) {
    return ((BNW + splits - 1) / splits + 3) & ~3;
}

// Push: the partials arrive in a receive buffer of this CTA laid out
// [S][rows_per][stride] fp32 (stride = Mp + 4, Mp = M rounded up to 4: the
// padding spreads the rows of one token over the banks).
__host__ __device__ __forceinline__ int push_stride(int M) { return ((M + 3) & ~3) + 4; }

__host__ __device__ __forceinline__ uint32_t push_recv_bytes(int M, int splits) {
    const int rows_per = owner_rows(splits);
    return (static_cast<uint32_t>(splits * rows_per * push_stride(M) * 4) + 127u) & ~127u;
}

// Bytes the owner of rows [lo, lo + width) receives (its mbarrier's tx count).
__device__ __forceinline__ uint32_t push_expect_bytes(int M, int splits, int width) {
    return static_cast<uint32_t>(splits * width * ((M + 3) & ~3) * 4);
}

// Send row nl (0..127) of this CTA's partial, v[0..M), to the CTA that owns
// it: owner.recv[rank][nl - owner.lo][0..Mp), counted on owner.recv_full.
template <int MT>
__device__ __forceinline__ void push_send(const float (&v)[MT], int M, int nl, uint32_t rank,
                                          int splits, float* recv, uint64_t* recv_full) {
    const int rows_per = owner_rows(splits);
    const int owner = nl / rows_per;
    const int rloc = nl - owner * rows_per;
    const uint32_t dst =
        map_to_rank(smem_u32(recv + (static_cast<int>(rank) * rows_per + rloc) * push_stride(M)),
                    static_cast<uint32_t>(owner));
    const uint32_t bar = map_to_rank(smem_u32(recv_full), static_cast<uint32_t>(owner));
#pragma unroll
    for (int c = 0; c < MT / 4; ++c)
        if (4 * c < M)
            st_async_v4(dst + 16u * c, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3], bar);
}

// After a receive wait that gave up (the status word is already set): a
// peer that has not sent yet could still write into this CTA's receive
// buffer, so the CTA must not exit before its peers.  A cluster barrier
// waits for every non-exited thread of the cluster (PTX ISA, barrier.cluster):
// peers that finished have exited and are not waited for, and every other
// peer's waits are bounded and it sends before it exits, so this completes.
__device__ __forceinline__ void outlive_peers() { cluster_sync_all(); }

// Sum the received partials of rows [lo, lo + width) (call after recv_full
// completed); every thread of the CTA takes part.
template <typename Out>
__device__ __forceinline__ void push_reduce(const float* recv, int splits, int lo, int width,
                                            int M, Out out) {
    if (width <= 0) return;
    const int rows_per = owner_rows(splits);
    const int stride = push_stride(M);
    const int split_step = rows_per * stride;
    // walk i = threadIdx.x, +kThreads, ... as (m, r) without dividing
    const int dm = kThreads / width, dr = kThreads - dm * width;
    int m = static_cast<int>(threadIdx.x) / width;
    int r = static_cast<int>(threadIdx.x) - m * width;
    while (m < M) {
        const float* p = recv + r * stride + m;
        float part[kMaxSplits];
#pragma unroll
        for (int j = 0; j < kMaxSplits; ++j) part[j] = j < splits ? p[j * split_step] : 0.0f;
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxSplits; ++j)
            if (j < splits) acc += part[j];
        out(m, lo + r, acc);
        r += dr;
        m += dm;
        if (r >= width) {
            r -= width;
            ++m;
        }
    }
}

// Pull: every CTA left its partial D^T tile [MT][BNW] at `red`; after a
// cluster barrier each owner reads the S partials of its rows.  Owners hold
// multiples of 4 rows starting on a multiple of 4 (owner_rows), so an item
// is 4 consecutive rows of one token: one 16-byte load per peer, all S
// loads issued before any sum (one distributed-shared-memory round trip),
// then the 4 lanes summed in rank order -- the same sums as one row at a
// time.  A second cluster barrier must keep every CTA alive until its peers
// have read it.
template <int S, typename Out>
__device__ __forceinline__ void pull_reduce_s(const float* red, int lo, int width, int M,
                                              Out out) {
    static_assert(owner_rows(S) % 4 == 0, "owners hold whole 4-row groups");
    const int groups = width / 4;  // width: owner_rows(S), or the last owner's rest
    const int items = groups * M;
    uint32_t peer[S];
#pragma unroll
    for (int j = 0; j < S; ++j) peer[j] = map_to_rank(smem_u32(red), j);
    for (int i = static_cast<int>(threadIdx.x); i < items; i += kThreads) {
        const int m = i / groups;
        const int r = lo + 4 * (i - m * groups);
        const uint32_t off = static_cast<uint32_t>((m * BNW + r) * 4);
        float4 part[S];
#pragma unroll
        for (int j = 0; j < S; ++j) part[j] = ld_dsmem_v4(peer[j] + off);
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
        for (int j = 0; j < S; ++j) {
            a0 += part[j].x;
            a1 += part[j].y;
            a2 += part[j].z;
            a3 += part[j].w;
        }
        out(m, r, a0);
        out(m, r + 1, a1);
        out(m, r + 2, a2);
        out(m, r + 3, a3);
    }
}

template <typename Out>
__device__ __forceinline__ void pull_reduce(const float* red, int splits, int lo, int width,
                                            int M, Out out) {
    switch (splits) {
        case 1: pull_reduce_s<1>(red, lo, width, M, out); break;
        case 2: pull_reduce_s<2>(red, lo, width, M, out); break;
        case 3: pull_reduce_s<3>(red, lo, width, M, out); break;
        case 4: pull_reduce_s<4>(red, lo, width, M, out); break;
        case 5: pull_reduce_s<5>(red, lo, width, M, out); break;
        case 6: pull_reduce_s<6>(red, lo, width, M, out); break;
        case 7: pull_reduce_s<7>(red, lo, width, M, out); break;
        default: pull_reduce_s<8>(red, lo, width, M, out); break;
    }
}

}  // namespace decode
}  // namespace fp8k
