// Block-scaled FP8 GEMM: one activation scale per token per 128 inputs and
// one weight scale per 128 x 128 block,
//
//   y[m, n] = bf16_rn( sum_kb s_x[m, kb] * s_w[n / 128, kb] * P[m, n, kb] ),
//   P[m, n, kb] = sum_{k in block kb} e4m3(xq[m, k]) * e4m3(wq[n, k])  (fp32).
//
// "FP8 Inference Explained, in depth", "Inside a quantized linear layer":
// block-wise scales vary along k, so the kernel multiplies each block's
// partial sum by that block's scales as it goes; "FP8 Quantization",
// "Granularity": one weight scale per 128 x 128 tile.  (The 128-element
// promotion interval is also the one "Quantization: FP8 inference and
// KV-cache quantization", "Training in FP8 or lower", reports for
// DeepSeek-V3.)
//
// On tcgen05 the scaling cannot ride inside the MMA (the block-scaled MMA
// kinds take power-of-two scales per 32 elements), so each 128-deep k-block
// is accumulated on its own in TMEM and promoted by CUDA cores:
//   * the MMA warp writes the k-block's partial tile into one of two TMEM
//     buffers (double-buffered, so the tensor core runs ahead by one k-block);
//   * epilogue warps load it with tcgen05.ld, multiply by s_x * s_w and add
//     it to fp32 accumulators held in registers, then hand the buffer back.
// Two kernels share this scheme:
//   gemm_blockwise_prefill  persistent 128 x 256 output tiles (two weight
//                           blocks), 8 epilogue warps of 128 columns each;
//   gemm_blockwise_decode   M <= 64: swap-AB weight streaming with a cluster
//                           split-K (as gemm_decode.cu); the partials are
//                           already scaled when they are summed through
//                           distributed shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "decode_common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace fp8k {
namespace {

constexpr int kBlock = 128;  // scale block edge (K for both operands, N for W)

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// ============================================================================
// Prefill: persistent 128 x 256 tiles.
// ============================================================================
namespace pf {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int KSTEP = 32;
constexpr int STAGES = 4;
constexpr int kGroupM = 16;
constexpr int kEpiWarps = 8;   // 2 per TMEM lane quarter, 128 columns each
constexpr int kCols = BN / (kEpiWarps / 4);
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t A_TILE = BM * BK;
constexpr uint32_t B_TILE = BN * BK;
constexpr uint32_t STAGE_BYTES = A_TILE + B_TILE;
constexpr uint32_t TMEM_COLS = 2 * BN;  // two k-block buffers

struct Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t kfull[2];   // k-block partial in TMEM buffer b is complete
    uint64_t kempty[2];  // every epilogue warp has read buffer b
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 1024 + STAGES * STAGE_BYTES + sizeof(Bars);

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& m_blk, int& n_blk) {
    const int per_group = kGroupM * num_n;
    const int g = t / per_group;
    const int first_m = g * kGroupM;
    const int gm = min(kGroupM, num_m - first_m);
    const int local = t - g * per_group;
    m_blk = first_m + local % gm;
    n_blk = local / gm;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_blockwise_prefill(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const float* __restrict__ s_x,
                           const float* __restrict__ s_w, __nv_bfloat16* __restrict__ y, int M,
                           int N, int K, unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_TILE;
    Bars* bars = reinterpret_cast<Bars*>(sB + STAGES * B_TILE);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_m = (M + BM - 1) / BM;
    const int num_n = (N + BN - 1) / BN;
    const int tiles = num_m * num_n;
    const int nk = (K + BK - 1) / BK;
    const int NB = (N + kBlock - 1) / kBlock;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->kfull[b], 1);
            mbar_init(&bars->kempty[b], kEpiWarps);
        }
        mbar_init(&bars->drain, 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;

    pdl_wait_primary();

    if (warp == 0) {
        // ---- TMA producer ----
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
            int m_blk, n_blk;
            tile_coords(t, num_m, num_n, m_blk, n_blk);
            for (int kb = 0; kb < nk; ++kb) {
                if (!(ok = warp_wait(&bars->empty[stage], phase ^ 1u, abort_flag, status))) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars->full[stage], STAGE_BYTES);
                    tma_load_2d(sA + stage * A_TILE, &tmA, &bars->full[stage], kb * BK, m_blk * BM);
                    tma_load_2d(sB + stage * B_TILE, &tmB, &bars->full[stage], kb * BK, n_blk * BN);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer: one k-block per TMEM buffer, alternating ----
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
        uint32_t stage = 0, phase = 0, count = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
            for (int kb = 0; kb < nk; ++kb, ++count) {
                const uint32_t buf = count & 1u, use = count >> 1;
                if (!(ok = warp_wait(&bars->kempty[buf], (use & 1u) ^ 1u, abort_flag, status)))
                    break;
                if (!(ok = warp_wait(&bars->full[stage], phase, abort_flag, status))) break;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    const uint64_t a0 = sdesc_kmajor_sw128(smem_u32(sA + stage * A_TILE));
                    const uint64_t b0 = sdesc_kmajor_sw128(smem_u32(sB + stage * B_TILE));
#pragma unroll
                    for (int kk = 0; kk < BK / KSTEP; ++kk)
                        mma_f8(d_tmem, a0 + 2 * kk, b0 + 2 * kk, idesc, kk != 0);
                    mma_commit(&bars->empty[stage]);
                    mma_commit(&bars->kfull[buf]);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0) {
            mma_commit(&bars->drain);
            wait_drain(&bars->drain, status);
        }
        __syncwarp();
    } else {
        // ---- epilogue warps: lane quarter warp % 4, column slice (warp-2)/4 ----
        const int quarter = warp & 3;
        const int slice = (warp - 2) >> 2;
        const int row_in_tile = quarter * 32 + lane;
        const bool vec_ok = (N % 8) == 0;
        const int KB = nk;
        uint32_t count = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
            int m_blk, n_blk;
            tile_coords(t, num_m, num_n, m_blk, n_blk);
            const int m = m_blk * BM + row_in_tile;
            const bool row_ok = m < M;
            const int n0 = n_blk * BN + slice * kCols;
            const int nb = n0 / kBlock;
            const bool nb_ok = nb < NB;
            const float* sxr = s_x + static_cast<int64_t>(row_ok ? m : 0) * KB;
            const float* swr = s_w + static_cast<int64_t>(nb_ok ? nb : 0) * KB;
            float acc[kCols];
#pragma unroll
            for (int j = 0; j < kCols; ++j) acc[j] = 0.0f;
            float sx_next = row_ok ? __ldg(sxr) : 0.0f;
            float sw_next = nb_ok ? __ldg(swr) : 0.0f;
            for (int kb = 0; kb < nk; ++kb, ++count) {
                const float c = sx_next * sw_next;
                if (kb + 1 < nk) {
                    sx_next = row_ok ? __ldg(sxr + kb + 1) : 0.0f;
                    sw_next = nb_ok ? __ldg(swr + kb + 1) : 0.0f;
                }
                const uint32_t buf = count & 1u, use = count >> 1;
                if (!(ok = warp_wait(&bars->kfull[buf], use & 1u, abort_flag, status))) break;
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       buf * BN + slice * kCols;
                // 16 columns per load: 128 accumulators + staging stay in registers
#pragma unroll
                for (int h = 0; h < kCols / 16; ++h) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(taddr + h * 16, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; j += 2)
                        fma2(acc[h * 16 + j], acc[h * 16 + j + 1], __uint_as_float(r[j]),
                             __uint_as_float(r[j + 1]), c, c);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->kempty[buf]);
            }
            if (!ok) break;
            if (row_ok && n0 < N) {
                __nv_bfloat16* yrow = y + static_cast<int64_t>(m) * N;
                if (vec_ok && n0 + kCols <= N) {
                    uint4* dst = reinterpret_cast<uint4*>(yrow + n0);
#pragma unroll
                    for (int j = 0; j < kCols / 8; ++j)
                        dst[j] = make_uint4(pack_bf16x2(acc[8 * j], acc[8 * j + 1]),
                                            pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]),
                                            pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]),
                                            pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]));
                } else {
#pragma unroll
                    for (int j = 0; j < kCols; ++j)
                        if (n0 + j < N) yrow[n0 + j] = __float2bfloat16_rn(acc[j]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace pf

// ============================================================================
// Decode: swap-AB weight streaming, cluster split-K.
// ============================================================================
namespace dc {

using namespace decode;

constexpr int kMaxStages = 8;

template <int MT>
struct Cfg {
    static constexpr uint32_t X_TILE = MT * BK;
    static constexpr uint32_t STAGE_BYTES = W_TILE + X_TILE;
    static constexpr uint32_t RED_BYTES = MT * BNW * 4;  // pull: scaled partial in the ring
    static constexpr uint32_t TMEM_COLS = 2 * MT < 32 ? 32 : 2 * MT;  // two k-block buffers
    // Push the scaled partials into a dedicated receive buffer up to 16
    // tokens; pull beyond (as in gemm_decode.cu).
    static constexpr bool kPush = MT <= 16;
};

struct Bars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t kfull[2];
    uint64_t kempty[2];
    uint64_t drain;
    uint64_t recv_full;  // push: the S partials of this CTA's rows have arrived
    uint32_t tmem_base;
    int abort;
};

// [ring | receive buffer (push) | Bars] after up to 1 KB of alignment; the
// ring gets what is left of the budget that lets kCtasPerSm CTAs share an SM.
struct Layout {
    uint32_t recv_bytes;
    int stages;
    size_t smem;
};

template <int MT>
Layout layout_of(int M, int splits, int64_t budget) {
    using C = Cfg<MT>;
    Layout l;
    l.recv_bytes = C::kPush ? push_recv_bytes(M, splits) : 0u;
    const int64_t room =
        budget - 1024 - static_cast<int64_t>(sizeof(Bars)) - l.recv_bytes;
    const int st = static_cast<int>(room / C::STAGE_BYTES);
    l.stages = st < kMaxStages ? st : kMaxStages;
    l.smem = 1024 + static_cast<size_t>(l.stages) * C::STAGE_BYTES + l.recv_bytes + sizeof(Bars);
    return l;
}

template <int MT>
__global__ void __launch_bounds__(kThreads)
    gemm_blockwise_decode(const __grid_constant__ CUtensorMap tmW,
                          const __grid_constant__ CUtensorMap tmX, const float* __restrict__ s_x,
                          const float* __restrict__ s_w, __nv_bfloat16* __restrict__ y, int M,
                          int N, int K, int splits, int stages, uint32_t recv_bytes,
                          unsigned* status) {
    using C = Cfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* ring = smem;
    float* recv = reinterpret_cast<float*>(smem + stages * C::STAGE_BYTES);  // push
    Bars* bars = reinterpret_cast<Bars*>(smem + stages * C::STAGE_BYTES + recv_bytes);
    float* red = reinterpret_cast<float*>(smem);  // pull: [MT][BNW], after the main loop

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_blk = blockIdx.y;
    const uint32_t rank = cluster_ctarank();
    const int nk = (K + BK - 1) / BK;
    const int per = nk / splits, rem = nk % splits;
    const int kb0 = static_cast<int>(rank) * per + min(static_cast<int>(rank), rem);
    const int nkb = per + (static_cast<int>(rank) < rem ? 1 : 0);
    // output rows [lo, hi) of the slab are reduced and stored by this CTA
    const int rows_per = owner_rows(splits);
    const int lo = static_cast<int>(rank) * rows_per;
    const int hi = min(BNW, lo + rows_per);
    const int width = hi > lo ? hi - lo : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->kfull[b], 1);
            mbar_init(&bars->kempty[b], 4);
        }
        mbar_init(&bars->drain, 1);
        if constexpr (C::kPush) {
            mbar_init(&bars->recv_full, 1);
            mbar_arrive_expect_tx(&bars->recv_full, push_expect_bytes(M, splits, width));
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Push: peers may send partials once every CTA's barriers are initialised.
    if constexpr (C::kPush) cluster_arrive();
    const uint32_t tmem_base = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;

    if (warp == 0) {
        // ---- TMA producer (only L2 prefetches before the wait, as in
        // gemm_decode.cu) ----
        const uint64_t w_policy = policy_evict_first();
        if (lane == 0) {
            const int pf = nkb < kL2PrefetchBlocks ? nkb : kL2PrefetchBlocks;
            for (int i = 0; i < pf; ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * BK, n_blk * BNW);
        }
        __syncwarp();
        pdl_wait_primary();
        int stage = 0;
        uint32_t phase = 0;
        for (int i = 0; i < nkb; ++i) {
            if (!warp_wait(&bars->empty[stage], phase ^ 1u, abort_flag, status)) break;
            if (lane == 0) {
                uint8_t* st = ring + stage * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&bars->full[stage], C::STAGE_BYTES);
                tma_load_2d_hint(st, &tmW, &bars->full[stage], (kb0 + i) * BK, n_blk * BNW,
                                 w_policy);
                tma_load_2d(st + W_TILE, &tmX, &bars->full[stage], (kb0 + i) * BK, 0);
            }
            __syncwarp();
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer: k-block i into TMEM buffer i % 2 ----
        pdl_wait_primary();
        constexpr uint32_t idesc = idesc_e4m3_f32(BNW, MT);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            const uint32_t buf = i & 1, use = static_cast<uint32_t>(i) >> 1;
            if (!(ok = warp_wait(&bars->kempty[buf], (use & 1u) ^ 1u, abort_flag, status))) break;
            if (!(ok = warp_wait(&bars->full[stage], phase, abort_flag, status))) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = smem_u32(ring + stage * C::STAGE_BYTES);
                const uint64_t a0 = sdesc_kmajor_sw128(st);
                const uint64_t b0 = sdesc_kmajor_sw128(st + W_TILE);
#pragma unroll
                for (int kk = 0; kk < BK / KSTEP; ++kk)
                    mma_f8(tmem_base + buf * MT, a0 + 2 * kk, b0 + 2 * kk, idesc, kk != 0);
                mma_commit(&bars->empty[stage]);
                mma_commit(&bars->kfull[buf]);
            }
            __syncwarp();
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (lane == 0) {
            mma_commit(&bars->drain);
            wait_drain(&bars->drain, status);
        }
        __syncwarp();
    } else {
        // ---- epilogue warps: TMEM lanes (= weight rows) of this warp's quarter ----
        pdl_wait_primary();
        const int quarter = warp & 3;
        const int nl = quarter * 32 + lane;
        const int KB = nk;
        const bool nb_ok = n_blk * BNW < N;
        float acc[MT];
#pragma unroll
        for (int j = 0; j < MT; ++j) acc[j] = 0.0f;
        // lane j holds the scales of tokens j and j + 32 for the current k-block
        auto sx_of = [&](int kb, int tok) {
            return tok < M ? __ldg(s_x + static_cast<int64_t>(tok) * KB + kb) : 0.0f;
        };
        int kb = kb0;
        float sx0 = nkb > 0 ? sx_of(kb, lane) : 0.0f;
        float sx1 = (MT > 32 && nkb > 0) ? sx_of(kb, lane + 32) : 0.0f;
        float sw = (nb_ok && nkb > 0) ? __ldg(s_w + static_cast<int64_t>(n_blk) * KB + kb) : 0.0f;
        bool ok = true;
        for (int i = 0; i < nkb; ++i, ++kb) {
            const float c0 = sx0, c1 = sx1, cw = sw;
            if (i + 1 < nkb) {
                sx0 = sx_of(kb + 1, lane);
                if (MT > 32) sx1 = sx_of(kb + 1, lane + 32);
                sw = nb_ok ? __ldg(s_w + static_cast<int64_t>(n_blk) * KB + kb + 1) : 0.0f;
            }
            const uint32_t buf = i & 1, use = static_cast<uint32_t>(i) >> 1;
            if (!(ok = warp_wait(&bars->kfull[buf], use & 1u, abort_flag, status))) break;
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * MT;
            if constexpr (MT == 16) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(taddr, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    acc[j] = fmaf(__uint_as_float(r[j]), cw * __shfl_sync(0xFFFFFFFFu, c0, j),
                                  acc[j]);
            } else {
#pragma unroll
                for (int h = 0; h < MT / 32; ++h) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + h * 32, r);
                    tmem_ld_wait();
                    const float ch = h == 0 ? c0 : c1;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        acc[h * 32 + j] = fmaf(__uint_as_float(r[j]),
                                               cw * __shfl_sync(0xFFFFFFFFu, ch, j),
                                               acc[h * 32 + j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->kempty[buf]);
        }
        if (!ok) {
#pragma unroll
            for (int j = 0; j < MT; ++j) acc[j] = 0.0f;
        }
        if constexpr (C::kPush) {
            // Sent even after a failed wait (as zeros) so that every owner's
            // barrier completes.
            cluster_wait();
            push_send<MT>(acc, M, nl, rank, splits, recv, &bars->recv_full);
        } else {
            // every MMA has finished (last kfull) and every stage was
            // consumed: the ring is idle and holds the scaled partial tile
#pragma unroll
            for (int j = 0; j < MT; ++j) red[j * BNW + nl] = acc[j];
        }
    }

    // the partials are already scaled: y[m, n] = bf16(sum)
    auto store = [&](int m, int r, float sum) {
        const int n = n_blk * BNW + r;
        if (n < N) y[static_cast<int64_t>(m) * N + n] = __float2bfloat16_rn(sum);
    };
    if constexpr (C::kPush) {
        if (warp < 2) cluster_wait();
        // every tcgen05 operation of this CTA has completed: free TMEM
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem_base, C::TMEM_COLS);
        }
        // Nothing remote touches this CTA after its partials have arrived.
        if (warp_wait_cluster_noabort(&bars->recv_full, 0, 4 * kWaitLimitNs, status))
            push_reduce(recv, splits, lo, width, M, store);
        else
            outlive_peers();
    } else {
        tc_fence_before();
        cluster_sync_all();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem_base, C::TMEM_COLS);
        }
        pull_reduce(red, splits, lo, width, M, store);
        // Peers may still be reading this CTA's partial.
        cluster_sync_all();
    }
}

template <int MT>
cudaError_t launch_mt(const GemmArgs& a) {
    CUtensorMap tmW, tmX;
    if (!encode_tmap_u8(&tmW, a.wq, a.N, a.K, a.K, BK, BNW)) return cudaErrorInvalidValue;
    if (!encode_tmap_u8(&tmX, a.xq, a.M, a.K, a.K, BK, MT)) return cudaErrorInvalidValue;
    const int n_tiles = (a.N + BNW - 1) / BNW;
    const int nk = (a.K + BK - 1) / BK;
    const int splits =
        choose_splits(n_tiles, nk, a.num_sms, a.decode_clusters ? a.decode_clusters + 2 * 9 : nullptr);
    // as in gemm_decode.cu: a grid of at most two CTAs per SM gets the
    // two-per-SM budget (deeper ring)
    const bool two = static_cast<int64_t>(n_tiles) * splits <= 2 * a.num_sms;
    const Layout l = layout_of<MT>(a.M, splits, two ? kCtaSmem2 : kCtaSmem);
    if (l.stages < 2 || (!Cfg<MT>::kPush && Cfg<MT>::RED_BYTES > l.stages * Cfg<MT>::STAGE_BYTES))
        return cudaErrorInvalidConfiguration;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(splits, n_tiles);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = l.smem;
    cfg.stream = a.stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_blockwise_decode<MT>, tmW, tmX, a.s_tok, a.s_w,
                              static_cast<__nv_bfloat16*>(a.y), a.M, a.N, a.K, splits, l.stages,
                              l.recv_bytes, a.status);
}

}  // namespace dc

}  // namespace

cudaError_t prepare_gemm_blockwise() {
    cudaError_t e = cudaFuncSetAttribute(pf::gemm_blockwise_prefill,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(pf::kSmemBytes));
    if (e != cudaSuccess) return e;
    for (auto* k : {dc::gemm_blockwise_decode<16>, dc::gemm_blockwise_decode<32>,
                    dc::gemm_blockwise_decode<64>}) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(decode::kCtaSmem2));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_blockwise(const GemmArgs& a) {
    if (a.M <= 16) return dc::launch_mt<16>(a);
    if (a.M <= 32) return dc::launch_mt<32>(a);
    if (a.M <= kBlockwiseDecodeMaxM) return dc::launch_mt<64>(a);

    CUtensorMap tmA, tmB;
    if (!encode_tmap_u8(&tmA, a.xq, a.M, a.K, a.K, pf::BK, pf::BM)) return cudaErrorInvalidValue;
    if (!encode_tmap_u8(&tmB, a.wq, a.N, a.K, a.K, pf::BK, pf::BN)) return cudaErrorInvalidValue;
    const int tiles = ((a.M + pf::BM - 1) / pf::BM) * ((a.N + pf::BN - 1) / pf::BN);
    const int grid = tiles < a.num_sms ? tiles : a.num_sms;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(pf::kThreads);
    cfg.dynamicSmemBytes = pf::kSmemBytes;
    cfg.stream = a.stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pf::gemm_blockwise_prefill, tmA, tmB, a.s_tok, a.s_w,
                              static_cast<__nv_bfloat16*>(a.y), a.M, a.N, a.K, a.status);
}

}  // namespace fp8k
