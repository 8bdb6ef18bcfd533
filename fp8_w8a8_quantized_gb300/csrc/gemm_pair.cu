// Scaled FP8 GEMM for every M above the decode sizes, on pairs of SMs
// (tcgen05 cta_group::2).
//
//   y[m, n] = bf16_rn((acc[m, n] * s_tok[m]) * s_w[n]),
//   acc[m, n] = sum_k e4m3(xq[m, k]) * e4m3(wq[n, k])      (fp32, in TMEM)
//
// ("FP8 Inference Explained, in depth", "Inside a quantized linear layer";
// "FP8 Quantization", "How FP8 Matmul Works at the Hardware Level"), with a
// 256 x 256 output tile per cluster of two CTAs on two SMs.  One MMA instruction (M = 256, N = 256, K = 32) runs on
// both SMs' tensor cores: each CTA holds its own 128 rows of the activation
// tile and half of the weight tile, so per SM and per 128 of K, TMA writes
// 32 KB into shared memory instead of the 48 KB a one-SM 128 x 256 tile
// needs, for the same number of MMA flops per SM.  A ring stage holds 256 of
// K (two 128-byte swizzle columns per operand), so each barrier round trip
// and each commit covers eight MMAs: per-stage overhead, not bandwidth, was
// what held the tensor pipe back with 128-deep stages (measured on GB300).
//
// Per CTA (192 threads):
//   warp 0      TMA producer: its 128 activation rows and 128 weight rows of
//               each 256-deep k-block into a 3-stage ring (64 KB a stage);
//               completion is counted on the even CTA's barrier (cta_group::2
//               TMA);
//   warp 1      allocates the pair's TMEM (collectively with the peer); in the
//               even CTA it issues the pair MMAs and multicasts each commit to
//               both CTAs' barriers;
//   warps 2..5  epilogue of this CTA's 128 rows (tcgen05.ld of its own TMEM),
//               scale, bf16, store; they return the accumulator buffer to the
//               even CTA's MMA warp by remote mbarrier arrives.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace fp8k {
namespace {

constexpr int BM = 256;      // output rows per pair (128 per CTA)
constexpr int BN = 256;      // output columns per pair (B split 128 / 128)
constexpr int BK = 256;      // bytes of K per stage (two 128-byte swizzle columns)
constexpr int BKS = 128;     // bytes of K per swizzle column / TMA box
constexpr int KSTEP = 32;    // K of one tcgen05.mma kind::f8f6f4
constexpr int STAGES = 3;
constexpr int kGroupM = 8;   // row-block groups for L2 reuse of weight tiles
constexpr int kThreads = 192;
constexpr int kAccBufs = 2;  // TMEM accumulator buffers of BN columns
constexpr uint32_t A_TILE = (BM / 2) * BK;
constexpr uint32_t B_TILE = (BN / 2) * BK;
constexpr uint32_t STAGE_BYTES = A_TILE + B_TILE;
constexpr uint32_t TMEM_COLS = kAccBufs * BN;

struct Bars {
    uint64_t full[STAGES];     // even CTA: both CTAs' tiles of the stage landed
    uint64_t empty[STAGES];    // both CTAs: the pair MMAs finished with the stage
    uint64_t acc_full[kAccBufs];
    uint64_t acc_empty[kAccBufs];  // even CTA: both epilogues read the buffer
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const float* __restrict__ s_tok, const float* __restrict__ s_w,
                     __nv_bfloat16* __restrict__ y, int M, int N, int K, unsigned* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_TILE;
    Bars* bars = reinterpret_cast<Bars*>(sB + STAGES * B_TILE);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int pairs = gridDim.x >> 1;
    const int num_m = (M + BM - 1) / BM;
    const int num_n = (N + BN - 1) / BN;
    const int tiles = num_m * num_n;
    const int nk = (K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 8);  // 4 epilogue warps x 2 CTAs
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
        tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised (and the TMEM allocated) before
    // either CTA signals the other's barriers
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;

    pdl_wait_primary();

    if (warp == 0) {
        // ---- TMA producer (both CTAs) ----
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int t = pair; ok && t < tiles; t += pairs) {
            int m_blk, n_blk;
            tile_coords(t, num_m, num_n, m_blk, n_blk);
            const int a_row = m_blk * BM + static_cast<int>(rank) * (BM / 2);
            const int b_row = n_blk * BN + static_cast<int>(rank) * (BN / 2);
            for (int kb = 0; kb < nk; ++kb) {
                if (!(ok = warp_wait(&bars->empty[stage], phase ^ 1u, abort_flag, status))) break;
                if (lane == 0) {
                    const uint32_t full0 = map_to_rank(smem_u32(&bars->full[stage]), 0);
                    if (leader) mbar_arrive_expect_tx(&bars->full[stage], 2 * STAGE_BYTES);
#pragma unroll
                    for (int j = 0; j < BK / BKS; ++j) {
                        tma_load_2d_pair(sA + stage * A_TILE + j * (A_TILE / 2), &tmA, full0,
                                         kb * BK + j * BKS, a_row);
                        tma_load_2d_pair(sB + stage * B_TILE + j * (B_TILE / 2), &tmB, full0,
                                         kb * BK + j * BKS, b_row);
                    }
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        if (leader) {
            // ---- MMA issuer for the pair ----
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int local = 0;
            for (int t = pair; ok && t < tiles; t += pairs, ++local) {
                const int buf = local % kAccBufs;
                const uint32_t acc_phase = (local / kAccBufs) & 1;
                if (!(ok = warp_wait_cluster(&bars->acc_empty[buf], acc_phase ^ 1u, abort_flag,
                                             status)))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!(ok = warp_wait(&bars->full[stage], phase, abort_flag, status))) break;
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t a0 = sdesc_kmajor_sw128(smem_u32(sA + stage * A_TILE));
                        const uint64_t b0 = sdesc_kmajor_sw128(smem_u32(sB + stage * B_TILE));
#pragma unroll
                        for (int kk = 0; kk < BK / KSTEP; ++kk) {
                            const int j = kk / (BKS / KSTEP), w = kk % (BKS / KSTEP);
                            mma_f8_pair(d_tmem, a0 + ((j * (A_TILE / 2)) >> 4) + 2 * w,
                                        b0 + ((j * (B_TILE / 2)) >> 4) + 2 * w, idesc,
                                        (kb | kk) != 0);
                        }
                        mma_commit_pair(&bars->empty[stage], 0x3);
                    }
                    __syncwarp();
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok && lane == 0) mma_commit_pair(&bars->acc_full[buf], 0x3);
                __syncwarp();
            }
            // every pair MMA has finished before TMEM is freed
            if (lane == 0) {
                mma_commit_pair(&bars->drain, 0x1);
                wait_drain(&bars->drain, status);
            }
            __syncwarp();
        }
    } else {
        // ---- epilogue warps 2..5 of both CTAs: this CTA's 128 rows ----
        const int quarter = warp & 3;
        const int row_in_tile = static_cast<int>(rank) * (BM / 2) + quarter * 32 + lane;
        const bool vec_ok = (N % 8) == 0;
        int local = 0;
        for (int t = pair; t < tiles; t += pairs, ++local) {
            int m_blk, n_blk;
            tile_coords(t, num_m, num_n, m_blk, n_blk);
            const int buf = local % kAccBufs;
            const uint32_t acc_phase = (local / kAccBufs) & 1;
            const int m = m_blk * BM + row_in_tile;
            const bool row_ok = m < M;
            // The tile's scales, loaded before its accumulator is ready: the
            // token scale of this lane's row, and in swl[c] the weight scale
            // of column c * 32 + lane (broadcast to the warp by shuffles).
            const float st = row_ok ? __ldg(s_tok + m) : 0.0f;
            float swl[BN / 32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                const int n = n_blk * BN + c * 32 + lane;
                swl[c] = n < N ? __ldg(s_w + n) : 0.0f;
            }
            if (!warp_wait(&bars->acc_full[buf], acc_phase, abort_flag, status)) break;
            tc_fence_after();
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN;
            __nv_bfloat16* yrow = y + static_cast<int64_t>(row_ok ? m : 0) * N;
            // 32 columns: scale, round to bf16, store (16-byte stores when the
            // row is 16-byte aligned and the chunk is whole).
            auto store_chunk = [&](const uint32_t (&r)[32], float sw_lane, int c) {
                uint32_t packed[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float s0 = __shfl_sync(0xFFFFFFFFu, sw_lane, 2 * j);
                    const float s1 = __shfl_sync(0xFFFFFFFFu, sw_lane, 2 * j + 1);
                    const float v0 = (__uint_as_float(r[2 * j]) * st) * s0;
                    const float v1 = (__uint_as_float(r[2 * j + 1]) * st) * s1;
                    packed[j] = pack_bf16x2(v0, v1);
                }
                const int n0 = n_blk * BN + c * 32;
                if (row_ok && n0 < N) {
                    if (vec_ok && n0 + 32 <= N) {
                        uint4* dst = reinterpret_cast<uint4*>(yrow + n0);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1],
                                                packed[4 * j + 2], packed[4 * j + 3]);
                    } else {
                        // unrolled with a guard per column: a loop bound on
                        // N would index packed[] at run time and put it in
                        // local memory for every chunk
                        uint16_t* dst = reinterpret_cast<uint16_t*>(yrow + n0);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (n0 + j < N)
                                dst[j] = static_cast<uint16_t>(packed[j >> 1] >> ((j & 1) * 16));
                    }
                }
            };
            // TMEM loads double-buffered: chunk c + 1 is in flight while
            // chunk c is scaled and stored.
            uint32_t ra[32], rb[32];
            tmem_ld_32x32b_x32(tbase, ra);
            tmem_ld_wait_regs(ra);
#pragma unroll
            for (int c = 0; c < BN / 32; c += 2) {
                tmem_ld_32x32b_x32(tbase + (c + 1) * 32, rb);
                store_chunk(ra, swl[c], c);
                tmem_ld_wait_regs(rb);
                if (c + 2 < BN / 32) {
                    tmem_ld_32x32b_x32(tbase + (c + 2) * 32, ra);
                } else {
                    // accumulator read: return the buffer to the even CTA's MMA warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_cluster(map_to_rank(smem_u32(&bars->acc_empty[buf]), 0));
                }
                store_chunk(rb, swl[c + 1], c + 1);
                if (c + 2 < BN / 32) tmem_ld_wait_regs(ra);
            }
            __syncwarp();
        }
    }

    // Neither CTA may free TMEM or exit while the pair MMAs, the peer's TMA
    // completions on this CTA's barriers or the peer's remote arrives can
    // still touch it.
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace

cudaError_t prepare_gemm_pair() {
    return cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemBytes));
}

// Clusters of two that can be resident at once (a cluster needs two free SMs
// of one TPC); the persistent grid is sized to it.
int gemm_pair_resident_clusters(int num_sms) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0)
        n = num_sms / 2;
    return n;
}

cudaError_t launch_gemm_pair(const GemmArgs& a) {
    CUtensorMap tmA, tmB;
    if (!encode_tmap_u8(&tmA, a.xq, a.M, a.K, a.K, BKS, BM / 2)) return cudaErrorInvalidValue;
    if (!encode_tmap_u8(&tmB, a.wq, a.N, a.K, a.K, BKS, BN / 2)) return cudaErrorInvalidValue;
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    const int max_pairs = a.pair_clusters > 0 ? a.pair_clusters : a.num_sms / 2;
    const int pairs = tiles < max_pairs ? tiles : max_pairs;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel, tmA, tmB, a.s_tok, a.s_w,
                              static_cast<__nv_bfloat16*>(a.y), a.M, a.N, a.K, a.status);
}

}  // namespace fp8k
