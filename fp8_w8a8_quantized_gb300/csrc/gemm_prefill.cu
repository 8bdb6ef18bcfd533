// Scaled FP8 GEMM for prefill-sized M on the 5th-generation tensor cores.
//
//   y[m, n] = bf16_rn((acc[m, n] * s_tok[m]) * s_w[n]),
//   acc[m, n] = sum_k e4m3(xq[m, k]) * e4m3(wq[n, k])      (fp32, in TMEM)
//
// "FP8 Inference Explained, in depth", "Inside a quantized linear layer": the
// per-token and per-channel scales are constant along k, so they are applied
// once to the fp32 dot product in the epilogue; "FP8 Quantization", "How FP8
// Matmul Works at the Hardware Level": E4M3 x E4M3 -> FP32 accumulate -> BF16.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: 128-byte-swizzled K-major tiles of xq (128 x 128
//               bytes) and wq (256 x 128 bytes) into a 4-stage shared ring;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (kind::f8f6f4, M=128, N=256, K=32) from one lane; each stage
//               is released to the producer by tcgen05.commit;
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulator (each warp owns
//               the 32 TMEM lanes its rank allows), scale, bf16, store.
// The accumulator is double-buffered in TMEM (2 x 256 columns) so the
// epilogue of one tile overlaps the main loop of the next.  Tiles are walked
// in groups of kGroupM row blocks so concurrently running CTAs share both the
// weight and the activation tiles in L2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace fp8k {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;      // bytes of K per stage = one 128-byte swizzle row
constexpr int KSTEP = 32;    // K of one tcgen05.mma kind::f8f6f4
constexpr int STAGES = 4;
constexpr int kGroupM = 16;
constexpr int kThreads = 192;
constexpr uint32_t A_TILE = BM * BK;
constexpr uint32_t B_TILE = BN * BK;
constexpr uint32_t STAGE_BYTES = A_TILE + B_TILE;
constexpr uint32_t TMEM_COLS = 512;

struct Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 1024 /* alignment slack */ + STAGES * STAGE_BYTES + sizeof(Bars);

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
    gemm_prefill_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const float* __restrict__ s_tok,
                        const float* __restrict__ s_w, __nv_bfloat16* __restrict__ y, int M, int N,
                        int K, unsigned* status) {
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

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 128);
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

    // Everything above overlaps the previous kernel; inputs are read below.
    pdl_wait_primary();

    // Each role loop is run by a whole warp (lane 0 issues, waits are
    // warp-uniform), so every warp is converged at the aligned instructions.
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
        // ---- MMA issuer ----
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        int local = 0;
        for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!(ok = warp_wait(&bars->acc_empty[buf], acc_phase ^ 1u, abort_flag, status))) break;
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
                        // advancing K by 32 bytes inside the swizzle atom moves
                        // the descriptor start address by 32 >> 4 = 2
                        mma_f8(d_tmem, a0 + 2 * kk, b0 + 2 * kk, idesc, (kb | kk) != 0);
                    }
                    mma_commit(&bars->empty[stage]);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok && lane == 0) mma_commit(&bars->acc_full[buf]);
            __syncwarp();
        }
        // every MMA this warp issued has finished before TMEM is freed
        if (lane == 0) {
            mma_commit(&bars->drain);
            wait_drain(&bars->drain, status);
        }
        __syncwarp();
    } else {
        // ---- epilogue warps 2..5: TMEM lane quarter = warp rank % 4 ----
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        const bool vec_ok = (N % 8) == 0;
        const bool sw_vec = (reinterpret_cast<uintptr_t>(s_w) & 15u) == 0;
        int local = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++local) {
            int m_blk, n_blk;
            tile_coords(t, num_m, num_n, m_blk, n_blk);
            const int buf = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            if (!warp_wait(&bars->acc_full[buf], acc_phase, abort_flag, status)) break;
            tc_fence_after();
            const int m = m_blk * BM + row_in_tile;
            const bool row_ok = m < M;
            const float st = row_ok ? __ldg(s_tok + m) : 0.0f;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN;
            __nv_bfloat16* yrow = y + static_cast<int64_t>(row_ok ? m : 0) * N;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + c * 32, r);
                tmem_ld_wait();
                if (c == BN / 32 - 1) {
                    // accumulator fully read: hand the buffer back to the MMA warp
                    tc_fence_before();
                    mbar_arrive(&bars->acc_empty[buf]);
                }
                const int n0 = n_blk * BN + c * 32;
                if (row_ok && n0 < N) {
                    float sw[32];
                    if (sw_vec && n0 + 32 <= N) {
                        const float4* p = reinterpret_cast<const float4*>(s_w + n0);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 v = __ldg(p + j);
                            sw[4 * j] = v.x;
                            sw[4 * j + 1] = v.y;
                            sw[4 * j + 2] = v.z;
                            sw[4 * j + 3] = v.w;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) sw[j] = n0 + j < N ? __ldg(s_w + n0 + j) : 0.0f;
                    }
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float v0 = (__uint_as_float(r[2 * j]) * st) * sw[2 * j];
                        const float v1 = (__uint_as_float(r[2 * j + 1]) * st) * sw[2 * j + 1];
                        packed[j] = pack_bf16x2(v0, v1);
                    }
                    if (vec_ok && n0 + 32 <= N) {
                        uint4* dst = reinterpret_cast<uint4*>(yrow + n0);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1],
                                                packed[4 * j + 2], packed[4 * j + 3]);
                    } else {
                        uint16_t* dst = reinterpret_cast<uint16_t*>(yrow + n0);
                        for (int j = 0; j < 32 && n0 + j < N; ++j)
                            dst[j] = static_cast<uint16_t>(packed[j >> 1] >> ((j & 1) * 16));
                    }
                }
                __syncwarp();
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

}  // namespace

cudaError_t prepare_gemm_prefill() {
    return cudaFuncSetAttribute(gemm_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemBytes));
}

cudaError_t launch_gemm_prefill(const GemmArgs& a) {
    CUtensorMap tmA, tmB;
    if (!encode_tmap_u8(&tmA, a.xq, a.M, a.K, a.K, BK, BM)) return cudaErrorInvalidValue;
    if (!encode_tmap_u8(&tmB, a.wq, a.N, a.K, a.K, BK, BN)) return cudaErrorInvalidValue;
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    const int grid = tiles < a.num_sms ? tiles : a.num_sms;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_prefill_kernel, tmA, tmB, a.s_tok, a.s_w,
                              static_cast<__nv_bfloat16*>(a.y), a.M, a.N, a.K, a.status);
}

}  // namespace fp8k
