// Scaled FP8 GEMM for decode-sized M (M <= 64 tokens): weight streaming.
//
// Same result as the prefill kernel,
//   y[m, n] = bf16_rn((acc[m, n] * s_tok[m]) * s_w[n]),
//   acc[m, n] = sum_k e4m3(xq[m, k]) * e4m3(wq[n, k])  (fp32),
// but at decode batch sizes the layer is bound by reading W once from HBM
// ("FP8 Inference Explained, in depth", "What FP8 buys during serving": decode
// speed is set by memory bandwidth), so the kernel is shaped around the weight
// stream:
//   * operands swapped: 128 rows of W fill the MMA's M = 128 side and the
//     tokens (padded to MT = 16/32/64 with TMA zero fill) the narrow N side,
//     so D^T[n, m] accumulates in TMEM (128 lanes x MT columns);
//   * split-K over a thread-block cluster of S CTAs (one cluster per 128-row
//     weight slab), sized so that the grid fills every SM with kCtasPerSm
//     CTAs: several small CTAs per SM keep more independent TMA producers in
//     flight than one deep ring (measured on GB300);
//   * each CTA streams its K slice of W through a TMA ring; the X tile of the
//     same K slice rides along in the same stage;
//   * the S partial D^T tiles are summed through distributed shared memory in
//     fixed rank order (deterministic), then scaled and stored as bf16 by
//     all CTAs of the cluster, each owning 128/S rows.
// Under programmatic dependent launch, what the kernel reads before
// griddepcontrol.wait depends on its predecessor: after the library's own
// quantizer (which releases it only once every earlier kernel has finished)
// it fills its ring with weights at once; otherwise it only prefetches the
// first weight tiles into L2, so an early start cannot observe stale inputs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "decode_common.cuh"
#include "ptx.cuh"

namespace fp8k {
namespace {

using namespace decode;
constexpr int kWBoxRows = 128;  // weight tile fetched as BNW / kWBoxRows boxes

template <int MT>
struct Cfg {
    static constexpr uint32_t X_TILE = MT * BK;
    static constexpr uint32_t STAGE_BYTES = W_TILE + X_TILE;
    static constexpr int STAGES = (kCtaSmem - 1024 - 512) / STAGE_BYTES;
    static_assert(STAGES >= 2, "ring depth");
    static constexpr uint32_t RING = STAGES * STAGE_BYTES;
    static constexpr uint32_t RED_BYTES = MT * BNW * 4;  // fp32 partial D^T, aliases the ring
    static_assert(RED_BYTES <= RING, "partial tile must fit in the ring");
    static_assert(STAGES <= 16, "barrier arrays hold 16 stages");
    static constexpr uint32_t TMEM_COLS = MT < 32 ? 32 : MT;
};

struct Bars {
    uint64_t full[16];
    uint64_t empty[16];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    float s_tok[64];  // token scales, staged once for the reduction
};

template <int MT>
constexpr size_t smem_bytes() {
    return 1024 + Cfg<MT>::RING + sizeof(Bars);
}

template <int MT>
__global__ void __launch_bounds__(kThreads)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX, const float* __restrict__ s_tok,
                       const float* __restrict__ s_w, __nv_bfloat16* __restrict__ y, int M, int N,
                       int K, int splits, int w_early, unsigned* status) {
    using C = Cfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    Bars* bars = reinterpret_cast<Bars*>(smem + C::RING);
    float* red = reinterpret_cast<float*>(smem);  // [MT][BNW], valid after the main loop
    uint8_t* ring = smem;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_blk = blockIdx.y;
    const uint32_t rank = cluster_ctarank();
    const int nk = (K + BK - 1) / BK;
    int kb0, nkb;
    split_range(static_cast<int>(rank), nk, splits, &kb0, &nkb);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->acc_full, 1);
        mbar_init(&bars->drain, 1);
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
    // the next kernel on the stream may start its prologue now (it waits for
    // this grid's completion before touching memory)
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;

    // Role loops run on whole warps (lane 0 issues, waits warp-uniform).
    if (warp == 0) {
        // ---- TMA producer ----
        const uint64_t w_policy = policy_evict_first();
        // Weights before the wait: when this launch follows the library's own
        // quantizer (w_early), every earlier kernel has finished, so the first
        // stages are filled with weights at once.  Otherwise only prefetch the
        // first weight tiles into L2 (the point of coherence): nothing stale can
        // reach shared memory even if the previous kernel still writes them.
        const int pre = w_early ? (nkb < C::STAGES ? nkb : C::STAGES) : 0;
        if (lane == 0) {
            if (w_early) {
                for (int i = 0; i < pre; ++i) {
                    mbar_arrive_expect_tx(&bars->full[i], C::STAGE_BYTES);
                    for (int b = 0; b < BNW / kWBoxRows; ++b)
                        tma_load_2d_hint(ring + i * C::STAGE_BYTES + b * kWBoxRows * BK, &tmW,
                                         &bars->full[i], (kb0 + i) * BK,
                                         n_blk * BNW + b * kWBoxRows, w_policy);
                }
            } else {
                const int pf = nkb < kL2PrefetchBlocks ? nkb : kL2PrefetchBlocks;
                for (int i = 0; i < pf; ++i)
                    for (int b = 0; b < BNW / kWBoxRows; ++b)
                        tma_prefetch_l2_2d(&tmW, (kb0 + i) * BK, n_blk * BNW + b * kWBoxRows);
            }
        }
        __syncwarp();
        pdl_wait_primary();
        if (lane == 0)
            for (int i = 0; i < pre; ++i)
                tma_load_2d(ring + i * C::STAGE_BYTES + W_TILE, &tmX, &bars->full[i],
                            (kb0 + i) * BK, 0);
        __syncwarp();
        uint32_t stage = pre % C::STAGES, phase = pre == C::STAGES ? 1u : 0u;
        for (int i = pre; i < nkb; ++i) {
            if (!warp_wait(&bars->empty[stage], phase ^ 1u, abort_flag, status)) break;
            if (lane == 0) {
                uint8_t* st = ring + stage * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&bars->full[stage], C::STAGE_BYTES);
                for (int b = 0; b < BNW / kWBoxRows; ++b)
                    tma_load_2d_hint(st + b * kWBoxRows * BK, &tmW, &bars->full[stage],
                                     (kb0 + i) * BK, n_blk * BNW + b * kWBoxRows, w_policy);
                tma_load_2d(st + W_TILE, &tmX, &bars->full[stage], (kb0 + i) * BK, 0);
            }
            __syncwarp();
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----
        pdl_wait_primary();
        constexpr uint32_t idesc = idesc_e4m3_f32(BNW, MT);
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            if (!(ok = warp_wait(&bars->full[stage], phase, abort_flag, status))) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = smem_u32(ring + stage * C::STAGE_BYTES);
                const uint64_t a0 = sdesc_kmajor_sw128(st);
                const uint64_t b0 = sdesc_kmajor_sw128(st + W_TILE);
#pragma unroll
                for (int kk = 0; kk < BK / KSTEP; ++kk)
                    mma_f8(tmem_base, a0 + 2 * kk, b0 + 2 * kk, idesc, (i | kk) != 0);
                mma_commit(&bars->empty[stage]);
            }
            __syncwarp();
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (lane == 0) {
            if (ok && nkb > 0) mma_commit(&bars->acc_full);
            mma_commit(&bars->drain);
            wait_drain(&bars->drain, status);
        }
        __syncwarp();
    } else {
        // ---- epilogue warps: TMEM lanes (= weight rows) of this warp's quarter ----
        pdl_wait_primary();
        const int quarter = warp & 3;
        const int nl = quarter * 32 + lane;
        float v[MT];
        bool have = false;
        if (nkb > 0) {
            have = warp_wait(&bars->acc_full, 0, abort_flag, status);
            if (have) {
                tc_fence_after();
                tmem_ld_cols<MT>(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16), v);
            }
        }
        if (!have) {
#pragma unroll
            for (int j = 0; j < MT; ++j) v[j] = 0.0f;
        }
        // The ring is idle once the accumulator is complete (every stage was
        // consumed by an MMA that has finished): reuse it for the partial.
#pragma unroll
        for (int j = 0; j < MT; ++j) red[j * BNW + nl] = v[j];
        if (warp == 2)
            for (int m = lane; m < M; m += 32) bars->s_tok[m] = __ldg(s_tok + m);
    }

    // All partials of the cluster are in shared memory after this barrier.
    cluster_sync_all();

    {
        // This CTA owns weight rows [lo, hi) of the slab.  Each thread keeps
        // one row (its weight scale in a register, its peers' partial
        // addresses mapped once) and walks tokens m = g, g + groups, ...; the
        // S partial loads of an output are independent, issued together and
        // summed in rank order (deterministic).
        const int rows_per = (BNW + splits - 1) / splits;
        const int lo = static_cast<int>(rank) * rows_per;
        const int hi = min(BNW, lo + rows_per);
        const int width = hi - lo;
        const int groups = width > 0 ? kThreads / width : 0;
        if (groups > 0 && static_cast<int>(threadIdx.x) < groups * width) {
            const int r = lo + static_cast<int>(threadIdx.x) % width;
            const int n = n_blk * BNW + r;
            const float sw = n < N ? __ldg(s_w + n) : 0.0f;
            const uint32_t base = smem_u32(red) + static_cast<uint32_t>(r * 4);
            uint32_t peer[kMaxSplits];
#pragma unroll
            for (int j = 0; j < kMaxSplits; ++j) peer[j] = j < splits ? map_to_rank(base, j) : 0u;
#pragma unroll 4
            for (int m = static_cast<int>(threadIdx.x) / width; m < M; m += groups) {
                const uint32_t off = static_cast<uint32_t>(m * BNW * 4);
                float part[kMaxSplits];
#pragma unroll
                for (int j = 0; j < kMaxSplits; ++j)
                    part[j] = j < splits ? ld_dsmem_f32(peer[j] + off) : 0.0f;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < kMaxSplits; ++j)
                    if (j < splits) acc += part[j];
                if (n < N)
                    y[static_cast<int64_t>(m) * N + n] =
                        __float2bfloat16_rn((acc * bars->s_tok[m]) * sw);
            }
        }
    }

    // Peers may still be reading this CTA's partial.
    cluster_sync_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int MT>
cudaError_t launch_mt(const GemmArgs& a) {
    CUtensorMap tmW, tmX;
    if (!encode_tmap_u8(&tmW, a.wq, a.N, a.K, a.K, BK, kWBoxRows)) return cudaErrorInvalidValue;
    if (!encode_tmap_u8(&tmX, a.xq, a.M, a.K, a.K, BK, MT)) return cudaErrorInvalidValue;
    const int n_tiles = (a.N + BNW - 1) / BNW;
    const int nk = (a.K + BK - 1) / BK;
    const int splits = choose_splits(n_tiles, nk, a.num_sms);

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(splits, n_tiles);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes<MT>();
    cfg.stream = a.stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_decode_kernel<MT>, tmW, tmX, a.s_tok, a.s_w,
                              static_cast<__nv_bfloat16*>(a.y), a.M, a.N, a.K, splits,
                              a.w_early ? 1 : 0, a.status);
}

}  // namespace

cudaError_t prepare_gemm_decode() {
    cudaError_t e;
    for (auto* k : {gemm_decode_kernel<16>, gemm_decode_kernel<32>, gemm_decode_kernel<64>}) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(gemm_decode_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<16>()));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_decode_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<32>()));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_decode_kernel<64>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem_bytes<64>()));
}

cudaError_t launch_gemm_decode(const GemmArgs& a) {
    if (a.M <= 16) return launch_mt<16>(a);
    if (a.M <= 32) return launch_mt<32>(a);
    return launch_mt<64>(a);
}

}  // namespace fp8k
