// Scaled FP8 GEMM for decode-sized and mid-size M (M <= 256 tokens): weight
// streaming.
//
// Same result as the paired-SM kernel (gemm_pair.cu),
//   y[m, n] = bf16_rn((acc[m, n] * s_tok[m]) * s_w[n]),
//   acc[m, n] = sum_k e4m3(xq[m, k]) * e4m3(wq[n, k])  (fp32),
// but at decode batch sizes the layer is bound by reading W once from HBM
// ("FP8 Inference Explained, in depth", "What FP8 buys during serving": decode
// speed is set by memory bandwidth), so the kernel is shaped around the weight
// stream:
//   * operands swapped: 128 rows of W fill the MMA's M = 128 side and the
//     tokens (padded to MT = 16/32/64/128/256 with TMA zero fill) the N side,
//     so D^T[n, m] accumulates in TMEM (128 lanes x MT columns); 128- and
//     256-token tiles (32 and 48 KB ring stages, 64 and 128 KB partials) run
//     two CTAs or one per SM, the narrower ones kCtasPerSm;
//   * split-K over a thread-block cluster of S CTAs (one cluster per 128-row
//     weight slab), sized so that the grid fills every SM with as many CTAs
//     as the tile width allows: several small CTAs per SM keep more
//     independent TMA producers in flight than one deep ring (measured on
//     GB300);
//   * each CTA streams its K slice of W through a TMA ring; the X tile of the
//     same K slice rides along in the same stage;
//   * each CTA of the cluster owns 128/S rows of the slab's output and sums
//     their S partials in fixed rank order (deterministic), scales them and
//     stores bf16.  Up to 16 tokens every CTA sends the partial rows of each
//     owner straight into a dedicated receive buffer of that owner (st.async,
//     counted on the owner's mbarrier): the partials leave as soon as the
//     accumulator is read, and no cluster barrier is needed.  Wider token
//     tiles (whose buffer would cost a ring stage) leave their partial in the
//     idle ring; owners pull after a cluster barrier, and a second barrier
//     keeps every CTA alive until its peers have read it.
// Under programmatic dependent launch the kernel may start while earlier
// kernels still run (the quantizer before it releases it at once): before
// griddepcontrol.wait it only prefetches its first weight tiles into L2, the
// point of coherence, so an early start cannot observe stale inputs.
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
constexpr int kMaxStages = 8;

template <int MT>
struct Cfg {
    static constexpr uint32_t X_TILE = MT * BK;
    static constexpr uint32_t STAGE_BYTES = W_TILE + X_TILE;
    static constexpr uint32_t TMEM_COLS = MT < 32 ? 32 : MT;
    static constexpr uint32_t RED_BYTES = MT * BNW * 4;  // pull: partial D^T in the ring
};

template <int MT>
struct Bars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full;
    uint64_t drain;
    uint64_t recv_full;  // push: the S partials of this CTA's rows have arrived
    uint32_t tmem_base;
    int abort;
    float s_tok[MT < 64 ? 64 : MT];  // token scales, staged for the reduction
    float s_w[BNW];    // weight scales of the rows this CTA reduces
};

// Shared-memory layout of one launch: [ring | receive buffer | Bars], after
// up to 1 KB of alignment.  The receive buffer (push only) holds
// [S][rows_per][Mp + 4] fp32 partials (Mp = M rounded up to 4; the padding
// spreads the rows of one token over the shared-memory banks).  The ring
// gets what is left of the per-CTA budget that lets kCtasPerSm CTAs share
// an SM.
struct Layout {
    uint32_t recv_bytes;
    int stages;
    size_t smem;
};

template <int MT, bool PUSH>
Layout layout_of(int M, int splits, int64_t budget) {
    using C = Cfg<MT>;
    Layout l;
    l.recv_bytes = PUSH ? push_recv_bytes(M, splits) : 0u;
    const int64_t room =
        budget - 1024 - static_cast<int64_t>(sizeof(Bars<MT>)) - l.recv_bytes;
    int st = static_cast<int>(room / C::STAGE_BYTES);
    l.stages = st < kMaxStages ? st : kMaxStages;
    l.smem = 1024 + static_cast<size_t>(l.stages) * C::STAGE_BYTES + l.recv_bytes + sizeof(Bars<MT>);
    return l;
}

// Barrier of the four epilogue warps (named barrier 1, 128 threads).
__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// y[m, n] = bf16((v[j] * s_tok[m]) * s_w_n) for tokens m = m0 + j < M, one
// weight row n per lane (a warp stores 32 consecutive outputs of a token).
template <int NV>
__device__ __forceinline__ void store_rows_direct(const float (&v)[NV], int m0, int M, int N,
                                                  int n, const float* s_tok, float s_w_n,
                                                  __nv_bfloat16* __restrict__ y) {
    if (n >= N) return;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int m = m0 + j;
        if (m < M)
            y[static_cast<int64_t>(m) * N + n] = __float2bfloat16_rn((v[j] * s_tok[m]) * s_w_n);
    }
}

// PUSH: partials pushed into a dedicated receive buffer (no cluster barrier
// after the main loop); otherwise pulled from the idle ring, or, unsplit
// (S = 1), stored by each CTA straight from its accumulator.
template <int MT, bool PUSH>
__global__ void __launch_bounds__(kThreads)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX, const float* __restrict__ s_tok,
                       const float* __restrict__ s_w, __nv_bfloat16* __restrict__ y, int M, int N,
                       int K, int splits, int stages, uint32_t recv_bytes, unsigned* status) {
    using C = Cfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* ring = smem;
    float* recv = reinterpret_cast<float*>(smem + stages * C::STAGE_BYTES);  // push
    Bars<MT>* bars = reinterpret_cast<Bars<MT>*>(smem + stages * C::STAGE_BYTES + recv_bytes);
    float* red = reinterpret_cast<float*>(smem);  // pull: [MT][BNW], after the main loop

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_blk = blockIdx.y;
    const uint32_t rank = cluster_ctarank();
    const int nk = (K + BK - 1) / BK;
    int kb0, nkb;
    split_range(static_cast<int>(rank), nk, splits, &kb0, &nkb);
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
        mbar_init(&bars->acc_full, 1);
        mbar_init(&bars->drain, 1);
        if constexpr (PUSH) {
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
    // the next kernel on the stream may start its prologue now (it waits for
    // this grid's completion before touching memory)
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Push: peers may send partials once every CTA's barriers are
    // initialised (first half of a split cluster barrier; the wait comes
    // before sending).
    if constexpr (PUSH) cluster_arrive();
    const uint32_t tmem_base = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;

    // Role loops run on whole warps (lane 0 issues, waits warp-uniform).
    if (warp == 0) {
        // ---- TMA producer ----
        const uint64_t w_policy = policy_evict_first();
        // Before the wait only prefetch the first weight tiles into L2 (the
        // point of coherence): nothing stale can reach shared memory even if
        // an earlier kernel still writes them.
        if (lane == 0) {
            const int pf = nkb < kL2PrefetchBlocks ? nkb : kL2PrefetchBlocks;
            for (int i = 0; i < pf; ++i)
                for (int b = 0; b < BNW / kWBoxRows; ++b)
                    tma_prefetch_l2_2d(&tmW, (kb0 + i) * BK, n_blk * BNW + b * kWBoxRows);
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
                for (int b = 0; b < BNW / kWBoxRows; ++b)
                    tma_load_2d_hint(st + b * kWBoxRows * BK, &tmW, &bars->full[stage],
                                     (kb0 + i) * BK, n_blk * BNW + b * kWBoxRows, w_policy);
                tma_load_2d(st + W_TILE, &tmX, &bars->full[stage], (kb0 + i) * BK, 0);
            }
            __syncwarp();
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----
        pdl_wait_primary();
        constexpr uint32_t idesc = idesc_e4m3_f32(BNW, MT);
        int stage = 0;
        uint32_t phase = 0;
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
            if (++stage == stages) {
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
        // Stage the scales the reduction needs while the main loop runs, so
        // no global load sits between the accumulator and the output.
        if (warp == 2) {
            for (int m = lane; m < M; m += 32) bars->s_tok[m] = __ldg(s_tok + m);
        } else if (warp == 3) {
            for (int r = lo + lane; r < hi; r += 32) {
                const int n = n_blk * BNW + r;
                bars->s_w[r] = n < N ? __ldg(s_w + n) : 0.0f;
            }
        }
        const int quarter = warp & 3;
        const int nl = quarter * 32 + lane;
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        bool have = false;
        if constexpr (MT <= 64) {
            float v[MT];
            if (nkb > 0) {
                have = warp_wait(&bars->acc_full, 0, abort_flag, status);
                if (have) {
                    tc_fence_after();
                    tmem_ld_cols<MT>(tacc, v);
                }
            }
            tc_fence_before();
            if (!have) {
#pragma unroll
                for (int j = 0; j < MT; ++j) v[j] = 0.0f;
            }
            if constexpr (PUSH) {
                // Sent even after a failed wait (as zeros) so that every
                // owner's barrier completes.
                cluster_wait();
                push_send<MT>(v, M, nl, rank, splits, recv, &bars->recv_full);
            } else if (splits == 1) {
                // Unsplit: this CTA owns the whole slab; scale and store
                // straight from registers (no ring copy, no cluster barrier).
                epi_bar_sync();  // the scales staged by warps 2 and 3
                store_rows_direct<MT>(v, 0, M, N, n_blk * BNW + nl, bars->s_tok,
                                      bars->s_w[nl], y);
            } else {
                // The ring is idle once the accumulator is complete (every
                // stage was consumed by an MMA that has finished): reuse it.
#pragma unroll
                for (int j = 0; j < MT; ++j) red[j * BNW + nl] = v[j];
            }
        } else {
            static_assert(!PUSH, "wide token tiles pull");
            // The same through the idle ring, 32 token columns at a time
            // (a wide tile's accumulator row would not fit in registers).
            if (nkb > 0) have = warp_wait(&bars->acc_full, 0, abort_flag, status);
            if (have) tc_fence_after();
            if (splits == 1) epi_bar_sync();  // the scales staged by warps 2 and 3
#pragma unroll 1
            for (int h = 0; h < MT / 32; ++h) {
                uint32_t r[32];
                if (have) {
                    tmem_ld_32x32b_x32(tacc + h * 32, r);
                    tmem_ld_wait();
                }
                if (splits == 1) {
                    // unsplit: scale and store straight from registers
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = have ? __uint_as_float(r[j]) : 0.0f;
                    store_rows_direct<32>(v, h * 32, M, N, n_blk * BNW + nl, bars->s_tok,
                                          bars->s_w[nl], y);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        red[(h * 32 + j) * BNW + nl] = have ? __uint_as_float(r[j]) : 0.0f;
                }
            }
            tc_fence_before();
        }
    }

    // y[m, n] = bf16((sum * s_tok[m]) * s_w[n]) for slab row r
    auto store = [&](int m, int r, float acc) {
        const int n = n_blk * BNW + r;
        if (n < N)
            y[static_cast<int64_t>(m) * N + n] =
                __float2bfloat16_rn((acc * bars->s_tok[m]) * bars->s_w[r]);
    };
    if constexpr (PUSH) {
        if (warp < 2) cluster_wait();
        // every tcgen05 operation of this CTA has completed: free TMEM
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem_base, C::TMEM_COLS);
        }
        // The S partials of rows [lo, hi) arrive from every CTA of the
        // cluster (this one included).  Nothing remote touches this CTA
        // afterwards, so it may exit without a barrier.
        if (warp_wait_cluster_noabort(&bars->recv_full, 0, 4 * kWaitLimitNs, status))
            push_reduce(recv, splits, lo, width, M, store);
        else
            outlive_peers();
    } else if (splits == 1) {
        // unsplit: the epilogue warps have stored the outputs; every tcgen05
        // operation has completed once all warps are here
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem_base, C::TMEM_COLS);
        }
    } else {
        // All partials of the cluster are in shared memory after this
        // barrier, and every tcgen05 operation of this CTA has completed.
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

template <int MT, bool PUSH>
cudaError_t launch_mt(const GemmArgs& a, int splits, uint32_t budget) {
    CUtensorMap tmW, tmX;
    if (!encode_tmap_u8(&tmW, a.wq, a.N, a.K, a.K, BK, kWBoxRows)) return cudaErrorInvalidValue;
    if (!encode_tmap_u8(&tmX, a.xq, a.M, a.K, a.K, BK, MT)) return cudaErrorInvalidValue;
    const int n_tiles = (a.N + BNW - 1) / BNW;
    const Layout l = layout_of<MT, PUSH>(a.M, splits, budget);
    if (l.stages < 2 ||
        (!PUSH && splits > 1 && Cfg<MT>::RED_BYTES > l.stages * Cfg<MT>::STAGE_BYTES))
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
    return cudaLaunchKernelEx(&cfg, gemm_decode_kernel<MT, PUSH>, tmW, tmX, a.s_tok, a.s_w,
                              static_cast<__nv_bfloat16*>(a.y), a.M, a.N, a.K, splits, l.stages,
                              l.recv_bytes, a.status);
}

// Never launched: the occupancy calculator's stand-in for the decode GEMMs
// (same block size and shared-memory footprint, which is what limits them
// to kCtasPerSm CTAs per SM).  Asked about the real kernels, the calculator
// reports one CTA per SM for cluster launches, while three are resident
// (measured); for this stand-in it reports the residency that is measured.
__global__ void __launch_bounds__(kThreads) decode_residency_probe() {}

}  // namespace

int gemm_decode_resident_clusters(int size, int ctas_per_sm) {
    const uint32_t smem = ctas_per_sm >= 3 ? kCtaSmem : ctas_per_sm == 2 ? kCtaSmem2 : kCtaSmem1;
    if (cudaFuncSetAttribute(decode_residency_probe, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(decode_residency_probe,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(size, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_residency_probe, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t prepare_gemm_decode() {
    struct {
        const void* k;
        uint32_t smem;
    } const kernels[] = {
        {reinterpret_cast<const void*>(gemm_decode_kernel<16, true>), kCtaSmem2},
        {reinterpret_cast<const void*>(gemm_decode_kernel<32, false>), kCtaSmem2},
        {reinterpret_cast<const void*>(gemm_decode_kernel<64, false>), kCtaSmem2},
        {reinterpret_cast<const void*>(gemm_decode_kernel<128, false>), kCtaSmem2},
        {reinterpret_cast<const void*>(gemm_decode_kernel<256, false>), kCtaSmem1},
    };
    for (const auto& k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(k.k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k.k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(k.smem));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_decode(const GemmArgs& a) {
    const int n_tiles = (a.N + BNW - 1) / BNW;
    const int* clusters3 = a.decode_clusters ? a.decode_clusters + 2 * 9 : nullptr;
    const int nk = (a.K + BK - 1) / BK;
    // pushed partials (up to 16 tokens): the busy-slot rule; pulled: the
    // target-CTA rule
    const int splits = a.M <= 16 ? choose_splits(n_tiles, nk, a.num_sms, clusters3)
                                 : choose_splits_pull(n_tiles, nk, clusters3);
    // A grid of at most two CTAs per SM gets the two-per-SM budget: a 4-5
    // stage ring instead of 3 (measured on the 8B decode step, 3852 -> 3923
    // GB/s; limiting it to token tiles of up to 16 was slower).  Partials are
    // pushed up to 16 tokens and pulled beyond (pushing at 32 tokens in the
    // two-per-SM grids, where the receive buffer fits beside a 4-stage ring,
    // measured 3924 against 3960 GB/s for the step).
    const bool two = static_cast<int64_t>(n_tiles) * splits <= 2 * a.num_sms;
    const uint32_t budget = two ? kCtaSmem2 : kCtaSmem;
    if (a.M <= 16) return launch_mt<16, true>(a, splits, budget);
    if (a.M <= 32) return launch_mt<32, false>(a, splits, budget);
    if (a.M <= 64) return launch_mt<64, false>(a, splits, budget);
    // Wider token tiles: a 32 KB (128 tokens) or 48 KB (256) ring stage and a
    // 64 / 128 KB partial, so two CTAs or one share an SM; the split is
    // chosen for that footprint by the fewest-waves rule.
    const int* clusters2 = a.decode_clusters ? a.decode_clusters + 1 * 9 : nullptr;
    const int* clusters1 = a.decode_clusters;
    if (a.M <= 128)
        return launch_mt<128, false>(
            a, choose_splits_min_waves(n_tiles, nk, 2 * a.num_sms, clusters2), kCtaSmem2);
    // Unsplit, a 256-token tile needs no ring room for a partial: two CTAs
    // (two 48 KB stages each) then share an SM.
    const int s256 = choose_splits_min_waves(n_tiles, nk, a.num_sms, clusters1);
    return launch_mt<256, false>(a, s256, s256 == 1 ? kCtaSmem2 : kCtaSmem1);
}

}  // namespace fp8k
