// Self-test of the bounded waits that every GEMM kernel of the library uses.
//
// The GEMM kernels never wait without a limit: each mbarrier wait gives up
// after a fixed time, raises a CTA-wide abort flag that makes the other
// roles of the CTA give up too, drains the tensor-core operations it issued,
// frees its tensor memory, sets a bit in the device status word and returns
// (fp8_device_status() then reports FP8_ERR_TIMEOUT).  In a correct run none
// of this happens, so this kernel makes it happen on purpose, with the same
// primitives and the same teardown order as the decode GEMM, on a barrier
// that nothing ever arrives on and with a short caller-given limit:
//   warp 0  (MMA issuer role)  waits for a ring stage that is never filled,
//           gives up after limit_ns, commits and drains, as the GEMMs do;
//   warp 1  allocates and frees 32 TMEM columns around the test;
//   warp 2  (epilogue role)    waits for an accumulator that is never
//           committed, with the GEMMs' own long limit, and must return as
//           soon as the issuer's abort flag is up.
// Nothing faults and nothing waits without a bound: the kernel ends after
// about limit_ns, and the context stays usable.
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace fp8k {
namespace {

struct SelfTestShared {
    uint64_t full;      // a ring stage: no producer ever arrives on it
    uint64_t acc_full;  // an accumulator: no MMA is ever committed to it
    uint64_t drain;     // the issuer's teardown commit
    uint32_t tmem_base;
    int abort;
};

__global__ void __launch_bounds__(96)
    wait_timeout_selftest(uint64_t limit_ns, unsigned* status, unsigned long long* report) {
    __shared__ SelfTestShared sh;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&sh.full, 1);
        mbar_init(&sh.acc_full, 1);
        mbar_init(&sh.drain, 1);
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    volatile int* abort_flag = &sh.abort;
    const uint64_t t0 = globaltimer_ns();
    if (warp == 0) {
        const bool ok = warp_wait(&sh.full, 0, abort_flag, status, limit_ns);
        if (lane == 0) {
            // teardown of the GEMMs' issuer: the commit arrives once every
            // tcgen05 operation this thread issued has completed (none here)
            mma_commit(&sh.drain);
            wait_drain(&sh.drain, status);
            report[0] = ok ? 0ull : 1ull;
            report[2] = globaltimer_ns() - t0;
        }
        __syncwarp();
    } else if (warp == 2) {
        const bool have = warp_wait(&sh.acc_full, 0, abort_flag, status);
        if (lane == 0) {
            report[1] = have ? 0ull : 1ull;
            report[3] = globaltimer_ns() - t0;
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(sh.tmem_base, 32);
    }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, unsigned* status,
                                         unsigned long long* report, cudaStream_t st) {
    wait_timeout_selftest<<<1, 96, 0, st>>>(limit_ns, status, report);
    return cudaGetLastError();
}

}  // namespace fp8k
