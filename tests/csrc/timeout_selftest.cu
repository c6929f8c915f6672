// Self-test of the bounded pipeline waits in
// paged_split_kv_gather_gb300/csrc/device_utils.cuh and split_common.cuh (test
// infrastructure).
//
// One CTA of two warps.  An mbarrier is initialised with an arrival count of
// one and nothing ever arrives on it, so a wait on its first phase can only end
// by giving up.  Warp 0 waits through the consumer-side helper (wait_stage),
// warp 1 through the raw bounded wait; each must return false after the
// library's limit (kWaitLimitNs) and record FDEC_DEVERR_TIMEOUT in the error
// word, exactly as the split kernels do, after which the kernel returns
// normally: no copy is in flight, so nothing outlives the CTA.
#include <cstdint>

#include "../../paged_split_kv_gather_gb300/csrc/split_common.cuh"

using namespace fdec;

__global__ void __launch_bounds__(64) timeout_selftest_kernel(unsigned* err, unsigned long long* waited_ns) {
    __shared__ __align__(8) uint64_t bars[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bars[0]), 1);  // full[0] of a one-stage ring: nothing will fill it
        mbar_init(smem_addr(&bars[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    const uint64_t t0 = global_timer_ns();
    bool ok;
    if (warp == 0) {
        ok = wait_stage<1>(bars, 0);  // stage 0 completes bars[0 % 2] in phase 0
    } else {
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(smem_addr(&bars[1]), 0);
        ok = __shfl_sync(0xffffffffu, got, 0) != 0;
    }
    const uint64_t t1 = global_timer_ns();
    if (!ok && lane == 0) {
        atomicOr(err, FDEC_DEVERR_TIMEOUT << (8 * warp));
        waited_ns[warp] = t1 - t0;
    }
}

extern "C" int timeout_selftest(void* err, void* waited_ns) {
    timeout_selftest_kernel<<<1, 64>>>(static_cast<unsigned*>(err), static_cast<unsigned long long*>(waited_ns));
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" unsigned long long timeout_selftest_limit_ns() { return kWaitLimitNs; }
