// Tensor-pipe rate of the tcgen05 MMA shapes the dense-query kernel issues
// (test infrastructure).  One CTA per SM, one issuing thread: `iters` rounds of
// eight M128 x K16 products of one shape, back to back, then one commit and a
// bounded wait.  Operands are zeros (the rate does not depend on the values).
//
// Shapes (mode):
//   0  Q K^T form: A and B K-major in shared memory, N 64
//   1  Q K^T form with A in tensor memory, N 64
//   2  P V form: A (P) in tensor memory, B (V) MN-major, N 128
//   3  A and B K-major in shared memory, N 128
//   4  A and B K-major in shared memory, N 256
//   5  one 64-token block of the two-tile kernel, per tile: 4 P V (N 128, A in
//      tensor memory) then 8 Q K^T (N 64, A in tensor memory)
#include <cstdint>

#include "../../paged_split_kv_gather_gb300/csrc/device_utils.cuh"
#include "../../paged_split_kv_gather_gb300/csrc/tc_common.cuh"

using namespace fdec;

__global__ void __launch_bounds__(128, 1) tc_mma_rate_kernel(int mode, int iters, unsigned* err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    // operands: A at [0, 16 KB), B at [32 KB, 64 KB)
    for (int i = threadIdx.x; i < 65536 / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(smem_addr(&tslot), 512);
        tmem_relinquish();
    }
    fence_proxy_async_shared();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = tslot;
    if (threadIdx.x == 0) {
        const uint64_t da = smem_desc_sw128(smem_addr(sm), 16, 1024);
        const uint64_t db = smem_desc_sw128(smem_addr(sm + 32768), 16, 1024);
        const uint64_t dv = smem_desc_sw128(smem_addr(sm + 32768), 8192, 1024);  // MN-major, 64-element blocks 8 KB apart
        const uint32_t i64 = idesc_f16(128, 64, false, false, false);
        const uint32_t i128 = idesc_f16(128, 128, false, false, false);
        const uint32_t i256 = idesc_f16(128, 256, false, false, false);
        const uint32_t i128v = idesc_f16(128, 128, false, false, true);
        // tensor memory: accumulators in columns 0..255, A operands at 256 (8 columns per K step)
        for (int it = 0; it < iters; ++it) {
            switch (mode) {
                case 0:
                    for (int ks = 0; ks < 8; ++ks) tc_mma_f16(tm, da + (ks & 3) * 2, db + (ks & 3) * 2, i64, ks > 0);
                    break;
                case 1:
                    for (int ks = 0; ks < 8; ++ks) tc_mma_f16_ts(tm, tm + 256 + 8 * (ks & 3), db + (ks & 3) * 2, i64, ks > 0);
                    break;
                case 2:
                    for (int ks = 0; ks < 8; ++ks) tc_mma_f16_ts(tm, tm + 256 + 8 * (ks & 3), dv + (ks & 1) * 128, i128v, ks > 0);
                    break;
                case 3:
                    for (int ks = 0; ks < 8; ++ks) tc_mma_f16(tm, da + (ks & 3) * 2, db + (ks & 3) * 2, i128, ks > 0);
                    break;
                case 4:
                    for (int ks = 0; ks < 8; ++ks) tc_mma_f16(tm, da + (ks & 3) * 2, db + (ks & 3) * 2, i256, ks > 0);
                    break;
                default:  // 5: per tile t (256 columns each): O at +64, S at +0, P and Q read at +0 / +192
                    for (int t = 0; t < 2; ++t) {
                        const uint32_t base = tm + 256 * t;
                        for (int ks = 0; ks < 4; ++ks) tc_mma_f16_ts(base + 64, base + 8 * ks, dv + (ks & 1) * 128, i128v, true);
                        for (int ks = 0; ks < 8; ++ks) tc_mma_f16_ts(base, base + 192 + 8 * (ks & 3), db + (ks & 3) * 2, i64, ks > 0);
                    }
                    break;
            }
        }
        tc_commit(smem_addr(&bar));
        if (!mbar_wait_bounded(smem_addr(&bar), 0)) atomicAdd(err, 1u);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) tmem_dealloc(tm, 512);
}

// Runs `iters` rounds of `mode` on every SM after a short warm-up launch; writes the
// launch's time in milliseconds (CUDA events) to *ms.  Returns 0, or a nonzero code
// on a CUDA error.
extern "C" int tc_mma_rate(int mode, int iters, unsigned* err, float* ms) {
    const int smem = 200 * 1024;  // one CTA per SM
    if (cudaFuncSetAttribute(tc_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 1;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess) return 2;
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return 3;
    tc_mma_rate_kernel<<<sms, 128, smem>>>(mode, iters / 20 + 1, err);
    cudaEventRecord(a);
    tc_mma_rate_kernel<<<sms, 128, smem>>>(mode, iters, err);
    cudaEventRecord(b);
    const cudaError_t e = cudaEventSynchronize(b);
    if (e == cudaSuccess) cudaEventElapsedTime(ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : 4;
}
