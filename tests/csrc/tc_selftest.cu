// Self-test of the tcgen05 operand layouts and descriptors in
// paged_split_kv_gather_gb300/csrc/tc_common.cuh (test infrastructure).
//
//   D1 (128 x 64)  = A (128 x 128, K-major) * B (64 x 128, K-major)^T
//   D2 (128 x 128) = P (128 x 64, K-major)  * V (64 x 128, MN-major: stored [k][n])
//   D3 (128 x 128) = P (128 x 64, in tensor memory: lane = row, element pairs per
//                    32-bit column) * V (as for D2)
//
// One CTA of 128 threads; all operands are copied into 128B-swizzled shared
// memory by plain stores, the MMAs are issued by thread 0, and the four warps
// read the accumulators back from tensor memory.
#include <cstdint>

#include "../../paged_split_kv_gather_gb300/csrc/device_utils.cuh"
#include "../../paged_split_kv_gather_gb300/csrc/tc_common.cuh"

using namespace fdec;

// Byte offset of element (row, e) in a swizzled operand whose rows hold 64-element
// blocks (regions of `rows` x 128 B).
__device__ __forceinline__ uint32_t swz(int row, int e, int rows) {
    const int region = e >> 6, within = e & 63;
    return region * rows * 128 + row * 128 + ((((within >> 3) ^ (row & 7)) & 7) << 4) + (within & 7) * 2;
}

__global__ void __launch_bounds__(128) tc_selftest_kernel(const uint16_t* a, const uint16_t* b, const uint16_t* pm,
                                                         const uint16_t* v, float* d1, float* d2, float* d3,
                                                         unsigned* err) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t base = smem_addr(smem);
    uint8_t* s = smem + ((1024u - (base & 1023u)) & 1023u);
    uint8_t* sa_ = s;              // 2 regions x 128 rows x 128 B = 32 KB
    uint8_t* sb_ = s + 32768;      // 2 regions x 64 rows = 16 KB
    uint8_t* sp_ = s + 49152;      // 1 region x 128 rows = 16 KB
    uint8_t* sv_ = s + 65536;      // 2 regions x 64 rows (K) = 16 KB
    uint64_t* bar = reinterpret_cast<uint64_t*>(s + 81920);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s + 81920 + 64);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int i = tid; i < 128 * 128; i += 128) {
        const int r = i / 128, e = i % 128;
        *reinterpret_cast<uint16_t*>(sa_ + swz(r, e, 128)) = a[i];
    }
    for (int i = tid; i < 64 * 128; i += 128) {
        const int r = i / 128, e = i % 128;
        *reinterpret_cast<uint16_t*>(sb_ + swz(r, e, 64)) = b[i];
        *reinterpret_cast<uint16_t*>(sv_ + swz(r, e, 64)) = v[i];  // V stored [k = r][n = e]
    }
    for (int i = tid; i < 128 * 64; i += 128) {
        const int r = i / 64, e = i % 64;
        *reinterpret_cast<uint16_t*>(sp_ + swz(r, e, 128)) = pm[i];
    }
    if (tid == 0) {
        mbar_init(smem_addr(bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), 512);
        tmem_relinquish();
    }
    fence_proxy_async_shared();  // the generic stores above are read by the tensor cores
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    {  // row `row` of P into tensor-memory columns 256..287 of this lane
        uint32_t w[32];
        for (int c = 0; c < 32; ++c)
            w[c] = static_cast<uint32_t>(pm[row * 64 + 2 * c]) | (static_cast<uint32_t>(pm[row * 64 + 2 * c + 1]) << 16);
        tmem_st32_u(lane_addr + 256, w);
        tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    if (tid == 0) {
        const uint32_t i1 = idesc_f16(128, 64, true, false, false);
        for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = smem_desc_sw128(smem_addr(sa_) + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(smem_addr(sb_) + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
            tc_mma_f16(tmem, ad, bd, i1, ks > 0);
        }
        const uint32_t i2 = idesc_f16(128, 128, true, false, true);
        for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ad = smem_desc_sw128(smem_addr(sp_) + ks * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(smem_addr(sv_) + ks * 2048, 8192, 1024);
            tc_mma_f16(tmem + 128, ad, bd, i2, ks > 0);
        }
        for (int ks = 0; ks < 4; ++ks) {  // A from tensor memory: 8 columns (16 K elements) per step
            const uint64_t bd = smem_desc_sw128(smem_addr(sv_) + ks * 2048, 8192, 1024);
            tc_mma_f16_ts(tmem + 384, tmem + 256 + ks * 8, bd, i2, ks > 0);
        }
        tc_commit(smem_addr(bar));
    }
    if (!mbar_wait_bounded(smem_addr(bar), 0)) {
        if (lane == 0) atomicOr(err, 1u);
    }
    tc_fence_after_sync();
    float vals[32];
    for (int c = 0; c < 64; c += 32) {
        tmem_ld32(lane_addr + c, vals);
        tmem_wait_ld();
        for (int j = 0; j < 32; ++j) d1[row * 64 + c + j] = vals[j];
    }
    for (int c = 0; c < 128; c += 32) {
        tmem_ld32(lane_addr + 128 + c, vals);
        tmem_wait_ld();
        for (int j = 0; j < 32; ++j) d2[row * 128 + c + j] = vals[j];
        tmem_ld32(lane_addr + 384 + c, vals);
        tmem_wait_ld();
        for (int j = 0; j < 32; ++j) d3[row * 128 + c + j] = vals[j];
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

extern "C" int tc_selftest(const uint16_t* a, const uint16_t* b, const uint16_t* p, const uint16_t* v, float* d1,
                           float* d2, float* d3, unsigned* err) {
    const int smem = 81920 + 1024 + 1024;
    if (cudaFuncSetAttribute(tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 1;
    tc_selftest_kernel<<<1, 128, smem>>>(a, b, p, v, d1, d2, d3, err);
    if (cudaGetLastError() != cudaSuccess) return 2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
