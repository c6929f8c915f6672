// append.cu -- paged KV append: scatter new tokens' K and V rows into the pages
// the page table names (the write side of the cache), for 16-bit caches and for
// E4M3 code caches alike (rows are moved as bytes).
//
// warps_per_token warps per new token (grid-stride over tokens): the token's
// sequence, position and page id are read once per warp, then the lanes stride over
// the 16-byte chunks of its K rows and V rows (every KV head), four chunks in flight
// per lane, loads before stores.  One warp per token when there are many tokens;
// when there are few, enough warps that each lane moves one chunk.  Each chunk lands at base + page * stride_page + head * stride_head +
// slot * stride_token of its pool.  HBM-bound: the new rows are read once and
// written once.  (Measured on 64 sequences x 512 tokens, 8 KV heads, D 128: one
// thread per chunk, each reading the token's indices and page id itself, took
// 57.3 us: its dependent loads, one chunk per thread at a time, left it
// latency-bound.)
#include <algorithm>
#include <atomic>
#include <cstdint>

#include "../../include/fdec.h"
#include "fdec_internal.h"

namespace fdec {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) append_kernel(AppendParams p, int wpt) {
    constexpr int U = 4;  // chunks in flight per lane
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int chunks_row = p.row_bytes / 16;
    const int per_kv = p.hk * chunks_row;  // chunks of the token's K rows (and of its V rows)
    const int page_mask = (1 << p.page_shift) - 1;
    for (int64_t w = warp0; w < static_cast<int64_t>(p.n_tokens) * wpt; w += nwarps) {
        const int64_t i = w / wpt;
        const int sub = static_cast<int>(w - i * wpt);
        const int b = __ldg(p.batch_indices + i);
        const int t = __ldg(p.positions + i);
        const int pi = t >> p.page_shift;
        if (t < 0 || pi >= p.pt_stride || b < 0 || b >= p.batch) {
            if (lane == 0 && sub == 0 && p.err != nullptr) atomicOr(p.err, FDEC_DEVERR_SEQ_LEN);
            continue;
        }
        const int page = __ldg(p.page_table + static_cast<int64_t>(b) * p.pt_stride + pi);
        if (page < 0 || page >= p.k_pages || page >= p.v_pages) {  // the token is skipped for K and V alike
            if (lane == 0 && sub == 0 && p.err != nullptr) atomicOr(p.err, FDEC_DEVERR_PAGE_ID);
            continue;
        }
        const int64_t slot = t & page_mask;
        const uint8_t* ksrc = p.k_new + i * p.new_st;
        const uint8_t* vsrc = p.v_new + i * p.new_st;
        uint8_t* kdst = p.k_base + static_cast<int64_t>(page) * p.k_sp + slot * p.k_st;
        uint8_t* vdst = p.v_base + static_cast<int64_t>(page) * p.v_sp + slot * p.v_st;
        for (int c0 = sub * 32 + lane; c0 < 2 * per_kv; c0 += 32 * wpt * U) {
            uint4 val[U];
            uint8_t* dst[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * wpt * u;  // K chunks first, then V chunks
                dst[u] = nullptr;
                if (c < 2 * per_kv) {
                    const bool is_v = c >= per_kv;
                    const int cc = is_v ? c - per_kv : c;
                    const int h = cc / chunks_row, ch = cc - h * chunks_row;
                    val[u] = __ldg(reinterpret_cast<const uint4*>((is_v ? vsrc : ksrc) + h * p.new_sh + ch * 16));
                    dst[u] = (is_v ? vdst : kdst) + h * (is_v ? p.v_sh : p.k_sh) + ch * 16;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (dst[u] != nullptr) *reinterpret_cast<uint4*>(dst[u]) = val[u];
        }
    }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
    static std::atomic<int> sms[64];  // SM count per device, queried once (0 = not yet)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int n_sms = dev >= 0 && dev < 64 ? sms[dev].load(std::memory_order_relaxed) : 0;
    if (n_sms == 0) {
        e = cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) sms[dev].store(n_sms, std::memory_order_relaxed);
    }
    if (p.n_tokens == 0 || p.hk == 0 || p.row_bytes < 16) return cudaSuccess;
    const int64_t chunks = 2LL * p.hk * (p.row_bytes / 16);  // per token
    const int64_t full_warps = static_cast<int64_t>(n_sms) * 8 * (kAppendThreads / 32);
    int wpt = 1;  // warps per token
    if (static_cast<int64_t>(p.n_tokens) * 4 < full_warps)  // few tokens: one chunk per lane
        wpt = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((chunks + 31) / 32, 64)));
    int64_t blocks = (static_cast<int64_t>(p.n_tokens) * wpt * 32 + kAppendThreads - 1) / kAppendThreads;
    if (blocks > static_cast<int64_t>(n_sms) * 8) blocks = static_cast<int64_t>(n_sms) * 8;
    append_kernel<<<static_cast<unsigned>(blocks), kAppendThreads, 0, s>>>(p, wpt);
    return cudaGetLastError();
}

}  // namespace fdec
