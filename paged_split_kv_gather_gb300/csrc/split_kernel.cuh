// split_kernel.cuh -- the GQA split producer for paged-KV decode (SIMT, fp32).
//
// One CTA handles one work item (a run of 64-token blocks of one sequence) for
// one KV head and one group of query rows (rows = q_len x heads-per-KV-head).
// Every query row of the group reuses the same staged K/V tile.
//
//   warp NW (producer): walks the page table and moves 32-token K and V stages
//       into shared memory.  Pages of >= 8 tokens go by 4-D TMA tensor copies
//       (one box of up to 32 token rows x 64 dims per page and 64-dim region,
//       128-byte swizzle); smaller pages by 16-byte cp.async into the same
//       swizzled layout.  A ring of S stages with full/empty mbarriers; every
//       wait is bounded.
//   warps 0..NW-1 (consumers): warp w takes stages w, w+NW, ... and keeps its
//       own online-softmax state (m, l, o) for the CTA's query rows:
//         q.K  : lane = token, fp32 packed FMA over head_dim, q a shared-memory
//                broadcast (the swizzle makes the lane-per-row reads conflict-free)
//         max  : warp-shuffle max per row, running max m in log2 units
//         p.V  : lane = pair of dims, fp32 packed FMA over the stage's tokens
//   epilogue: the NW warp states are merged in shared memory by log-sum-exp and
//       written as one partial (m, l, unnormalised o) of this split, or as the
//       final out / lse when the split covers the whole sequence.
//
// Stage layout (per K and per V): D/64 regions of [32 rows][128 bytes]; the
// 16-byte chunk c of row r sits at chunk position c ^ (r & 7) (TMA SWIZZLE_128B).
//
// The loop bound is the run-time sequence length (device seq_lens), while the
// grid and partial slots come from the planned capacity; idle items write an
// empty partial (m = -inf, l = 0) that the reduction skips.
#pragma once

#include <cmath>

#include "../../include/fdec.h"
#include "device_utils.cuh"
#include "fdec_internal.h"

namespace fdec {

template <int D>
struct SplitShape;
// NW consumer warps, RCMAX largest query-row group, MINB CTAs per SM to aim for,
// SMAX largest stage count.
template <> struct SplitShape<64>  { static constexpr int NW = 8, RCMAX = 16, MINB = 2, SMAX = 16; };
template <> struct SplitShape<128> { static constexpr int NW = 8, RCMAX = 16, MINB = 1, SMAX = 16; };
template <> struct SplitShape<192> { static constexpr int NW = 4, RCMAX = 8,  MINB = 1, SMAX = 16; };
template <> struct SplitShape<256> { static constexpr int NW = 4, RCMAX = 8,  MINB = 1, SMAX = 16; };
template <> struct SplitShape<512> { static constexpr int NW = 2, RCMAX = 4,  MINB = 1, SMAX = 16; };

template <int D, int RC>
struct SplitLayout {
    static constexpr int NW = SplitShape<D>::NW;
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr int REGIONS = D / 64;
    static constexpr int REGION_BYTES = kStageTokens * 128;       // 32 rows x 128 B
    static constexpr int HALF_BYTES = REGIONS * REGION_BYTES;      // K (or V) of one stage
    static constexpr int STAGE_BYTES = 2 * HALF_BYTES;             // K regions then V regions
    static constexpr int BAR_BYTES = 256;
    static constexpr int Q_BYTES = RC * D * 4;
    static constexpr int P_BYTES = NW * kStageTokens * RC * 8;     // p as (p, p) pairs
    static constexpr int ALIGN_SLACK = 1024;                       // stage area is 1024-byte aligned
    static constexpr int FIXED = BAR_BYTES + Q_BYTES + P_BYTES + ALIGN_SLACK;
    static constexpr int BUDGET = (232448 / SplitShape<D>::MINB) - 1024;
    static constexpr int S_FIT = (BUDGET - FIXED) / STAGE_BYTES;
    static constexpr int S = S_FIT > SplitShape<D>::SMAX ? SplitShape<D>::SMAX : S_FIT;
    static constexpr int SMEM = FIXED + S * STAGE_BYTES;
    static_assert(S >= NW, "each consumer warp needs its own stage in flight");
    static_assert(2 * S * 8 <= BAR_BYTES, "barrier area too small");
    static_assert(NW * RC * (D + 2) * 4 <= S * STAGE_BYTES, "merge scratch must fit the stage area");
    static_assert((BAR_BYTES + Q_BYTES + P_BYTES) % 16 == 0, "alignment");
};

template <int RC>
__device__ __forceinline__ void load_p_pairs(const float2* src, float2 (&pr)[RC]) {
    if constexpr (RC % 2 == 0) {
#pragma unroll
        for (int j = 0; j < RC / 2; ++j) {
            const float4 x = reinterpret_cast<const float4*>(src)[j];
            pr[2 * j] = make_float2(x.x, x.y);
            pr[2 * j + 1] = make_float2(x.z, x.w);
        }
    } else {
        pr[0] = src[0];
    }
}

template <int D, int RC, bool BF16>
__global__ void __launch_bounds__(SplitLayout<D, RC>::THREADS, SplitShape<D>::MINB)
split_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap tmk,
             const __grid_constant__ CUtensorMap tmv) {
    using Lay = SplitLayout<D, RC>;
    constexpr int NW = Lay::NW;
    constexpr int S = Lay::S;
    constexpr int REGIONS = Lay::REGIONS;
    constexpr int REGION_BYTES = Lay::REGION_BYTES;
    constexpr int HALF_BYTES = Lay::HALF_BYTES;
    constexpr int STAGE_BYTES = Lay::STAGE_BYTES;
    constexpr int DP = D / 64;  // dim pairs per lane in p.V
    constexpr float kLn2 = 0.69314718055994530942f;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + S;
    float* q_s = reinterpret_cast<float*>(smem + Lay::BAR_BYTES);
    float2* p_s = reinterpret_cast<float2*>(q_s + RC * D);
    uint8_t* stages;
    {
        const uint32_t raw = smem_addr(smem) + Lay::BAR_BYTES + Lay::Q_BYTES + Lay::P_BYTES;
        const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
        stages = smem + Lay::BAR_BYTES + Lay::Q_BYTES + Lay::P_BYTES + pad;
    }

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WorkItem it = p.items[blockIdx.x];
    const int b = it.seq;
    const int kvh = blockIdx.y;
    const int row0 = blockIdx.z * RC;

    int L = p.seq_lens[b];
    const int cap = p.capacity[b];
    if (L > cap || L < 0) {
        if (threadIdx.x == 0) atomicOr(p.err, FDEC_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : cap;
    }
    const int tok_begin = it.block_begin * kBlockTokens;
    const int tok_end = min(it.block_end * kBlockTokens, L);
    const int n_stage = tok_end > tok_begin ? (tok_end - tok_begin + kStageTokens - 1) / kStageTokens : 0;
    const bool tma_mode = p.page_shift >= 3;  // pages of >= 8 tokens

    if (threadIdx.x == 0) {
        const uint32_t full_count = tma_mode ? 1u : 32u;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), full_count);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        fence_mbar_init();
    }
    if (warp == NW && lane == 0 && tma_mode) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    // The group's query rows in fp32, pre-multiplied by scale*log2(e).
    for (int idx = threadIdx.x; idx < RC * D; idx += Lay::THREADS) {
        const int r = idx / D;
        const int d = idx - r * D;
        const int row = row0 + r;
        float v = 0.f;
        if (row < p.rows) {
            const int qi = row / p.group;
            const int h = kvh * p.group + (row - qi * p.group);
            v = load_16bit<BF16>(p.q + static_cast<int64_t>(b * p.q_len + qi) * p.q_stride_tok +
                                 static_cast<int64_t>(h) * p.q_stride_head + d) *
                p.scale_log2;
        }
        q_s[idx] = v;
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------------------ producer
        if (n_stage == 0) return;
        const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride;
        const int page_mask = (1 << p.page_shift) - 1;
        int issued = 0;
        bool ok = true;
        if (tma_mode) {
            // Boxes of BR token rows, NB boxes per 32-token stage; the page id of
            // box n is held by lane n % 32, one group of 32 boxes ahead.
            const int BR = min(1 << p.page_shift, kStageTokens);
            const int NB = kStageTokens / BR;
            const int n_box = (tok_end - tok_begin + BR - 1) / BR;
            const uint32_t box_bytes = static_cast<uint32_t>(BR) * 2u * (2u * D);  // K and V
            auto box_page = [&](int n) -> int {
                return n < n_box ? __ldg(pt + ((tok_begin + n * BR) >> p.page_shift)) : -1;
            };
            int pid = box_page(lane);
            int pid_next = box_page(32 + lane);
            int group = 0;
            for (int i = 0; i < n_stage; ++i) {
                const int s = i % S;
                if (i >= S) {
                    bool got = true;
                    if (lane == 0) got = mbar_wait_bounded(smem_addr(&empty[s]), ((i / S) - 1) & 1);
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        break;
                    }
                }
                const int box0 = i * NB;
                if ((box0 >> 5) != group) {  // NB divides 32: a stage never straddles two groups
                    pid = pid_next;
                    group = box0 >> 5;
                    pid_next = box_page((group + 1) * 32 + lane);
                }
                // lane j < NB checks box box0 + j
                const int my_page = __shfl_sync(0xffffffffu, pid, (box0 + lane) & 31);
                const bool in_range = lane < NB && box0 + lane < n_box;
                const bool valid = in_range && my_page >= 0 && my_page < p.k_pages && my_page < p.v_pages;
                if (in_range && !valid) atomicOr(p.err, FDEC_DEVERR_PAGE_ID);
                const unsigned vmask = __ballot_sync(0xffffffffu, valid);
                const uint32_t fbar = smem_addr(&full[s]);
                if (lane == 0) mbar_arrive_expect_tx(fbar, static_cast<uint32_t>(__popc(vmask)) * box_bytes);
                for (int j = 0; j < NB; ++j) {
                    const int page = __shfl_sync(0xffffffffu, my_page, j);
                    if (lane == 0 && ((vmask >> j) & 1u)) {
                        const int slot0 = (tok_begin + (box0 + j) * BR) & page_mask;
                        uint8_t* kdst = stages + s * STAGE_BYTES + j * BR * 128;
                        int ck[4], cv[4];
                        ck[0] = 0;
                        ck[p.k_pos_slot] = slot0;
                        ck[p.k_pos_head] = kvh;
                        ck[p.k_pos_page] = page;
                        cv[0] = 0;
                        cv[p.v_pos_slot] = slot0;
                        cv[p.v_pos_head] = kvh;
                        cv[p.v_pos_page] = page;
#pragma unroll
                        for (int r = 0; r < REGIONS; ++r) {
                            tma_load_4d(smem_addr(kdst + r * REGION_BYTES), &tmk, r * 64, ck[1], ck[2], ck[3], fbar);
                            tma_load_4d(smem_addr(kdst + HALF_BYTES + r * REGION_BYTES), &tmv, r * 64, cv[1], cv[2],
                                        cv[3], fbar);
                        }
                    }
                }
                issued = i + 1;
            }
        } else {
            // Small pages: 16-byte cp.async per (row, chunk) into the swizzled layout.
            constexpr int CHUNKS = D / 8;
            for (int i = 0; i < n_stage; ++i) {
                const int s = i % S;
                if (i >= S) {
                    bool got = true;
                    if (lane == 0) got = mbar_wait_bounded(smem_addr(&empty[s]), ((i / S) - 1) & 1);
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        break;
                    }
                }
                const int t_lane = tok_begin + i * kStageTokens + lane;
                const bool in_range = t_lane < tok_end;
                const int my_page = in_range ? __ldg(pt + (t_lane >> p.page_shift)) : -1;
                const bool valid = in_range && my_page >= 0 && my_page < p.k_pages && my_page < p.v_pages;
                if (in_range && !valid) atomicOr(p.err, FDEC_DEVERR_PAGE_ID);
                uint8_t* sbase = stages + s * STAGE_BYTES;
                for (int idx = lane; idx < kStageTokens * CHUNKS; idx += 32) {
                    const int row = idx / CHUNKS;
                    const int c = idx - row * CHUNKS;
                    const int page = __shfl_sync(0xffffffffu, my_page, row);
                    const bool ok_row = __shfl_sync(0xffffffffu, valid, row);
                    if (ok_row) {
                        const int slot = (tok_begin + i * kStageTokens + row) & page_mask;
                        const uint32_t off = (c >> 3) * REGION_BYTES + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                        cp_async_16(smem_addr(sbase + off),
                                    p.k_base + page * p.k_sp + kvh * p.k_sh + slot * p.k_st + c * 16);
                        cp_async_16(smem_addr(sbase + HALF_BYTES + off),
                                    p.v_base + page * p.v_sp + kvh * p.v_sh + slot * p.v_st + c * 16);
                    }
                }
                cp_async_arrive_noinc(smem_addr(&full[s]));
                issued = i + 1;
            }
        }
        // Do not leave while copies of this CTA may still be landing.
        for (int i = issued > S ? issued - S : 0; i < issued; ++i) {
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(smem_addr(&full[i % S]), (i / S) & 1);
            if (!__shfl_sync(0xffffffffu, got, 0)) ok = false;
        }
        if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------------------------- consumers
    float2 o2[RC][DP];
    float m[RC], l[RC];
    int lim[RC];  // last visible token of each row
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int k = 0; k < DP; ++k) o2[r][k] = make_float2(0.f, 0.f);
        const int qi = (row0 + r) / p.group;
        lim[r] = p.causal ? (L - p.q_len + qi) : (L - 1);
    }
    float2* pw = p_s + warp * kStageTokens * RC;
    const float4* q4 = reinterpret_cast<const float4*>(q_s);
    // Swizzled byte offsets: K chunk j of this lane's row; this lane's V dim pair in a row r with r & 7 == j.
    uint32_t koff[8], voff[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        koff[j] = static_cast<uint32_t>(lane * 128 + ((j ^ (lane & 7)) << 4));
        voff[j] = static_cast<uint32_t>(j * 128 + ((((lane >> 2) ^ j) & 7) << 4) + (lane & 3) * 4);
    }
    bool ok = true;

    for (int i = warp; i < n_stage; i += NW) {
        const int s = i % S;
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(smem_addr(&full[s]), (i / S) & 1);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
            ok = false;
            break;
        }
        const int t0 = tok_begin + i * kStageTokens;
        const int nv = min(kStageTokens, tok_end - t0);
        const uint8_t* Ks = stages + s * STAGE_BYTES;
        const uint8_t* Vs = Ks + HALF_BYTES;

        // q.K: this lane's token against every row of the group
        float2 acc[RC];
#pragma unroll
        for (int r = 0; r < RC; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll 8
        for (int c = 0; c < D / 8; ++c) {
            const uint4 kr = *reinterpret_cast<const uint4*>(Ks + (c >> 3) * REGION_BYTES + koff[c & 7]);
            const float2 k0 = unpack2<BF16>(kr.x);
            const float2 k1 = unpack2<BF16>(kr.y);
            const float2 k2 = unpack2<BF16>(kr.z);
            const float2 k3 = unpack2<BF16>(kr.w);
#pragma unroll
            for (int r = 0; r < RC; ++r) {
                const float4 qa = q4[r * (D / 4) + 2 * c];
                const float4 qb = q4[r * (D / 4) + 2 * c + 1];
                acc[r] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[r]);
                acc[r] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc[r]);
                acc[r] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[r]);
                acc[r] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc[r]);
            }
        }

        // online softmax over this stage's tokens (log2 units)
        const int t = t0 + lane;
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            float z = acc[r].x + acc[r].y;
            if (lane >= nv || t > lim[r]) z = -INFINITY;
            const float mx = warp_max(z);
            const float m_new = fmaxf(m[r], mx);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = exp2_approx(m[r] - m_use);
            const float pr = exp2_approx(z - m_use);
            l[r] = l[r] * alpha + pr;
            m[r] = m_new;
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int k = 0; k < DP; ++k) o2[r][k] = __fmul2_rn(o2[r][k], a2);
            pw[lane * RC + r] = make_float2(pr, pr);
        }
        __syncwarp();

        // p.V: this lane's dim pairs over the stage's tokens
        for (int tt0 = 0; tt0 < nv; tt0 += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int tt = tt0 + j;
                if (tt < nv) {
                    float2 pr[RC];
                    load_p_pairs<RC>(pw + tt * RC, pr);
                    const uint8_t* vrow = Vs + tt0 * 128 + voff[j];
#pragma unroll
                    for (int k = 0; k < DP; ++k) {
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow + k * REGION_BYTES);
                        const float2 v2 = unpack2<BF16>(w);
#pragma unroll
                        for (int r = 0; r < RC; ++r) o2[r][k] = __ffma2_rn(pr[r], v2, o2[r][k]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
#pragma unroll
    for (int r = 0; r < RC; ++r) l[r] = warp_sum(l[r]);
    if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);

    // ---------------------------------------------------------------------- epilogue
    named_barrier(1, NW * 32);  // every consumer is done with the stage buffers
    float* sm_m = reinterpret_cast<float*>(stages);  // [NW][RC]
    float* sm_l = sm_m + NW * RC;                     // [NW][RC]
    float* sm_o = sm_l + NW * RC;                     // [NW][RC][D]
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            sm_m[warp * RC + r] = m[r];
            sm_l[warp * RC + r] = l[r];
        }
    }
#pragma unroll
    for (int r = 0; r < RC; ++r)
#pragma unroll
        for (int k = 0; k < DP; ++k)
            *reinterpret_cast<float2*>(sm_o + (warp * RC + r) * D + k * 64 + 2 * lane) = o2[r][k];
    named_barrier(1, NW * 32);

    for (int idx = threadIdx.x; idx < RC * D; idx += NW * 32) {
        const int r = idx / D;
        const int d = idx - r * D;
        const int row = row0 + r;
        if (row >= p.rows) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * RC + r]);
        float Ls = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float e = exp2_approx(sm_m[w * RC + r] - M);
                Ls += sm_l[w * RC + r] * e;
                O += sm_o[(w * RC + r) * D + d] * e;
            }
        }
        if (it.slot < 0) {
            const int qi = row / p.group;
            const int h = kvh * p.group + (row - qi * p.group);
            const int64_t orow = static_cast<int64_t>(b * p.q_len + qi) * p.hq + h;
            p.out[orow * D + d] = Ls > 0.f ? O / Ls : 0.f;
            if (d == 0 && p.lse != nullptr) p.lse[orow] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
        } else {
            const int64_t prow = (static_cast<int64_t>(it.slot) * p.hk + kvh) * p.rows + row;
            p.part_o[prow * D + d] = O;
            if (d == 0) p.part_ml[prow] = make_float2(M, Ls);
        }
    }
}

template <int D, int RC, bool BF16>
cudaError_t launch_split_one(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                             cudaStream_t stream, bool launch) {
    using Lay = SplitLayout<D, RC>;
    static unsigned long long attr_done = 0;  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(split_kernel<D, RC, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Lay::SMEM);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&attr_done, 1ull << dev, __ATOMIC_RELEASE);
    }
    if (!launch) return cudaSuccess;
    split_kernel<D, RC, BF16><<<grid, Lay::THREADS, Lay::SMEM, stream>>>(p, tk, tv);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_split_rc(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc, dim3 grid,
                            cudaStream_t s, bool launch) {
    constexpr int RCMAX = SplitShape<D>::RCMAX;
    switch (rc) {
        case 1: return launch_split_one<D, 1, BF16>(p, tk, tv, grid, s, launch);
        case 2: return launch_split_one<D, 2, BF16>(p, tk, tv, grid, s, launch);
        case 4: return launch_split_one<D, 4, BF16>(p, tk, tv, grid, s, launch);
        case 8:
            if constexpr (RCMAX >= 8) return launch_split_one<D, 8, BF16>(p, tk, tv, grid, s, launch);
            break;
        case 16:
            if constexpr (RCMAX >= 16) return launch_split_one<D, 16, BF16>(p, tk, tv, grid, s, launch);
            break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_split_d(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc, bool bf16,
                           dim3 grid, cudaStream_t s, bool launch) {
    return bf16 ? launch_split_rc<D, true>(p, tk, tv, rc, grid, s, launch)
                : launch_split_rc<D, false>(p, tk, tv, rc, grid, s, launch);
}

}  // namespace fdec
