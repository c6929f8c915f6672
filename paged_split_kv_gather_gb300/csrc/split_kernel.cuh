// split_kernel.cuh -- the GQA split producer for paged-KV decode (SIMT, fp32).
//
// One CTA handles one work item (a run of 64-token blocks of one sequence) for
// one KV head and one group of query rows (rows = q_len x heads-per-KV-head).
// Every query row of the group reuses the same staged K/V tile.
//
//   warp NW (producer): walks the page table and moves 32-token K and V stages
//       into shared memory with 1-D TMA bulk copies, one token row per lane,
//       into rows padded by 16 bytes (conflict-free lane-per-token reads).
//       A ring of S stages with full/empty mbarriers; every wait is bounded.
//   warps 0..NW-1 (consumers): warp w takes stages w, w+NW, ... and keeps its
//       own online-softmax state (m, l, o) for the CTA's query rows:
//         q.K  : lane = token, fp32 packed FMA over head_dim, q from shared memory
//         max  : warp-shuffle max per row, running max m in log2 units
//         p.V  : lane = pair of dims, fp32 packed FMA over the stage's tokens
//   epilogue: the NW warp states are merged in shared memory by log-sum-exp and
//       written as one partial (m, l, unnormalised o) of this split, or as the
//       final out / lse when the split covers the whole sequence.
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
template <> struct SplitShape<64>  { static constexpr int NW = 8, RCMAX = 16, MINB = 2, SMAX = 8; };
template <> struct SplitShape<128> { static constexpr int NW = 8, RCMAX = 16, MINB = 1, SMAX = 16; };
template <> struct SplitShape<192> { static constexpr int NW = 4, RCMAX = 8,  MINB = 1, SMAX = 16; };
template <> struct SplitShape<256> { static constexpr int NW = 4, RCMAX = 8,  MINB = 1, SMAX = 16; };
template <> struct SplitShape<512> { static constexpr int NW = 2, RCMAX = 4,  MINB = 1, SMAX = 16; };

template <int D, int RC>
struct SplitLayout {
    static constexpr int NW = SplitShape<D>::NW;
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr int ROW_BYTES = 2 * D;
    static constexpr int PITCH = 2 * D + 16;  // +16 B: lane-per-row 16-B reads hit distinct banks
    static constexpr int STAGE_BYTES = 2 * kStageTokens * PITCH;  // K rows then V rows
    static constexpr int BAR_BYTES = 256;
    static constexpr int Q_BYTES = RC * D * 4;
    static constexpr int P_BYTES = NW * kStageTokens * RC * 4;
    static constexpr int FIXED = BAR_BYTES + Q_BYTES + P_BYTES;
    static constexpr int BUDGET = (232448 / SplitShape<D>::MINB) - 1024;
    static constexpr int S_FIT = (BUDGET - FIXED) / STAGE_BYTES;
    static constexpr int S = S_FIT > SplitShape<D>::SMAX ? SplitShape<D>::SMAX : S_FIT;
    static constexpr int SMEM = FIXED + S * STAGE_BYTES;
    static_assert(S >= NW, "each consumer warp needs its own stage in flight");
    static_assert(2 * S * 8 <= BAR_BYTES, "barrier area too small");
    static_assert(NW * RC * (D + 2) * 4 <= S * STAGE_BYTES, "merge scratch must fit the stage area");
};

template <int RC>
__device__ __forceinline__ void load_p(const float* src, float (&pr)[RC]) {
    if constexpr (RC % 4 == 0) {
#pragma unroll
        for (int j = 0; j < RC / 4; ++j) {
            const float4 x = reinterpret_cast<const float4*>(src)[j];
            pr[4 * j] = x.x;
            pr[4 * j + 1] = x.y;
            pr[4 * j + 2] = x.z;
            pr[4 * j + 3] = x.w;
        }
    } else if constexpr (RC == 2) {
        const float2 x = *reinterpret_cast<const float2*>(src);
        pr[0] = x.x;
        pr[1] = x.y;
    } else {
        pr[0] = src[0];
    }
}

template <int D, int RC, bool BF16>
__global__ void __launch_bounds__(SplitLayout<D, RC>::THREADS, SplitShape<D>::MINB)
split_kernel(const SplitParams p) {
    using Lay = SplitLayout<D, RC>;
    constexpr int NW = Lay::NW;
    constexpr int S = Lay::S;
    constexpr int PITCH = Lay::PITCH;
    constexpr int ROW_BYTES = Lay::ROW_BYTES;
    constexpr int STAGE_BYTES = Lay::STAGE_BYTES;
    constexpr int DP = D / 64;  // dim pairs per lane in p.V
    constexpr float kLn2 = 0.69314718055994530942f;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + S;
    float* q_s = reinterpret_cast<float*>(smem + Lay::BAR_BYTES);
    float* p_s = q_s + RC * D;
    uint8_t* stages = reinterpret_cast<uint8_t*>(p_s + NW * kStageTokens * RC);

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

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        fence_mbar_init();
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
        const int64_t pt_row = static_cast<int64_t>(b) * p.pt_stride;
        const int page_mask = (1 << p.page_shift) - 1;
        int page_next = -1;
        {
            const int t = tok_begin + lane;
            if (t < tok_end) page_next = p.page_table[pt_row + (t >> p.page_shift)];
        }
        int issued = 0;
        bool ok = true;
        for (int i = 0; i < n_stage; ++i) {
            const int s = i % S;
            const int page = page_next;
            {
                const int t = tok_begin + (i + 1) * kStageTokens + lane;
                if (i + 1 < n_stage && t < tok_end) page_next = p.page_table[pt_row + (t >> p.page_shift)];
            }
            if (i >= S) {
                bool got = true;
                if (lane == 0) got = mbar_wait_bounded(smem_addr(&empty[s]), ((i / S) - 1) & 1);
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
            }
            const int t = tok_begin + i * kStageTokens + lane;
            const bool in_range = t < tok_end;
            const bool valid = in_range && page >= 0 && page < p.k_pages && page < p.v_pages;
            if (in_range && !valid) atomicOr(p.err, FDEC_DEVERR_PAGE_ID);
            const unsigned mask = __ballot_sync(0xffffffffu, valid);
            const uint32_t fbar = smem_addr(&full[s]);
            if (lane == 0) mbar_arrive_expect_tx(fbar, static_cast<uint32_t>(__popc(mask)) * 2u * ROW_BYTES);
            __syncwarp();
            if (valid) {
                const int slot = t & page_mask;
                const uint8_t* ks = p.k_base + page * p.k_sp + kvh * p.k_sh + slot * p.k_st;
                const uint8_t* vs = p.v_base + page * p.v_sp + kvh * p.v_sh + slot * p.v_st;
                uint8_t* kd = stages + s * STAGE_BYTES + lane * PITCH;
                bulk_g2s(smem_addr(kd), ks, ROW_BYTES, fbar);
                bulk_g2s(smem_addr(kd + kStageTokens * PITCH), vs, ROW_BYTES, fbar);
            }
            issued = i + 1;
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
    float* pw = p_s + warp * kStageTokens * RC;
    const float4* q4 = reinterpret_cast<const float4*>(q_s);
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
        const uint8_t* Vs = Ks + kStageTokens * PITCH;

        // q.K: this lane's token against every row of the group
        float2 acc[RC];
#pragma unroll
        for (int r = 0; r < RC; ++r) acc[r] = make_float2(0.f, 0.f);
        const uint8_t* krow = Ks + lane * PITCH;
#pragma unroll 2
        for (int c = 0; c < D / 8; ++c) {
            const uint4 kr = *reinterpret_cast<const uint4*>(krow + c * 16);
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
            pw[lane * RC + r] = pr;
        }
        __syncwarp();

        // p.V: this lane's dim pairs over the stage's tokens
        for (int tt = 0; tt < nv; ++tt) {
            float pr[RC];
            load_p<RC>(pw + tt * RC, pr);
            const uint8_t* vrow = Vs + tt * PITCH;
#pragma unroll
            for (int k = 0; k < DP; ++k) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow + (k * 64 + 2 * lane) * 2);
                const float2 v2 = unpack2<BF16>(w);
#pragma unroll
                for (int r = 0; r < RC; ++r) o2[r][k] = __ffma2_rn(make_float2(pr[r], pr[r]), v2, o2[r][k]);
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
cudaError_t launch_split_one(const SplitParams& p, dim3 grid, cudaStream_t stream, bool launch) {
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
    split_kernel<D, RC, BF16><<<grid, Lay::THREADS, Lay::SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_split_rc(const SplitParams& p, int rc, dim3 grid, cudaStream_t s, bool launch) {
    constexpr int RCMAX = SplitShape<D>::RCMAX;
    switch (rc) {
        case 1: return launch_split_one<D, 1, BF16>(p, grid, s, launch);
        case 2: return launch_split_one<D, 2, BF16>(p, grid, s, launch);
        case 4: return launch_split_one<D, 4, BF16>(p, grid, s, launch);
        case 8:
            if constexpr (RCMAX >= 8) return launch_split_one<D, 8, BF16>(p, grid, s, launch);
            break;
        case 16:
            if constexpr (RCMAX >= 16) return launch_split_one<D, 16, BF16>(p, grid, s, launch);
            break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_split_d(const SplitParams& p, int rc, bool bf16, dim3 grid, cudaStream_t s, bool launch) {
    return bf16 ? launch_split_rc<D, true>(p, rc, grid, s, launch) : launch_split_rc<D, false>(p, rc, grid, s, launch);
}

}  // namespace fdec
