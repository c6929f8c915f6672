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

#include "split_common.cuh"

namespace fdec {

template <int D>
struct SplitShape {
    // Register file allocation rounds a CTA up to whole groups of four warps, so
    // 12 warps (11 consumers + the producer) cost no more registers per thread
    // than 9 do.  RCMAX bounds the per-lane accumulators (RC x D/32 floats).
    static constexpr int NWMAX = D <= 128 ? 11 : (D <= 256 ? 7 : 3);
    static constexpr int RCMAX = D <= 128 ? 16 : (D <= 256 ? 8 : 4);
};

template <int D, int RC>
struct SplitLayout {
    static constexpr int REGIONS = StageGeom<D>::REGIONS;
    static constexpr int REGION_BYTES = StageGeom<D>::REGION_BYTES;
    static constexpr int HALF_BYTES = StageGeom<D>::HALF_BYTES;
    static constexpr int STAGE_BYTES = StageGeom<D>::STAGE_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int Q_BYTES = RC * D * 4;
    static constexpr int ALIGN_SLACK = 1024;                       // stage area is 1024-byte aligned
    static constexpr int BUDGET = 232448 - 1024;
    static constexpr int SMAX = 16;
    static constexpr int p_bytes(int nw) { return nw * kStageTokens * RC * 8; }  // p as (p, p) pairs
    static constexpr int fixed(int nw) { return BAR_BYTES + Q_BYTES + p_bytes(nw) + ALIGN_SLACK; }
    static constexpr int stages(int nw) {
        return (BUDGET - fixed(nw)) / STAGE_BYTES > SMAX ? SMAX : (BUDGET - fixed(nw)) / STAGE_BYTES;
    }
    // The most consumer warps that still leave a stage in flight beyond one per consumer.
    static constexpr int pick_nw() {
        for (int nw = SplitShape<D>::NWMAX; nw > 1; --nw)
            if (stages(nw) >= nw + 1) return nw;
        return 1;
    }
    static constexpr int NW = pick_nw();
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr int P_BYTES = p_bytes(NW);
    static constexpr int S = stages(NW);
    static constexpr int SMEM = fixed(NW) + S * STAGE_BYTES;
    static_assert(S >= NW, "each consumer warp needs its own stage in flight");
    static_assert(3 * S * 8 <= BAR_BYTES, "barrier area too small");
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
__global__ void __launch_bounds__(SplitLayout<D, RC>::THREADS, 1)
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

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // 2S: stage i uses full[i % 2S]
    uint64_t* empty = full + 2 * S;                       // S: stage i releases empty[i % S]
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

    const bool tma_mode = p.page_shift >= 3;  // pages of >= 8 tokens
    if (threadIdx.x == 0) init_stage_barriers<S>(full, empty, tma_mode);
    __syncthreads();  // barriers initialised (nothing before this waits on memory)
    // Launched as a programmatic dependent of the kernel before it in the stream: read
    // and write nothing but plan data before that kernel has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const ItemRange ir = item_range(p, it);

    if (warp == NW) {
        // The producer starts at once: its page-table reads overlap the length and q loads.
        if (lane == 0 && tma_mode) {
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
        }
        produce_stages<D, S>(p, &tmk, &tmv, full, empty, stages, b, kvh, ir, tma_mode);
        return;
    }
    if (threadIdx.x == 0) report_item_range(p, ir);
    const int L = ir.L, tok_begin = ir.tok_begin, tok_end = ir.tok_end, n_stage = ir.n_stage;
    // The group's query rows in fp32 ([RC][D]), pre-multiplied by scale*log2(e).
    {
        QChunks<RC, D, NW * 32> qc;
        qc.load(p, b, kvh, row0, threadIdx.x);
#pragma unroll
        for (int i = 0; i < qc.PER; ++i) {
            const int idx = qc.chunk(threadIdx.x, i);
            if (idx < qc.CH) {
                const uint32_t w[4] = {qc.v[i].x, qc.v[i].y, qc.v[i].z, qc.v[i].w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 pr = unpack2<BF16>(w[e]);
                    f[2 * e] = pr.x * p.scale_log2;
                    f[2 * e + 1] = pr.y * p.scale_log2;
                }
                *reinterpret_cast<float4*>(q_s + idx * 8) = make_float4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<float4*>(q_s + idx * 8 + 4) = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }
    named_barrier(1, NW * 32);

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
    const uint32_t q_base = smem_addr(q_s);
    const uint32_t pw_base = smem_addr(p_s + warp * kStageTokens * RC);
    const uint32_t stages_base = smem_addr(stages);
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
        if (!wait_stage<S>(full, i)) {
            ok = false;
            break;
        }
        const int t0 = tok_begin + i * kStageTokens;
        const int nv = min(kStageTokens, tok_end - t0);
        const uint32_t kbase = stages_base + s * STAGE_BYTES;
        const uint32_t vbase = kbase + HALF_BYTES;
        if (nv < kStageTokens) zero_v_tail<D>(stages + s * STAGE_BYTES, nv);

        // q.K: this lane's token against every row of the group (two partial
        // sums per row when registers allow, for independent FMA chains)
        float2 acc[RC], acc2[RC];
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            acc[r] = make_float2(0.f, 0.f);
            acc2[r] = make_float2(0.f, 0.f);
        }
        uint32_t ka[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) ka[j] = kbase + koff[j];
        // One 64-dim region (8 chunks of 8 dims) per iteration keeps the code small.
#pragma unroll 1
        for (int reg = 0; reg < REGIONS; ++reg) {
            const uint32_t qreg = q_base + reg * 256;
            static_for<0, 8>([&](auto cc) {
                constexpr int c = decltype(cc)::value;
                const uint4 kr = lds128<0>(ka[c] + reg * REGION_BYTES);
                const float2 k0 = unpack2<BF16>(kr.x);
                const float2 k1 = unpack2<BF16>(kr.y);
                const float2 k2 = unpack2<BF16>(kr.z);
                const float2 k3 = unpack2<BF16>(kr.w);
                static_for<0, RC>([&](auto rr) {
                    constexpr int r = decltype(rr)::value;
                    const float4 qa = lds128f<(r * D + 8 * c) * 4>(qreg);
                    const float4 qb = lds128f<(r * D + 8 * c + 4) * 4>(qreg);
                    if constexpr (RC <= 8) {
                        acc[r] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[r]);
                        acc2[r] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc2[r]);
                        acc[r] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[r]);
                        acc2[r] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc2[r]);
                    } else {  // many rows already give independent chains; save the registers
                        acc[r] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc[r]);
                        acc[r] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc[r]);
                        acc[r] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc[r]);
                        acc[r] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc[r]);
                    }
                });
            });
        }

        // Online softmax over this stage's tokens, in log2 units.  The running
        // max is raised (with the rescale of l and o) only when some token beats
        // it by more than kLazyRescale; otherwise p = exp2(z - m) <= 2^kLazyRescale.
        constexpr float kLazyRescale = 8.f;
#pragma unroll
        for (int r = 0; r < RC; ++r) {
            const int vis = min(nv, lim[r] - t0 + 1);  // tokens of this stage row r may see
            float z = (acc[r].x + acc[r].y) + (acc2[r].x + acc2[r].y);
            if (lane >= vis) z = -INFINITY;
            if (__any_sync(0xffffffffu, z > m[r] + kLazyRescale)) {
                const float m_new = fmaxf(m[r], warp_max(z));
                const float alpha = exp2_approx(m[r] - m_new);  // 0 when m was -inf
                l[r] *= alpha;
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int k = 0; k < DP; ++k) o2[r][k] = __fmul2_rn(o2[r][k], a2);
                m[r] = m_new;
            }
            const float pr = exp2_approx(z - (m[r] == -INFINITY ? 0.f : m[r]));
            l[r] += pr;
            *reinterpret_cast<float2*>(p_s + warp * kStageTokens * RC + lane * RC + r) = make_float2(pr, pr);
        }
        __syncwarp();

        // p.V: this lane's dim pairs over the stage's tokens, eight at a time
        const int groups = (nv + 7) >> 3;
        for (int g = 0; g < groups; ++g) {
            const uint32_t vg = vbase + g * 8 * 128;
            const uint32_t pg = pw_base + g * 8 * RC * 8;
            static_for<0, 8>([&](auto jj) {
                constexpr int j = decltype(jj)::value;
                float2 pr[RC];
                static_for<0, (RC + 1) / 2>([&](auto hh) {
                    constexpr int h = decltype(hh)::value;
                    if constexpr (2 * h + 1 < RC) {
                        const float4 x = lds128f<(j * RC + 2 * h) * 8>(pg);
                        pr[2 * h] = make_float2(x.x, x.y);
                        pr[2 * h + 1] = make_float2(x.z, x.w);
                    } else {
                        pr[2 * h] = lds64f<(j * RC + 2 * h) * 8>(pg);
                    }
                });
                const uint32_t vrow = vg + voff[j];
                static_for<0, DP>([&](auto kk) {
                    constexpr int k = decltype(kk)::value;
                    const float2 v2 = unpack2<BF16>(lds32<k * REGION_BYTES>(vrow));
#pragma unroll
                    for (int r = 0; r < RC; ++r) o2[r][k] = __ffma2_rn(pr[r], v2, o2[r][k]);
                });
            });
        }
        if (nv < kStageTokens) fence_proxy_async_shared();  // generic zeroing before the slot's next TMA write
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
#pragma unroll
    for (int r = 0; r < RC; ++r) l[r] = warp_sum(l[r]);
    if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);

    // ---------------------------------------------------------------------- epilogue
    named_barrier(1, NW * 32);  // every consumer is done with the stage buffers
    // The reduction (launched as a programmatic dependent) may start its launch now.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

    merge_and_store<NW, RC, D>(p, it, kvh, row0, sm_m, sm_l, sm_o);
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Lay::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Lay::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait in the kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kernel<D, RC, BF16>, p, tk, tv);
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
