// split_mma_kernel.cuh -- the GQA split producer on warp-level tensor cores.
//
// Same work decomposition, producer warp, stage ring and epilogue as the SIMT
// split kernel; the consumer warps do the two contractions with
// mma.sync.m16n8k16 (16-bit inputs, fp32 accumulation) instead of fp32 FMAs:
//
//   S = Q K^T   M = 16 query rows (the KV group's heads x q positions, zero-padded),
//               N = 32 tokens of the stage, K = head_dim.  Q's A fragments stay in
//               registers for the whole item; K's B fragments come from the
//               swizzled stage by ldmatrix (conflict-free).  Products of 16-bit
//               inputs are exact in fp32, so this is the fp32 dot product up to
//               summation order.
//   softmax     on the S accumulator fragments: scale, mask, quad-shuffle row max,
//               lazy rescale (the running max moves only when a score beats it by
//               more than 8 in log2 units), exp2.
//   O += P V    M = 16 rows, N = head_dim, K = 32 tokens.  The accumulator
//               fragments of S are the A fragments of P.  P is split into a
//               16-bit high part and a 16-bit residual (P = P_hi + P_lo, both
//               multiplied), so p keeps ~16 significant bits; V's B fragments come
//               from the stage by ldmatrix.trans.
//
// Why tensor cores here although decode is bandwidth-bound: with fp32 FMAs every
// query value (q.K) and every probability (p.V) must be broadcast to all lanes
// through shared memory, and a 16-byte broadcast costs four shared-memory
// wavefronts: ~1800 wavefronts per 32-token stage against ~760 cycles of HBM
// time per stage and SM at 6.8 TB/s for a group of 8 query heads.  The fragment
// layouts of m16n8k16 keep Q and P in registers, leaving ~260 wavefronts per stage
// (the K and V reads and the TMA writes).
#pragma once

#include "split_common.cuh"

namespace fdec {

template <int D>
struct MmaLayout {
    using G = StageGeom<D>;
    static constexpr int RC = 16;                 // query rows per M tile
    static constexpr int BAR_BYTES = 512;
    static constexpr int Q_BYTES = RC * D * 2;    // 16-bit q rows
    static constexpr int ALIGN_SLACK = 1024;
    // Two CTAs per SM (measured: 103 us against 131 us with one CTA of 7
    // consumers for 537 MB at 262144 tokens): each CTA gets half the shared
    // memory and four warps (3 consumers + the producer), 255 registers each.
    // head_dim 256 fits three stages and two consumers per CTA; head_dim 512
    // runs one CTA per SM (stages of 64 KB).
    static constexpr int CTAS_PER_SM = D <= 256 ? 2 : 1;
    // head_dim 512: the O accumulators of all 512 columns would need 256
    // registers, so two consumer warps share each stage, both computing S and
    // each accumulating P V for one half of the columns (DH).
    static constexpr int DSPLIT = D > 256 ? 2 : 1;
    static constexpr int DH = D / DSPLIT;
    // Q's A fragments stay in registers up to head_dim 192; at 256 the O
    // accumulators take 128 registers and the fragments are re-read from shared
    // memory (ldmatrix) at every k-step instead.
    static constexpr bool Q_IN_REGS = D <= 192;
    static constexpr int BUDGET = 232448 / CTAS_PER_SM - 1024;
    static constexpr int FIXED = BAR_BYTES + Q_BYTES + ALIGN_SLACK;
    static constexpr int S_FIT = (BUDGET - FIXED) / G::STAGE_BYTES;
    static constexpr int S = S_FIT > 16 ? 16 : S_FIT;
    static constexpr int NP = (S - 1) < 3 ? (S - 1) : 3;  // consumer groups (stages in flight at once)
    static constexpr int NW = NP * DSPLIT;                 // consumer warps
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr int SMEM = FIXED + S * G::STAGE_BYTES;
    static_assert(S >= NP + 1, "stage ring too small");
    static_assert(3 * S * 8 <= BAR_BYTES, "barrier area too small");
    static_assert(NP * RC * (D + 2) * 4 <= S * G::STAGE_BYTES, "merge scratch must fit the stage area");
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D (16x8, fp32) += A (16x16, row) * B (16x8, col), 16-bit inputs.
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Round (x, y) to a packed 16-bit pair (x in the low half), and the residual pair.
template <bool BF16>
__device__ __forceinline__ void split_pair(float x, float y, uint32_t& hi, uint32_t& lo) {
    if constexpr (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&l);
    } else {
        const __half2 h = __floats2half2_rn(x, y);
        const __half2 l = __floats2half2_rn(x - __low2float(h), y - __high2float(h));
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&l);
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(MmaLayout<D>::THREADS, MmaLayout<D>::CTAS_PER_SM)
split_mma_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
    using Lay = MmaLayout<D>;
    using G = StageGeom<D>;
    constexpr int NW = Lay::NW;
    constexpr int S = Lay::S;
    constexpr int RC = Lay::RC;
    constexpr int NP = Lay::NP;          // consumer groups, one stage each
    constexpr int DSPLIT = Lay::DSPLIT;  // warps per group (each owns DH columns of O)
    constexpr int DH = Lay::DH;
    constexpr int KSTEPS = D / 16;       // k-steps of S = Q K^T
    constexpr int NT = DH / 8;           // n-tiles of this warp's O

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + 2 * S;
    uint16_t* q_s = reinterpret_cast<uint16_t*>(smem + Lay::BAR_BYTES);
    uint8_t* stages;
    {
        const uint32_t raw = smem_addr(smem) + Lay::BAR_BYTES + Lay::Q_BYTES;
        const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
        stages = smem + Lay::BAR_BYTES + Lay::Q_BYTES + pad;
    }

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WorkItem it = p.items[blockIdx.x];
    const int b = it.seq;
    const int kvh = blockIdx.y;
    const int row0 = blockIdx.z * RC;
    const bool tma_mode = p.page_shift >= 3;
    if (threadIdx.x == 0) init_stage_barriers<S>(full, empty, tma_mode, DSPLIT);
    __syncthreads();  // barriers initialised (nothing before this waits on memory)
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
    // The group's query rows, as stored (16-bit, [RC][D]); rows past the group are zero.
    {
        QChunks<RC, D, NW * 32> qc;
        qc.load(p, b, kvh, row0, threadIdx.x);
#pragma unroll
        for (int i = 0; i < qc.PER; ++i) {
            const int idx = qc.chunk(threadIdx.x, i);
            if (idx < qc.CH) *reinterpret_cast<uint4*>(q_s + idx * 8) = qc.v[i];
        }
    }
    named_barrier(1, NW * 32);

    // ---------------------------------------------------------------------- consumers
    const int g = lane >> 2;   // fragment row (and row + 8)
    const int tq = lane & 3;   // fragment column pair
    const int mi = lane >> 3;  // ldmatrix: which 8x8 matrix this lane addresses

    constexpr int QREGS = Lay::Q_IN_REGS ? KSTEPS : 1;
    uint32_t qa[QREGS][4];
    const uint32_t q_lane = smem_addr(q_s) + ((mi & 1) * 8 + (lane & 7)) * (D * 2) + (mi >> 1) * 16;
    if constexpr (Lay::Q_IN_REGS) {
        static_for<0, KSTEPS>([&](auto kk_) {
            constexpr int kk = decltype(kk_)::value;
            ldmatrix_x4(q_lane + 2 * kk * 16, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
        });
    }
    // ldmatrix row addresses within a stage (swizzled: chunk c of row r at c ^ (r & 7)).
    uint32_t kb_row[2], kb_x[4], vb_row[2], vb_x[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        kb_row[j] = static_cast<uint32_t>((8 * (2 * j + (mi >> 1)) + (lane & 7)) * 128);
        vb_row[j] = static_cast<uint32_t>((16 * j + 8 * (mi & 1) + (lane & 7)) * 128);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        kb_x[j] = static_cast<uint32_t>(((2 * j + (mi & 1)) ^ (lane & 7)) << 4);
        vb_x[j] = static_cast<uint32_t>(((2 * j + (mi >> 1)) ^ (lane & 7)) << 4);
    }

    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};
    int lim[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int qi = (row0 + g + 8 * h) / p.group;
        lim[h] = p.causal ? (ir.L - p.q_len + qi) : (ir.L - 1);
    }
    const uint32_t stages_base = smem_addr(stages);
    bool ok = true;

    const int grp = warp / DSPLIT;             // consumer group: stages grp, grp + NP, ...
    const int half = warp - grp * DSPLIT;      // which DH columns of O this warp accumulates
    const uint32_t v_half = static_cast<uint32_t>(half * (DH / 64) * G::REGION_BYTES);
    for (int i = grp; i < ir.n_stage; i += NP) {
        const int s = i % S;
        if (!wait_stage<S>(full, i)) {
            ok = false;
            break;
        }
        const int t0 = ir.tok_begin + i * kStageTokens;
        const int nv = min(kStageTokens, ir.tok_end - t0);
        const uint32_t kbase = stages_base + s * G::STAGE_BYTES;
        const uint32_t vbase = kbase + G::HALF_BYTES;
        if (nv < kStageTokens) zero_v_tail<D>(stages + s * G::STAGE_BYTES, nv);

        // S = Q K^T for the stage's 32 tokens (4 n-tiles of 8)
        float sc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        static_for<0, KSTEPS>([&](auto kk_) {
            constexpr int kk = decltype(kk_)::value;
            constexpr int qk = Lay::Q_IN_REGS ? kk : 0;
            if constexpr (!Lay::Q_IN_REGS) ldmatrix_x4(q_lane + 2 * kk * 16, qa[0][0], qa[0][1], qa[0][2], qa[0][3]);
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4(kbase + (kk >> 2) * G::REGION_BYTES + kb_row[pr] + kb_x[kk & 3], b0, b1, b2, b3);
                mma_16816<BF16>(sc[2 * pr], qa[qk], b0, b1);
                mma_16816<BF16>(sc[2 * pr + 1], qa[qk], b2, b3);
            }
        });

        // softmax in log2 units on the fragments: element e of n-tile n is
        // row g + 8 * (e >> 1), token 8 n + 2 tq + (e & 1)
        const int vis0 = min(nv, lim[0] - t0 + 1);
        const int vis1 = min(nv, lim[1] - t0 + 1);
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = 8 * n + 2 * tq + (e & 1);
                float z = sc[n][e] * p.scale_log2;
                if (tok >= ((e >> 1) ? vis1 : vis0)) z = -INFINITY;
                sc[n][e] = z;
                if (e >> 1)
                    mx1 = fmaxf(mx1, z);
                else
                    mx0 = fmaxf(mx0, z);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        constexpr float kLazyRescale = 8.f;
        if (__any_sync(0xffffffffu, mx0 > mrow[0] + kLazyRescale || mx1 > mrow[1] + kLazyRescale)) {
            const float n0 = fmaxf(mrow[0], mx0), n1 = fmaxf(mrow[1], mx1);
            const float a0 = exp2_approx(mrow[0] - n0), a1 = exp2_approx(mrow[1] - n1);  // 0 when m was -inf
            lrow[0] *= a0;
            lrow[1] *= a1;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
            mrow[0] = n0;
            mrow[1] = n1;
        }
        const float mu0 = mrow[0] == -INFINITY ? 0.f : mrow[0];
        const float mu1 = mrow[1] == -INFINITY ? 0.f : mrow[1];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            sc[n][0] = exp2_approx(sc[n][0] - mu0);
            sc[n][1] = exp2_approx(sc[n][1] - mu0);
            sc[n][2] = exp2_approx(sc[n][2] - mu1);
            sc[n][3] = exp2_approx(sc[n][3] - mu1);
            lrow[0] += sc[n][0] + sc[n][1];
            lrow[1] += sc[n][2] + sc[n][3];
        }
        // P as A fragments of two k-steps of 16 tokens, split into high and residual parts
        uint32_t ph[2][4], pl[2][4];
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            split_pair<BF16>(sc[2 * k2][0], sc[2 * k2][1], ph[k2][0], pl[k2][0]);
            split_pair<BF16>(sc[2 * k2][2], sc[2 * k2][3], ph[k2][1], pl[k2][1]);
            split_pair<BF16>(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1], ph[k2][2], pl[k2][2]);
            split_pair<BF16>(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3], ph[k2][3], pl[k2][3]);
        }
        // O += P V
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            static_for<0, DH / 16>([&](auto jp_) {
                constexpr int jp = decltype(jp_)::value;  // 16-column group of this warp's half
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(vbase + v_half + (jp >> 2) * G::REGION_BYTES + vb_row[k2] + vb_x[jp & 3], b0, b1, b2,
                                  b3);
                mma_16816<BF16>(o[2 * jp], ph[k2], b0, b1);
                mma_16816<BF16>(o[2 * jp], pl[k2], b0, b1);
                mma_16816<BF16>(o[2 * jp + 1], ph[k2], b2, b3);
                mma_16816<BF16>(o[2 * jp + 1], pl[k2], b2, b3);
            });
        }
        if (nv < kStageTokens) fence_proxy_async_shared();  // generic zeroing before the slot's next TMA write
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
        lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
    }
    if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);

    // ---------------------------------------------------------------------- epilogue
    named_barrier(1, NW * 32);  // every consumer is done with the stage buffers
    // The reduction (launched as a programmatic dependent) may start its launch now.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float* sm_m = reinterpret_cast<float*>(stages);  // [NP][RC]
    float* sm_l = sm_m + NP * RC;                     // [NP][RC]
    float* sm_o = sm_l + NP * RC;                     // [NP][RC][D]
    if (tq == 0 && half == 0) {  // the warps of a group hold the same m and l
        sm_m[grp * RC + g] = mrow[0];
        sm_m[grp * RC + g + 8] = mrow[1];
        sm_l[grp * RC + g] = lrow[0];
        sm_l[grp * RC + g + 8] = lrow[1];
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        *reinterpret_cast<float2*>(sm_o + (grp * RC + g) * D + half * DH + 8 * n + 2 * tq) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(sm_o + (grp * RC + g + 8) * D + half * DH + 8 * n + 2 * tq) =
            make_float2(o[n][2], o[n][3]);
    }
    named_barrier(1, NW * 32);
    merge_and_store<NP, RC, D, NW * 32>(p, it, kvh, row0, sm_m, sm_l, sm_o);
}

template <int D, bool BF16>
cudaError_t launch_split_mma_one(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                                 cudaStream_t stream, bool launch) {
    using Lay = MmaLayout<D>;
    static unsigned long long attr_done = 0;  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(split_mma_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&attr_done, 1ull << dev, __ATOMIC_RELEASE);
    }
    if (!launch) return cudaSuccess;
    split_mma_kernel<D, BF16><<<grid, Lay::THREADS, Lay::SMEM, stream>>>(p, tk, tv);
    return cudaGetLastError();
}

}  // namespace fdec
