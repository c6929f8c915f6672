// split_common.cuh -- pieces shared by the split kernels: the stage geometry,
// the producer warp (page-table walk + TMA gather into swizzled stages), the
// zeroing of a partial stage's tail, and the epilogue that merges the consumer
// warps' (m, l, o) states and writes a partial or the final out / lse.
//
// Stage layout (per K and per V): D x (element bytes) / 128 regions of
// [32 rows][128 bytes] (D/64 for 16-bit storage, D/128 for E4M3 codes); the
// 16-byte chunk c of row r sits at chunk position c ^ (r & 7) (TMA SWIZZLE_128B).
// Stage i completes barrier full[i % 2S] (phase i / 2S) and is released on
// empty[i % S]; see the consumer loops for why 2S full barriers are needed.
#pragma once

#include <cmath>
#include <type_traits>

#include "../../include/fdec.h"
#include "device_utils.cuh"
#include "fdec_internal.h"

namespace fdec {

template <int I, int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for<I + 1, N>(f);
    }
}

template <int D, int TOK = kStageTokens, int EB = 2>
struct StageGeom {
    static constexpr int TOKENS = TOK;                         // token rows per stage
    static constexpr int ROW_BYTES = D * EB;                   // one token's K (or V) row
    static constexpr int REGIONS = ROW_BYTES / 128;
    static constexpr int REGION_BYTES = TOK * 128;             // TOK rows x 128 B
    static constexpr int HALF_BYTES = REGIONS * REGION_BYTES;  // K (or V) of one stage
    static constexpr int STAGE_BYTES = 2 * HALF_BYTES;         // K regions then V regions
};

// Byte offset of token row t of a stage's K (or V) half whose rows were staged in
// boxes of br rows (br divides the stage's rows; br = the stage's rows: the
// region-major layout [region][row][128 B]).  Box n = t / br holds rows n br .. + br - 1
// as [region][br rows][128 B], so region r of row t is at this offset + r br 128.  With
// br a multiple of 8, the 128-byte swizzle of row t still XORs by t & 7.
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t stage_row_offset(int t, int br) {
    return static_cast<uint32_t>((t / br) * (br * ROW_BYTES) + (t % br) * 128);
}

// Token rows per staged box of a 32-token stage as the producers stage it: pages of 8
// or 16 tokens in box-major kernels (TMA mode), the whole stage otherwise.
__device__ __forceinline__ int staged_box_rows(int page_shift, bool box_major) {
    return (box_major && page_shift >= 3 && page_shift < 5) ? (1 << page_shift) : kStageTokens;
}

// Token range of a work item, with the run-time length clamped to the planned
// capacity.  tok_end_alloc is the item's range by plan (its blocks), known
// before the run-time length arrives; bad records a length outside [0, capacity]
// for report_item_range.  No branch depends on the loaded length here, so the
// producer's page-table loads can be issued while it is in flight.
struct ItemRange {
    int L, tok_begin, tok_end, n_stage, tok_end_alloc;
    bool bad;
};

template <int TOK = kStageTokens>
__device__ __forceinline__ ItemRange item_range(const SplitParams& p, const WorkItem& it) {
    const int L0 = p.seq_lens[it.seq];
    const int cap = p.capacity[it.seq];
    ItemRange r;
    r.bad = L0 > cap || L0 < 0;
    r.L = L0 < 0 ? 0 : (L0 > cap ? cap : L0);
    r.tok_begin = it.block_begin * kBlockTokens;
    r.tok_end_alloc = it.block_end * kBlockTokens;
    r.tok_end = min(r.tok_end_alloc, r.L);
    r.n_stage = r.tok_end > r.tok_begin ? (r.tok_end - r.tok_begin + TOK - 1) / TOK : 0;
    return r;
}

// One thread of the CTA flags a length outside [0, capacity] (it was clamped).
__device__ __forceinline__ void report_item_range(const SplitParams& p, const ItemRange& ir) {
    if (ir.bad) atomicOr(p.err, FDEC_DEVERR_SEQ_LEN);
}

// Fetch the CTA's query rows: 16-byte chunk k of the (RC rows x D) block of 16-bit
// values, by threads tid = 0 .. NTHREADS-1, chunk k at tid + i NTHREADS.  All
// loads are issued before any of them is used (a loop that stores each value
// before loading the next waits one memory round trip per iteration); rows past
// p.rows are zero.  16-byte loads when q and its strides allow, else 2-byte loads.
template <int RC, int D, int NTHREADS>
struct QChunks {
    static constexpr int CH = RC * D / 8;
    static constexpr int PER = (CH + NTHREADS - 1) / NTHREADS;
    uint4 v[PER];

    __device__ __forceinline__ void load(const SplitParams& p, int b, int kvh, int row0, int tid) {
        const bool vec = ((reinterpret_cast<uintptr_t>(p.q) | static_cast<uintptr_t>(p.q_stride_tok * 2) |
                           static_cast<uintptr_t>(p.q_stride_head * 2)) & 15u) == 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int idx = tid + i * NTHREADS;
            v[i] = make_uint4(0u, 0u, 0u, 0u);
            const int r = idx / (D / 8);
            const int row = row0 + r;
            if (idx < CH && row < p.rows) {
                const int qi = row / p.group;
                const int h = kvh * p.group + (row - qi * p.group);
                const uint16_t* src = p.q + static_cast<int64_t>(b * p.q_len + qi) * p.q_stride_tok +
                                      static_cast<int64_t>(h) * p.q_stride_head + (idx - r * (D / 8)) * 8;
                if (vec) {
                    v[i] = __ldg(reinterpret_cast<const uint4*>(src));
                } else {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = static_cast<uint32_t>(__ldg(src + 2 * e)) |
                               (static_cast<uint32_t>(__ldg(src + 2 * e + 1)) << 16);
                    v[i] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
    // chunk index of v[i] (valid when < CH)
    __device__ __forceinline__ static int chunk(int tid, int i) { return tid + i * NTHREADS; }
};

// Initialise the 2S full and S empty barriers (thread 0).  Pages of >= 8 tokens
// complete a stage with one expect-tx arrival (TMA; tma_full_count 33 when the 32
// producer lanes also arrive after copying q8_0 scale rows); smaller pages with the
// 32 cp.async arrivals of the producer lanes.
template <int S>
__device__ __forceinline__ void init_stage_barriers(uint64_t* full, uint64_t* empty, bool tma_mode,
                                                    uint32_t empty_count = 1, uint32_t tma_full_count = 1) {
    const uint32_t full_count = tma_mode ? tma_full_count : 32u;
#pragma unroll
    for (int s = 0; s < S; ++s) {
        mbar_init(smem_addr(&full[s]), full_count);
        mbar_init(smem_addr(&full[S + s]), full_count);
        mbar_init(smem_addr(&empty[s]), empty_count);
    }
    fence_mbar_init();
}

// Copy the block-scale rows (SCB bytes each, K then V) of token `tok` (page, slot) into
// row `row` of a stage's scale area [K: TOK rows][V: TOK rows].
template <int TOK, int SCB>
__device__ __forceinline__ void copy_scale_rows(const SplitParams& p, uint8_t* sc, int row, int64_t page, int kvh,
                                                int slot) {
    static_assert(SCB == 8 || SCB == 16, "scale rows of 8 or 16 bytes");
    const uint8_t* ks = p.ks_base + page * p.ks_sp + kvh * p.ks_sh + slot * p.ks_st;
    const uint8_t* vs = p.vs_base + page * p.vs_sp + kvh * p.vs_sh + slot * p.vs_st;
    if constexpr (SCB == 16) {
        cp_async_16(smem_addr(sc + row * SCB), ks);
        cp_async_16(smem_addr(sc + (TOK + row) * SCB), vs);
    } else {
        cp_async_8(smem_addr(sc + row * SCB), ks);
        cp_async_8(smem_addr(sc + (TOK + row) * SCB), vs);
    }
}

// The producer warp: fills stage i (TOK tokens) into slot i % S once the slot is released.
// EB: bytes per stored K/V element (2: 16-bit, 1: E4M3 or q8_0 codes).  SCB > 0 (q8_0
// caches): each stage also gets its tokens' K and V block-scale rows (SCB bytes each) in
// the slot's area of sc_ring (2 TOK SCB bytes per slot); in TMA mode every lane then
// arrives once on the stage's full barrier after its copies (which counts those 32
// arrivals besides the expect-tx one).
// BOXMAJ: when a page holds fewer tokens than a stage, each page's rows land as one box
// of every region ([box][region][BR rows][128 B], see stage_row_offset; the tensor map's
// box spans all regions) instead of one box per region into the region-major layout:
// a TMA instruction costs about the same whatever its size, and with one box per region
// the producer's issue time bounded the stream at page sizes 8 and 16.
template <int D, int S, int TOK = kStageTokens, int EB = 2, int SCB = 0, bool BOXMAJ = false>
__device__ __forceinline__ void produce_stages(const SplitParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv, uint64_t* full,
                               uint64_t* empty, uint8_t* stages, int b, int kvh, const ItemRange& ir,
                               bool tma_mode, uint8_t* sc_ring = nullptr) {
    using G = StageGeom<D, TOK, EB>;
    static_assert(TOK % 32 == 0 && TOK <= 256, "stage rows");
    static_assert(SCB == 0 || TOK == 32, "scale rows: one token per lane");
    static_assert(G::ROW_BYTES % 128 == 0, "rows of whole 128-byte regions");
    const int lane = threadIdx.x & 31;
    const int tok_begin = ir.tok_begin;
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride;
    const int page_mask = (1 << p.page_shift) - 1;
    int issued = 0;
    bool ok = true;
    if (tma_mode) {
        // Boxes of BR token rows, NB boxes per stage; the page id of box n is
        // held by lane n % 32, one group of 32 boxes ahead.  The first two groups
        // are loaded before the run-time length is known (bounded by the item's
        // planned blocks and the table row, so every read is in bounds; ids of
        // boxes past the length are never used).
        // (boxes never cross a page: a stage starts on a 64-token block boundary)
        const int BR = min(1 << p.page_shift, min(TOK, kBlockTokens));
        const int NB = TOK / BR;
        auto box_page = [&](int n) -> int {
            const int t = tok_begin + n * BR;
            return (t < ir.tok_end_alloc && (t >> p.page_shift) < p.pt_stride) ? __ldg(pt + (t >> p.page_shift)) : -1;
        };
        int pid = box_page(lane);
        int pid_next = box_page(32 + lane);
        const int tok_end = ir.tok_end, n_stage = ir.n_stage;
        if (n_stage == 0) return;
        const int n_box = (tok_end - tok_begin + BR - 1) / BR;
        const uint32_t box_bytes = static_cast<uint32_t>(BR) * 2u * G::ROW_BYTES;  // K and V
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
            const uint32_t fbar = smem_addr(&full[i % (2 * S)]);
            if (lane == 0) mbar_arrive_expect_tx(fbar, static_cast<uint32_t>(__popc(vmask)) * box_bytes);
            __syncwarp();
            if (valid) {  // lane j issues box j (every region in one instruction when the box spans the stage)
                const int slot0 = (tok_begin + (box0 + lane) * BR) & page_mask;
                const uint32_t kdst = smem_addr(stages + s * G::STAGE_BYTES + lane * BR * (BOXMAJ ? G::ROW_BYTES : 128));
                if (NB == 1 || BOXMAJ) {
                    tma_load_kv_box(kdst, tmk, slot0, 0, kvh, my_page, fbar);
                    tma_load_kv_box(kdst + G::HALF_BYTES, tmv, slot0, 0, kvh, my_page, fbar);
                } else {
                    for (int r = 0; r < G::REGIONS; ++r) {
                        tma_load_kv_box(kdst + r * G::REGION_BYTES, tmk, slot0, r, kvh, my_page, fbar);
                        tma_load_kv_box(kdst + G::HALF_BYTES + r * G::REGION_BYTES, tmv, slot0, r, kvh, my_page, fbar);
                    }
                }
            }
            if constexpr (SCB > 0) {
                const int tok = tok_begin + i * TOK + lane;  // lane = row of the stage
                const int spage = __shfl_sync(0xffffffffu, pid, (box0 + lane / BR) & 31);
                if (tok < tok_end && spage >= 0 && spage < p.k_pages && spage < p.v_pages)
                    copy_scale_rows<TOK, SCB>(p, sc_ring + s * (2 * TOK * SCB), lane, spage, kvh, tok & page_mask);
                cp_async_arrive_noinc(fbar);
            }
            issued = i + 1;
        }
    } else {
        // Small pages: 16-byte cp.async per (row, chunk) into the swizzled layout.
        const int tok_end = ir.tok_end, n_stage = ir.n_stage;
        if (n_stage == 0) return;
        constexpr int CHUNKS = G::ROW_BYTES / 16;
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
            uint8_t* sbase = stages + s * G::STAGE_BYTES;
            for (int rb = 0; rb < TOK; rb += 32) {  // 32 rows at a time: lane = row for the page lookup
                const int t_lane = tok_begin + i * TOK + rb + lane;
                const bool in_range = t_lane < tok_end;
                const int my_page = in_range ? __ldg(pt + (t_lane >> p.page_shift)) : -1;
                const bool valid = in_range && my_page >= 0 && my_page < p.k_pages && my_page < p.v_pages;
                if (in_range && !valid) atomicOr(p.err, FDEC_DEVERR_PAGE_ID);
                for (int idx = lane; idx < 32 * CHUNKS; idx += 32) {
                    const int r32 = idx / CHUNKS;
                    const int c = idx - r32 * CHUNKS;
                    const int page = __shfl_sync(0xffffffffu, my_page, r32);
                    const bool ok_row = __shfl_sync(0xffffffffu, valid, r32);
                    if (ok_row) {
                        const int row = rb + r32;
                        const int slot = (tok_begin + i * TOK + row) & page_mask;
                        const uint32_t off = (c >> 3) * G::REGION_BYTES + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                        cp_async_16(smem_addr(sbase + off),
                                    p.k_base + page * p.k_sp + kvh * p.k_sh + slot * p.k_st + c * 16);
                        cp_async_16(smem_addr(sbase + G::HALF_BYTES + off),
                                    p.v_base + page * p.v_sp + kvh * p.v_sh + slot * p.v_st + c * 16);
                    }
                }
                if constexpr (SCB > 0) {
                    if (valid) copy_scale_rows<TOK, SCB>(p, sc_ring + s * (2 * TOK * SCB), rb + lane, my_page, kvh,
                                                         t_lane & page_mask);
                }
            }
            cp_async_arrive_noinc(smem_addr(&full[i % (2 * S)]));
            issued = i + 1;
        }
    }
    // Do not leave while copies of this CTA may still be landing.
    for (int i = issued > S ? issued - S : 0; i < issued; ++i) {
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(smem_addr(&full[i % (2 * S)]), (i / (2 * S)) & 1);
        if (!__shfl_sync(0xffffffffu, got, 0)) ok = false;
    }
    if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);
}

// Consumer side of stage i: wait until it has landed.  Stage i completes
// full[i % 2S] in phase i / 2S.  Stages land out of order and a slot's phases
// are consumed by different warps, but the previous phase of this barrier (stage
// i - 2S) was consumed before stage i - S was issued, and that was issued before
// the caller's previous stage: so the barrier is in phase i / 2S or just past it,
// and the parity test is unambiguous.
template <int S>
__device__ __forceinline__ bool wait_stage(uint64_t* full, int i) {
    bool got = true;
    if ((threadIdx.x & 31) == 0) got = mbar_wait_bounded(smem_addr(&full[i % (2 * S)]), (i / (2 * S)) & 1);
    return __shfl_sync(0xffffffffu, got, 0) != 0;
}

// A partial (last) stage: rows past the sequence end hold whatever the page
// held; zero its V rows [nv, TOK) so that a fixed-size p.V loop adds 0 * 0.
// `threads` consecutive threads (from `tid` 0) share the work.
template <int D, int TOK = kStageTokens, int EB = 2>
__device__ __forceinline__ void zero_v_tail(uint8_t* stage, int nv, int tid = threadIdx.x & 31, int threads = 32,
                                            int br = TOK) {
    using G = StageGeom<D, TOK, EB>;
    uint8_t* vrows = stage + G::HALF_BYTES;
    for (int idx = tid; idx < (TOK - nv) * G::REGIONS * 8; idx += threads) {
        const int row = nv + idx / (G::REGIONS * 8);
        const int rem = idx % (G::REGIONS * 8);
        const uint32_t off = br == TOK ? (rem >> 3) * G::REGION_BYTES + row * 128
                                       : stage_row_offset<G::ROW_BYTES>(row, br) + (rem >> 3) * (br * 128);
        *reinterpret_cast<uint4*>(vrows + off + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (threads == 32) __syncwarp();
}

// Epilogue, after every consumer has written its state to the scratch
// sm_m [NW][RC], sm_l [NW][RC], sm_o [NW][RC][D] and passed a barrier: merge the
// NW states by log-sum-exp (m in log2 units) and write the split's partial or,
// when one split covers the sequence, out = O / L and lse = ln 2 * (M + log2 L).
// O is scaled by v_scale (the value scale of a quantised cache, 1 otherwise): the
// LSE merge is linear in O, so partials may carry it.
// NTHREADS consumer threads (from thread 0) share the work.
template <int NW, int RC, int D, int NTHREADS = NW * 32>
__device__ __forceinline__ void merge_and_store(const SplitParams& p, const WorkItem& it, int kvh, int row0,
                                                const float* sm_m, const float* sm_l, const float* sm_o) {
    constexpr float kLn2 = 0.69314718055994530942f;
    for (int idx = threadIdx.x; idx < RC * D; idx += NTHREADS) {
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
            const int64_t orow = static_cast<int64_t>(it.seq * p.q_len + qi) * p.hq + h;
            p.out[orow * D + d] = Ls > 0.f ? O / Ls * p.v_scale : 0.f;
            if (d == 0 && p.lse != nullptr) p.lse[orow] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
        } else {
            const int64_t prow = (static_cast<int64_t>(it.slot) * p.hk + kvh) * p.rows + row;
            p.part_o[prow * D + d] = O * p.v_scale;
            if (d == 0) p.part_ml[prow] = make_float2(M, Ls);
        }
    }
}

}  // namespace fdec
