// split_persist_kernel.cuh -- the persistent form of the tensor-core split kernel
// (16-bit caches, every head_dim).
//
// Why: with one CTA per work item, every CTA pays a pipeline fill (work item,
// length, page ids, first TMA: three dependent memory round trips) and the
// launch ends with the slowest CTA.  Measured on a flushed 131072-token decode
// (76 items x 4 KV heads, one wave of 304 CTAs), the K/V stream itself runs at
// 7.2-7.5 TB/s, but per-CTA rates spread by +-12 % under saturation, so the last
// CTAs finish ~4 us after the median one; cutting the items smaller to balance
// them costs ~5 us of fill and epilogue per extra CTA.
//
// Here the CTAs stay resident (two per SM) and take work units (a work item x
// a KV head x a 16-row query group) until none is left: CTA c starts with unit
// c, and the units past the grid are handed out by one 64-bit ticket counter, so
// a CTA that streams faster takes more of them.  (The planner keeps uniform runs
// of blocks: a first wave of big items with a tail of small ones, which balances
// the CTAs to within one small item, measured slower, as every unit adds a
// partial, a merge and a hand-over of the pipeline.)  Results do not
// depend on which CTA takes a unit: every unit has its fixed partial slot and
// is computed by the same code in the same order (its stage j by consumer warp
// j mod 3, the three warp states merged in warp order), so a fixed plan stays
// bitwise deterministic and equal to the one-CTA-per-item kernel.
//
// The counter needs no reset: every CTA takes units until one take fails, so a
// launch takes exactly (dynamic units + grid) = n_units tickets; a unit is the
// ticket modulo n_units.  (The plan upload and the no-alloc entry point zero it.)
//
// Pipeline (producer warp + 3 consumer warps, ring of S 32-token stages):
//   - the producer walks its units back to back: a unit's stages are padded to
//     a multiple of 3 (empty stages carry no data), so stage j of every unit
//     goes to consumer warp j mod 3; the unit's query rows (16-byte aligned
//     rows, one bulk copy each) land with its first stage in one of two query
//     buffers; a tag per ring slot names the unit buffer and j (2 j + buffer).  The next unit's
//     ticket, work item, length and first page ids are fetched while the last
//     three stages of the current unit are issued.
//   - a consumer warp resets its state at its first stage of a unit and, at its
//     last, writes its (m, l, O) into that stage's slot (kept, not released) and
//     counts itself in; the third warp to arrive merges the three states, writes
//     the partial (or out / lse), then releases the three kept slots and the
//     unit's query buffer.  No warp ever waits for another warp, so a failed
//     (bounded) wait cannot leave a warp stuck at a barrier.
#pragma once

#include "split_mma_kernel.cuh"

namespace fdec {

// Consumer side of stage i (the parity argument of wait_stage).  poll: wait by
// polling rather than suspended.  Measured on sm_103a: with pages of fewer than 32
// tokens (a stage lands as several TMA boxes) suspended consumers resumed late,
// 10 us of 47 on a speculative-decode batch, and polling wins; with whole-stage
// boxes suspending is better (polling warps take issue slots from the producers:
// +1.5 us at 131072 tokens).
template <int S>
__device__ __forceinline__ bool wait_stage_mode(uint64_t* full, int i, bool poll) {
    bool got = true;
    if ((threadIdx.x & 31) == 0) {
        const uint32_t bar = smem_addr(&full[i % (2 * S)]);
        const uint32_t parity = (i / (2 * S)) & 1;
        got = poll ? mbar_wait_polling(bar, parity) : mbar_wait_bounded(bar, parity);
    }
    return __shfl_sync(0xffffffffu, got, 0) != 0;
}

// What the producer tells the consumers about a unit (with its first stage).
struct UnitMeta {
    int seq, kvh, row0, slot;  // slot: partial slot, or -1 (the unit writes out / lse)
    int L;                     // run-time length, clamped to the planned capacity
    int tok_begin, tok_end;    // tokens streamed: clipped to L and, causal, to the last visible token
    int n_pad;                 // ring stages of the unit: a multiple of NP, at least NP
};

// BM: stages of pages smaller than a stage land box-major (one TMA box per page); the
// launch takes the BM = false instantiation for every other page size, whose row
// addresses are fixed at compile time (measured: the box-major build, identical in
// what it does at 64-token pages, ran 10 % slower there at 66-76 splits).
template <int D, bool BM = true>
struct PersistLayout {
    using G = StageGeom<D>;
    static constexpr int RC = 16;                      // query rows per unit (one M tile)
    // head_dim 512: two warps share each stage, each accumulating half of O's
    // columns (DH), as in MmaLayout; one CTA per SM (stages of 64 KB).
    static constexpr int DSPLIT = D > 256 ? 2 : 1;
    static constexpr int DH = D / DSPLIT;
    static constexpr int CTAS_PER_SM = D > 256 ? 1 : 2;  // = split_mma_persist_ctas_per_sm(D)
    static constexpr bool BOXMAJ = BM && DSPLIT == 1;    // one box per small page
    // Two query buffers (the next unit's rows land while the last one still reads its
    // own) where they fit beside enough stages; one above head_dim 192 (the producer
    // then starts a unit once the previous one is merged).
    static constexpr int QBUFS = D > 192 ? 1 : 2;
    static constexpr int Q_BYTES = RC * D * 2;         // one unit's query rows
    static constexpr int CTRL_BYTES = 2048;            // barriers, tags, unit records, merge scalars
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int BUDGET = 232448 / CTAS_PER_SM - 1024;
    static constexpr int FIXED = CTRL_BYTES + QBUFS * Q_BYTES + ALIGN_SLACK;
    static constexpr int S_FIT = (BUDGET - FIXED) / G::STAGE_BYTES;
    static constexpr int S = S_FIT > 16 ? 16 : S_FIT;
    static constexpr int NP = (S - 1) < 3 ? (S - 1) : 3;  // consumer groups (one stage each at a time)
    static constexpr int NW = NP * DSPLIT;                 // consumer warps
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr int SMEM = FIXED + S * G::STAGE_BYTES;
    // Where a group's O goes in its kept slot.  One warp per group: anywhere, rows of
    // D + 4 floats (bank spread).  Two warps per group: each into its own half of the
    // stage's V rows, which only it reads (its partner may still be reading K).
    static constexpr int O_BASE = DSPLIT == 1 ? 0 : G::HALF_BYTES;  // bytes into the slot
    static constexpr int O_ROW = DSPLIT == 1 ? D + 4 : DH;          // floats between rows
    static constexpr int O_HALF = RC * DH;                          // floats between column halves
    // control area
    static constexpr int OFF_FULL = 0;                 // 2S
    static constexpr int OFF_EMPTY = OFF_FULL + 2 * S * 8;   // S
    static constexpr int OFF_QFREE = OFF_EMPTY + S * 8;      // 2
    static constexpr int OFF_TAG = OFF_QFREE + 16;           // S ints
    static constexpr int OFF_UNIT = (OFF_TAG + S * 4 + 15) / 16 * 16;  // 2 UnitMeta
    static constexpr int OFF_ML = OFF_UNIT + 2 * static_cast<int>(sizeof(UnitMeta));  // [2][NP][RC] float2
    static constexpr int OFF_CNT = OFF_ML + 2 * NP * RC * 8;  // 2 ints
    static_assert(OFF_CNT + 8 <= CTRL_BYTES, "control area");
    static_assert(DSPLIT == 1 ? RC * O_ROW * 4 <= G::STAGE_BYTES : O_HALF * 4 <= G::HALF_BYTES / 2,
                  "a group's O must fit its kept slot");
    static_assert(NP >= 2 && S >= NP + 1, "stage ring too small");
};

// A work unit as the producer sees it: the unit index, its work item, the run-time
// length and capacity of its sequence, and this lane's page ids of box groups 0
// and 1 (TMA mode).
struct PUnit {
    int unit;  // -1: none
    int4 it;   // seq, block_begin, block_end, slot
    int L0, cap;
    int pid0, pid1;
};

__device__ __forceinline__ void punit_load_item(const SplitParams& p, PUnit& u, int upi) {
    const int idx = u.unit / upi;
    if (p.seq1_bps > 0) {
        const int ns = (p.seq1_blocks + p.seq1_bps - 1) / p.seq1_bps;
        u.it = make_int4(0, idx * p.seq1_bps, min((idx + 1) * p.seq1_bps, p.seq1_blocks), ns > 1 ? idx : -1);
    } else {
        u.it = __ldg(reinterpret_cast<const int4*>(p.items) + idx);
    }
}

// Page id of TMA box n (BR token rows) of the unit, or -1 past its planned blocks.
__device__ __forceinline__ int punit_box_page(const SplitParams& p, const PUnit& u, int n, int BR) {
    const int t = u.it.y * kBlockTokens + n * BR;
    const int32_t* pt = p.page_table + static_cast<int64_t>(u.it.x) * p.pt_stride;
    return (t < u.it.z * kBlockTokens && (t >> p.page_shift) < p.pt_stride) ? __ldg(pt + (t >> p.page_shift)) : -1;
}

// Length and first page ids (before the length is known: bounded by the item's
// planned blocks and the table row, so every read is in bounds).
__device__ __forceinline__ void punit_load_lens_pages(const SplitParams& p, PUnit& u, int lane, int BR,
                                                      bool tma_mode) {
    u.L0 = __ldg(p.seq_lens + u.it.x);
    u.cap = p.seq1_bps > 0 ? p.seq1_capacity : __ldg(p.capacity + u.it.x);
    if (tma_mode) {
        u.pid0 = punit_box_page(p, u, lane, BR);
        u.pid1 = punit_box_page(p, u, 32 + lane, BR);
    }
}

// The producer warp of the persistent kernel.  `first`: the CTA's first unit, its
// loads issued before the CTA's set-up so that they overlap it.
template <int D, int S, int NP, int QBUFS, bool BOXMAJ>
__device__ __forceinline__ void produce_units(const SplitParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                              uint64_t* full, uint64_t* empty, uint64_t* qfree, int* tag,
                                              UnitMeta* um, uint16_t* qbuf, uint8_t* stages, bool tma_mode,
                                              PUnit cur) {
    using G = StageGeom<D>;
    constexpr int RC = 16;
    constexpr int TOK = kStageTokens;
    const int lane = threadIdx.x & 31;
    const int rgc = (p.rows + RC - 1) / RC;
    const int upi = p.hk * rgc;                           // units per work item
    const int n_units = p.n_units;
    const int n_dyn = n_units - static_cast<int>(gridDim.x);  // units handed out by the ticket counter
    const int page_mask = (1 << p.page_shift) - 1;
    const int BR = tma_mode ? min(1 << p.page_shift, TOK) : 1;  // token rows per TMA box
    const int NB = TOK / BR;                                      // boxes per stage
    const uint32_t box_bytes = static_cast<uint32_t>(BR) * 2u * G::ROW_BYTES;  // K and V
    const uint32_t q_row_bytes = D * 2;

    auto load_item = [&](PUnit& u) { punit_load_item(p, u, upi); };
    auto box_page = [&](const PUnit& u, int n) -> int { return punit_box_page(p, u, n, BR); };
    auto load_lens_pages = [&](PUnit& u) { punit_load_lens_pages(p, u, lane, BR, tma_mode); };
    // Tickets: lane 0 takes one; resolved to a unit (or -1: no unit left).
    unsigned long long ticket = 0;
    auto take = [&]() {
        if (lane == 0) ticket = atomicAdd(p.ticket, 1ull);
    };
    auto resolve = [&]() -> int {
        const unsigned long long v = __shfl_sync(0xffffffffu, ticket, 0);
        const unsigned long long r = v % static_cast<unsigned long long>(n_units);
        return r < static_cast<unsigned long long>(n_dyn) ? static_cast<int>(gridDim.x) + static_cast<int>(r) : -1;
    };

    bool ok = true;
    int i = 0;  // ring stages issued
    int k = 0;  // units issued by this CTA
    bool pending = false;  // a ticket taken and not resolved
    PUnit nxt;
    nxt.unit = -1;
    // Look-ahead of the next unit, one step per issued stage over the last three stages
    // of the current one: 0 nothing yet, 1 ticket taken, 2 unit known and its work item
    // requested, 3 length and page ids requested.
    int ahead = 0;
    auto advance = [&]() {
        if (ahead == 0) {
            if (n_dyn > 0) {
                take();
                pending = true;
                ahead = 1;
            } else {
                ahead = 3;
            }
        } else if (ahead == 1) {
            nxt.unit = resolve();
            pending = false;
            if (nxt.unit >= 0) {
                load_item(nxt);
                ahead = 2;
            } else {
                ahead = 3;
            }
        } else if (ahead == 2) {
            load_lens_pages(nxt);
            ahead = 3;
        }
    };
    auto wait_slot = [&](int idx) -> bool {
        bool got = true;
        if (idx >= S && lane == 0) got = mbar_wait_bounded(smem_addr(&empty[idx % S]), ((idx / S) - 1) & 1);
        return __shfl_sync(0xffffffffu, got, 0) != 0;
    };

    while (ok && cur.unit >= 0) {
        const int cb = k % QBUFS;
        // ---- the unit's record
        const int rem = cur.unit % upi;
        const int kvh = rem / rgc;
        const int row0 = (rem % rgc) * RC;
        const int seq = cur.it.x;
        const bool bad = cur.L0 > cur.cap || cur.L0 < 0;
        if (bad && lane == 0) atomicOr(p.err, FDEC_DEVERR_SEQ_LEN);
        const int L = cur.L0 < 0 ? 0 : (cur.L0 > cur.cap ? cur.cap : cur.L0);
        const int tok_begin = cur.it.y * kBlockTokens;
        int tok_end = min(cur.it.z * kBlockTokens, L);
        if (p.causal) {  // no row of the unit sees past L - Q + (its last q position)
            const int last_row = min(row0 + RC, p.rows) - 1;
            tok_end = min(tok_end, L - p.q_len + last_row / p.group + 1);
        }
        const int n_stage = tok_end > tok_begin ? (tok_end - tok_begin + TOK - 1) / TOK : 0;
        const int n_pad = max(NP, (n_stage + NP - 1) / NP * NP);
        // ---- its query buffer and record are free once unit k - QBUFS has been merged
        if (k >= QBUFS) {
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(smem_addr(&qfree[cb]), ((k / QBUFS) - 1) & 1);
            if (!__shfl_sync(0xffffffffu, got, 0)) {
                ok = false;
                break;
            }
        }
        if (lane == 0) {
            UnitMeta m;
            m.seq = seq;
            m.kvh = kvh;
            m.row0 = row0;
            m.slot = cur.it.w;
            m.L = L;
            m.tok_begin = tok_begin;
            m.tok_end = tok_end;
            m.n_pad = n_pad;
            um[cb] = m;
        }
        const int n_box = tok_end > tok_begin ? (tok_end - tok_begin + BR - 1) / BR : 0;
        int pid = cur.pid0, pid_next = cur.pid1, group = 0;
        uint16_t* q_dst = qbuf + cb * RC * D;
        for (int j = 0; j < n_pad; ++j, ++i) {
            // The next unit is taken only near the end of this one (the producer runs about
            // S stages ahead of the consumers), so that a CTA that streams slowly takes
            // fewer.  (Taking it as a unit starts was measured slower on a ragged batch,
            // 382 against 283 us: the assignment then runs one unit ahead of the work.)
            if (j >= n_pad - 3 && ahead < 3) advance();
            const int s = i % S;
            if (!wait_slot(i)) {
                ok = false;
                break;
            }
            if (lane == 0) tag[s] = (j << 1) | cb;
            const uint32_t fbar = smem_addr(&full[i % (2 * S)]);
            uint8_t* sbase = stages + s * G::STAGE_BYTES;
            // the query rows travel with the unit's first stage (none for an empty unit)
            const int q_rows = (j == 0 && n_stage > 0) ? min(RC, p.rows - row0) : 0;
            if (j >= n_stage) {
                // a padding stage: no data, the phase completes on the arrivals alone
                if (tma_mode) {
                    if (lane == 0) mbar_arrive_expect_tx(fbar, 0u);
                } else {
                    mbar_arrive(fbar);
                    if (lane == 0) mbar_arrive(fbar);
                }
                continue;
            }
            if (tma_mode) {
                const int box0 = j * NB;
                if ((box0 >> 5) != group) {  // NB divides 32: a stage never straddles two groups
                    pid = pid_next;
                    group = box0 >> 5;
                    pid_next = box_page(cur, (group + 1) * 32 + lane);
                }
                const int my_page = __shfl_sync(0xffffffffu, pid, (box0 + lane) & 31);
                const bool in_range = lane < NB && box0 + lane < n_box;
                const bool valid = in_range && my_page >= 0 && my_page < p.k_pages && my_page < p.v_pages;
                if (in_range && !valid) atomicOr(p.err, FDEC_DEVERR_PAGE_ID);
                const unsigned vmask = __ballot_sync(0xffffffffu, valid);
                if (lane == 0)
                    mbar_arrive_expect_tx(fbar, static_cast<uint32_t>(__popc(vmask)) * box_bytes +
                                                    static_cast<uint32_t>(q_rows) * q_row_bytes);
                __syncwarp();
                if (lane < q_rows) {
                    const int row = row0 + lane;
                    const int qi = row / p.group;
                    const int h = kvh * p.group + (row - qi * p.group);
                    const uint16_t* src = p.q + static_cast<int64_t>(seq * p.q_len + qi) * p.q_stride_tok +
                                          static_cast<int64_t>(h) * p.q_stride_head;
                    bulk_g2s(smem_addr(q_dst + lane * D), src, q_row_bytes, fbar);
                }
                if (valid) {  // lane j issues box j (every region in one instruction when the box spans the
                              // stage or the layout is box-major)
                    const int slot0 = (tok_begin + (box0 + lane) * BR) & page_mask;
                    const uint32_t kdst = smem_addr(sbase + lane * BR * (BOXMAJ ? G::ROW_BYTES : 128));
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
            } else {
                // small pages: 16-byte cp.async per (row, chunk) into the swizzled layout
                if (q_rows > 0) {
                    if (lane == 0) mbar_expect_tx(fbar, static_cast<uint32_t>(q_rows) * q_row_bytes);
                    __syncwarp();
                    if (lane < q_rows) {
                        const int row = row0 + lane;
                        const int qi = row / p.group;
                        const int h = kvh * p.group + (row - qi * p.group);
                        const uint16_t* src = p.q + static_cast<int64_t>(seq * p.q_len + qi) * p.q_stride_tok +
                                              static_cast<int64_t>(h) * p.q_stride_head;
                        bulk_g2s(smem_addr(q_dst + lane * D), src, q_row_bytes, fbar);
                    }
                }
                constexpr int CHUNKS = G::ROW_BYTES / 16;
                const int32_t* pt = p.page_table + static_cast<int64_t>(seq) * p.pt_stride;
                const int t_lane = tok_begin + j * TOK + lane;
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
                        const int slot = (tok_begin + j * TOK + r32) & page_mask;
                        const uint32_t off = (c >> 3) * G::REGION_BYTES + r32 * 128 + (((c & 7) ^ (r32 & 7)) << 4);
                        cp_async_16(smem_addr(sbase + off),
                                    p.k_base + page * p.k_sp + kvh * p.k_sh + slot * p.k_st + c * 16);
                        cp_async_16(smem_addr(sbase + G::HALF_BYTES + off),
                                    p.v_base + page * p.v_sp + kvh * p.v_sh + slot * p.v_st + c * 16);
                    }
                }
                cp_async_arrive_noinc(fbar);
                if (lane == 0) mbar_arrive(fbar);  // orders the tag and unit record before the phase
            }
        }
        if (!ok) break;
        while (ahead < 3) advance();
        cur = nxt;
        nxt.unit = -1;
        ahead = 0;
        ++k;
    }
    if (!ok) {
        // Keep the ticket count of this launch exact: a CTA stops at its first failed take.
        if (n_dyn > 0) {
            bool more = true;
            if (pending) more = resolve() >= 0;
            else if (ahead == 3 && nxt.unit < 0) more = false;  // its failed take is already counted
            while (more) {
                take();
                more = resolve() >= 0;
            }
        }
    } else {
        // No unit left: one end tag per consumer group.
        for (int w = 0; w < NP; ++w, ++i) {
            if (!wait_slot(i)) {
                ok = false;
                break;
            }
            const int s = i % S;
            if (lane == 0) tag[s] = -1;
            const uint32_t fbar = smem_addr(&full[i % (2 * S)]);
            if (tma_mode) {
                if (lane == 0) mbar_arrive_expect_tx(fbar, 0u);
            } else {
                mbar_arrive(fbar);
                if (lane == 0) mbar_arrive(fbar);
            }
        }
    }
    // The reduction (a programmatic dependent) may start launching.
    if (lane == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Do not leave while copies of this CTA may still be landing.
    for (int x = i > S ? i - S : 0; x < i; ++x) {
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(smem_addr(&full[x % (2 * S)]), (x / (2 * S)) & 1);
        if (!__shfl_sync(0xffffffffu, got, 0)) ok = false;
    }
    if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);
}

// Merge the NP consumer states of a unit (m, l per row in ml[NP][RC]; O in the kept
// slots: column c of row r at (c / DH) O_HALF + r O_ROW + c % DH floats) and write the
// unit's partial or out / lse.
// One warp: lane r first takes the statistics of row r (max, weights, sum), then the
// lanes stride over (row, 4 columns) pairs with the row's values broadcast from its
// lane.  The arithmetic and its order are those of merge_and_store.
template <int D, int NP, int RC, int DH, int O_ROW, int O_HALF>
__device__ __forceinline__ void merge_unit(const SplitParams& p, const UnitMeta& u, const float2* ml,
                                           const float* const (&o_w)[NP], int lane) {
    constexpr float kLn2 = 0.69314718055994530942f;
    constexpr int C4 = D / 4;
    const int nrows = min(RC, p.rows - u.row0);
    float M = -INFINITY, Ls = 0.f, e[NP];
#pragma unroll
    for (int w = 0; w < NP; ++w) e[w] = 0.f;
    if (lane < nrows) {
#pragma unroll
        for (int w = 0; w < NP; ++w) M = fmaxf(M, ml[w * RC + lane].x);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NP; ++w) {
                e[w] = exp2_approx(ml[w * RC + lane].x - M);
                Ls += ml[w * RC + lane].y * e[w];
            }
        }
        const int row = u.row0 + lane;
        const int qi = row / p.group;
        const int h = u.kvh * p.group + (row - qi * p.group);
        if (u.slot < 0) {
            if (p.lse != nullptr)
                p.lse[static_cast<int64_t>(u.seq * p.q_len + qi) * p.hq + h] =
                    Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
        } else {
            p.part_ml[(static_cast<int64_t>(u.slot) * p.hk + u.kvh) * p.rows + row] = make_float2(M, Ls);
        }
    }
    const int total = nrows * C4;
    for (int x0 = 0; x0 < total; x0 += 32) {
        const int x = x0 + lane;
        const int r = min(x, total - 1) / C4;
        const float Mr = __shfl_sync(0xffffffffu, M, r);
        const float Lr = __shfl_sync(0xffffffffu, Ls, r);
        float er[NP];
#pragma unroll
        for (int w = 0; w < NP; ++w) er[w] = __shfl_sync(0xffffffffu, e[w], r);
        if (x >= total) continue;
        const int c4 = x - r * C4;
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Mr != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NP; ++w) {
                const int c = 4 * c4;
                const float4 v = *reinterpret_cast<const float4*>(o_w[w] + (c / DH) * O_HALF + r * O_ROW + c % DH);
                O.x += v.x * er[w];
                O.y += v.y * er[w];
                O.z += v.z * er[w];
                O.w += v.w * er[w];
            }
        }
        const int row = u.row0 + r;
        const int qi = row / p.group;
        const int h = u.kvh * p.group + (row - qi * p.group);
        if (u.slot < 0) {
            const int64_t orow = static_cast<int64_t>(u.seq * p.q_len + qi) * p.hq + h;
            *reinterpret_cast<float4*>(p.out + orow * D + 4 * c4) =
                Lr > 0.f ? make_float4(O.x / Lr * p.v_scale, O.y / Lr * p.v_scale, O.z / Lr * p.v_scale,
                                       O.w / Lr * p.v_scale)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const int64_t prow = (static_cast<int64_t>(u.slot) * p.hk + u.kvh) * p.rows + row;
            *reinterpret_cast<float4*>(p.part_o + prow * D + 4 * c4) =
                make_float4(O.x * p.v_scale, O.y * p.v_scale, O.z * p.v_scale, O.w * p.v_scale);
        }
    }
}

template <int D, bool BF16, bool BM>
__global__ void __launch_bounds__(PersistLayout<D, BM>::THREADS, PersistLayout<D, BM>::CTAS_PER_SM)
split_mma_persist_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
    using Lay = PersistLayout<D, BM>;
    using W = MmaWarp<D, BF16, false, false, Lay::BOXMAJ>;
    using G = StageGeom<D>;
    constexpr int S = Lay::S;
    constexpr int NP = Lay::NP;
    constexpr int NW = Lay::NW;
    constexpr int DSPLIT = Lay::DSPLIT;
    constexpr int DH = Lay::DH;
    constexpr int QBUFS = Lay::QBUFS;
    constexpr int RC = Lay::RC;
    constexpr int NT = W::NT;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::OFF_FULL);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + Lay::OFF_EMPTY);
    uint64_t* qfree = reinterpret_cast<uint64_t*>(smem + Lay::OFF_QFREE);
    int* tag = reinterpret_cast<int*>(smem + Lay::OFF_TAG);
    UnitMeta* um = reinterpret_cast<UnitMeta*>(smem + Lay::OFF_UNIT);
    float2* mls = reinterpret_cast<float2*>(smem + Lay::OFF_ML);  // [2][NP][RC]
    int* cnt = reinterpret_cast<int*>(smem + Lay::OFF_CNT);       // [2]
    uint16_t* qbuf = reinterpret_cast<uint16_t*>(smem + Lay::CTRL_BYTES);  // [QBUFS][RC][D]
    uint8_t* stages;
    {
        const uint32_t raw = smem_addr(smem) + Lay::CTRL_BYTES + QBUFS * Lay::Q_BYTES;
        const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
        stages = smem + Lay::CTRL_BYTES + QBUFS * Lay::Q_BYTES + pad;
    }

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool tma_mode = p.page_shift >= 3;
    // The producer's first unit: its work item, length and page ids are requested now,
    // before the set-up below, so that those round trips overlap it.
    PUnit first;
    first.unit = -1;
    if (warp == NW) {
        first.unit = blockIdx.x;
        punit_load_item(p, first, p.hk * ((p.rows + RC - 1) / RC));  // plan data
        // Launched as a programmatic dependent of the kernel before it in the stream (a
        // no-op without one): every input (lengths, page table, q, K, V) and every output
        // it may still read or write is touched only after that kernel has completed.  The
        // consumers' reads and writes follow the producer's stages.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        punit_load_lens_pages(p, first, lane, tma_mode ? min(1 << p.page_shift, kStageTokens) : 1, tma_mode);
    }
    if (threadIdx.x == 0) {
        // Stage barriers: TMA stages complete on one expect-tx arrival; small-page stages
        // on the 32 cp.async arrivals of the producer lanes plus one plain arrival of lane
        // 0, which orders its tag and unit-record writes before the phase completes.
        for (int x = 0; x < S; ++x) {
            mbar_init(smem_addr(&full[x]), tma_mode ? 1u : 33u);
            mbar_init(smem_addr(&full[S + x]), tma_mode ? 1u : 33u);
            mbar_init(smem_addr(&empty[x]), static_cast<uint32_t>(DSPLIT));  // the warps of a group
        }
        mbar_init(smem_addr(&qfree[0]), 1);
        mbar_init(smem_addr(&qfree[1]), 1);
        fence_mbar_init();
        cnt[0] = cnt[1] = 0;
    }
    // Query rows past a unit's group are never copied: zero the buffers once.
    for (int x = threadIdx.x; x < QBUFS * Lay::Q_BYTES / 16; x += Lay::THREADS)
        reinterpret_cast<uint4*>(qbuf)[x] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_shared();  // before the bulk copies overwrite rows of them
    __syncthreads();

    if (warp == NW) {
        if (lane == 0 && tma_mode) {
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
        }
        produce_units<D, S, NP, QBUFS, Lay::BOXMAJ>(p, &tmk, &tmv, full, empty, qfree, tag, um, qbuf, stages, tma_mode,
                                                    first);
        return;
    }

    // ---------------------------------------------------------------------- consumers
    W cw(lane, staged_box_rows(p.page_shift, Lay::BOXMAJ));
    const int g = cw.g, tq = cw.tq;
    const float sl[2] = {p.scale_log2, p.scale_log2};
    const bool poll = p.page_shift < 5;  // stages of several boxes (see wait_stage_mode)
    int lim[2] = {0, 0};
    bool ok = true;
    const int grp = warp / DSPLIT;         // consumer group: stage j of every unit goes to group j mod NP
    const int half = warp - grp * DSPLIT;  // which DH columns of O this warp accumulates
    static_assert(DSPLIT == 1 || !Lay::BOXMAJ, "warp pairs split V by regions of the region-major layout");
    const uint32_t v_half = static_cast<uint32_t>(half * (DH / 64) * G::REGION_BYTES);
    for (int i = grp;; i += NP) {
        const int s = i % S;
        if (!wait_stage_mode<S>(full, i, poll)) {
            ok = false;
            break;
        }
        const int t = tag[s];
        if (t < 0) break;  // no unit left
        const int cb = t & 1, j = t >> 1;
        const int tok_begin = um[cb].tok_begin, tok_end = um[cb].tok_end, n_pad = um[cb].n_pad;
        const uint16_t* q_s = qbuf + cb * RC * D;
        if (j < NP) {  // this group's first stage of the unit
            // the unit's query rows land with its stage 0 (stage i - j); that barrier is
            // still in this phase: its next use, stage i - j + 2S, cannot be issued before
            // this warp releases stage i
            if (j > 0 && !wait_stage_mode<S>(full, i - j, poll)) {
                ok = false;
                break;
            }
            cw.reset();
            cw.load_q(q_s);
            const int L = um[cb].L, row0 = um[cb].row0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int qi = (row0 + g + 8 * h) / p.group;
                lim[h] = p.causal ? (L - p.q_len + qi) : (L - 1);
            }
        }
        const int t0 = tok_begin + j * kStageTokens;
        const int nv = max(0, min(kStageTokens, tok_end - t0));
        uint8_t* st = stages + s * G::STAGE_BYTES;
        if (nv > 0) cw.stage(q_s, st, nv, min(nv, lim[0] - t0 + 1), min(nv, lim[1] - t0 + 1), sl, v_half);
        if (j < n_pad - NP) {
            if (nv > 0 && nv < kStageTokens) fence_proxy_async_shared();  // zeroed tail before the next TMA write
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
            continue;
        }
        // This group's last stage of the unit: its state goes into this (kept) slot.
        cw.finish_l();
        float2* ml = mls + cb * NP * RC;
        if (tq == 0 && half == 0) {  // the warps of a group hold the same m and l
            ml[grp * RC + g] = make_float2(cw.mrow[0], cw.lrow[0]);
            ml[grp * RC + g + 8] = make_float2(cw.mrow[1], cw.lrow[1]);
        }
        float* o_s = reinterpret_cast<float*>(st + Lay::O_BASE) + half * Lay::O_HALF;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            *reinterpret_cast<float2*>(o_s + g * Lay::O_ROW + 8 * n + 2 * tq) = make_float2(cw.o[n][0], cw.o[n][1]);
            *reinterpret_cast<float2*>(o_s + (g + 8) * Lay::O_ROW + 8 * n + 2 * tq) =
                make_float2(cw.o[n][2], cw.o[n][3]);
        }
        fence_proxy_async_shared();  // these generic writes precede the slot's next TMA fill
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(&cnt[cb], 1) == NW - 1;
            if (last) __threadfence_block();
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) continue;
        // The last warp of the unit: merge, store, release the kept slots and the buffer.
        const int kept0 = i - j + n_pad - NP;  // ring index of group 0's last stage of the unit
        const float* o_w[NP];
#pragma unroll
        for (int w = 0; w < NP; ++w)
            o_w[w] = reinterpret_cast<const float*>(stages + ((kept0 + w) % S) * G::STAGE_BYTES + Lay::O_BASE);
        const UnitMeta u = um[cb];
        merge_unit<D, NP, RC, DH, Lay::O_ROW, Lay::O_HALF>(p, u, ml, o_w, lane);
        __syncwarp();
        if (lane == 0) {
            cnt[cb] = 0;
#pragma unroll
            for (int w = 0; w < NP; ++w)
                for (int x = 0; x < DSPLIT; ++x) mbar_arrive(smem_addr(&empty[(kept0 + w) % S]));
            mbar_arrive(smem_addr(&qfree[cb]));
        }
    }
    if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);
}

template <int D, bool BF16, bool BM>
cudaError_t launch_split_mma_persist_one(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                         dim3 grid, cudaStream_t stream, bool launch) {
    using Lay = PersistLayout<D, BM>;
    static unsigned long long attr_done = 0;  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(split_mma_persist_kernel<D, BF16, BM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Lay::SMEM);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&attr_done, 1ull << dev, __ATOMIC_RELEASE);
    }
    if (!launch) return cudaSuccess;
    // A programmatic dependent of the previous kernel in the stream: its CTAs may become
    // resident while that kernel finishes (the producer waits for it before any input).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Lay::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Lay::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_mma_persist_kernel<D, BF16, BM>, p, tk, tv);
}

}  // namespace fdec
