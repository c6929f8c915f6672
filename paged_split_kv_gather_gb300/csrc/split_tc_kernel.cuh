// split_tc_kernel.cuh -- the dense-query split kernel on 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), for more than 16 query rows
// (q_len x group: speculative-decode and prefill chunks), head_dim D = 64, 128,
// 192 or 256.
//
// One CTA: one work item (a run of 64-token blocks) x one KV head x NT tiles of
// 128 query rows (rows = q positions x heads of the group, flattened).  The NT
// tiles share every staged K/V block (NT = 2 needs 2 x (128 + D) tensor-memory
// columns: head_dim up to 128).  With a causal mask the item's token range is
// clipped to the last token any row of the CTA can see.  Warps:
//   warp 0      TMA producer: 64-token K/V stages (the shared producer).
//   warp 1      MMA issuer (one lane), per tile t and block j:
//                 S_t  = Q_t K^T            M 128 rows, N 64 tokens, K = D dims  (D / 16 MMAs)
//                 O_t += P_t,hi V + P_t,lo V  M 128, N = D dims, K 64 tokens      (2 x 4 MMAs)
//               Q and K are K-major and V MN-major, 128B-swizzled in shared
//               memory; S_t, P_t and O_t live in tensor memory.  One tile: S_t has
//               two buffers (block parity), and S_t of block j + 1 is issued before
//               the P V products of block j wait for P_t, so it overlaps this
//               block's softmax.  Two tiles: Q_t is copied into tensor memory too
//               and is the A operand of Q K^T (so those products read only K from
//               shared memory), and each tile has one S_t buffer, S_t(j + 1) issued
//               after the P V products of block j; the tiles take turns with the
//               tensor cores.  P_t overwrites the S_t it came from (hi in the first
//               32 columns, lo in the next 32, two 16-bit values per column) and is
//               the A operand of the P V products, so P never goes through shared
//               memory.
//   warps 2+4t..5+4t  softmax warpgroup of tile t, thread = row = tensor-memory
//               lane: load the row of S, mask, row max in registers, exp2, and the
//               row of P stored back into tensor memory, per 16-token slice: one
//               f16 value when the slice's V is f16 (11 significant bits, one P V
//               product), else a bf16 high part and residual (~15 bits, two
//               products).  The lazy rescale of the row of O (only when the max
//               grew by more than 8 in log2 units; warp-uniform) first waits for
//               the previous block's P V products.  After the last block: O, l,
//               m -> one partial of the split, or out / lse.
//   warps 2+4NT..5+4NT  (bf16 caches) V conversion: warp w rewrites token slice
//               w of each stage as f16 in place when that is exact enough (its
//               largest |v| is 0 or in [2^-10, 65504]) and records the slice's mode;
//               the P V products of a stage wait for them (conv_full).
// Synchronisation: stage full / empty mbarriers (TMA / commit of the P V MMAs),
// and per tile s_full[2] (commit of the QK MMAs, per S buffer), p_full[2] (the
// four softmax warps, per buffer), o_done (commit of the P V MMAs) and o_final
// (commit after the last block's P V MMAs).  Every wait is bounded.  Ordering of the S / P buffers: the tensor cores execute
// one thread's MMAs in issue order, so S_t(j + 2), issued after the P V
// products of block j, overwrites P_t(j) only after they have read it.
#pragma once

#include "split_common.cuh"
#include "tc_common.cuh"

namespace fdec {

template <int NT, int D_, bool CONV = false>
struct TcLayout {
    static constexpr int D = D_;
    static constexpr int TM = 128;                 // query rows per tile
    static constexpr int ROWS = NT * TM;           // query rows per CTA
    static constexpr int TOK = 64;                 // tokens per stage / S tile
    using G = StageGeom<D, TOK>;
    static constexpr int Q_BYTES = TM * D * 2;     // per tile: D/64 regions x 128 rows x 128 B
    static constexpr int BAR_BYTES = 512;
    static constexpr int CONV_WARPS = CONV ? 4 : 0;  // V-slice conversion warps (bf16 caches)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_STAGES = OFF_Q + NT * Q_BYTES;
    static constexpr int S_FIT = (232448 - 1024 - BAR_BYTES - NT * Q_BYTES) / G::STAGE_BYTES;
    static constexpr int S = S_FIT > 6 ? 6 : S_FIT;  // stages
    static constexpr int OFF_BARS = OFF_STAGES + S * G::STAGE_BYTES;
    static constexpr int NBARS = 3 * S + 6 * NT + 1 + (CONV ? S : 0);
    static constexpr int SMEM = OFF_BARS + BAR_BYTES + 1024;  // + alignment slack
    static constexpr int THREADS = (2 + 4 * NT + CONV_WARPS) * 32;
    // Two tiles per CTA: Q in tensor memory as the A operand of Q K^T (the N = 64
    // products then read only K from shared memory, so they run at the full rate) and
    // one S / P buffer per tile.  One tile: Q in shared memory, two S / P buffers.
    static constexpr bool QTM = NT == 2;
    static constexpr int NSB = QTM ? 1 : 2;        // S / P buffers per tile
    // tensor memory per tile t (base TILE_COLS t): S / P buffers at +0 (and +64), O (D
    // columns) after them, then (QTM) Q as D / 2 columns of two 16-bit values
    static constexpr uint32_t O_COL = 64 * NSB;
    static constexpr uint32_t Q_COL = O_COL + D;
    static constexpr uint32_t TILE_COLS = Q_COL + (QTM ? D / 2 : 0);
    static constexpr uint32_t TMEM_COLS = NT * TILE_COLS <= 256 ? 256u : 512u;
    static_assert(NT * TILE_COLS <= 512, "tensor memory: S/P buffers, O (and Q) per tile");
    static_assert(S >= 2, "stages");
    static_assert(SMEM <= 232448, "shared memory");
    static_assert(NBARS * 8 + 8 + 4 * S <= BAR_BYTES, "barriers, tensor-memory address, slice modes");
    static_assert(NT == 1 || NT == 2, "tiles per CTA");
    static_assert(D % 64 == 0 && D <= 256, "P V is one MMA of N = head_dim (at most 256)");
};

// Byte offset of 16-byte chunk `chunk` (0..7) of row r in a 128B-swizzled region of 128-byte rows.
__device__ __forceinline__ uint32_t sw128_offset(int r, int chunk) {
    return static_cast<uint32_t>(r * 128 + (((chunk ^ r) & 7) << 4));
}

// (y & 0xffff0000) | (x >> 16): the bf16 truncations of x (low half) and y (high
// half) in one word, with a shift and a LOP3.  Written in PTX so that it stays
// those two instructions: byte-permute and float -> 16-bit conversion
// instructions issued by the softmax warps slow the tensor cores' MMA stream
// (measured on sm_103a), while shifts and logic ops do not.
__device__ __forceinline__ uint32_t pack_upper_halves(uint32_t x, uint32_t y) {
    uint32_t t, r;
    asm volatile("shr.u32 %0, %1, 16;" : "=r"(t) : "r"(x));
    asm volatile("lop3.b32 %0, %1, 0xffff0000, %2, 0xEA;" : "=r"(r) : "r"(y), "r"(t));
    return r;
}

// Per 16-bit half, the larger unsigned value.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float x, float y) {
    if constexpr (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __half2 h = __floats2half2_rn(x, y);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

template <int NT, int D, bool BF16>
__global__ void __launch_bounds__(TcLayout<NT, D, BF16>::THREADS, 1)
split_tc_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv) {
    constexpr bool CONV = BF16;  // bf16 caches: V slices converted to f16 where exact
    using Lay = TcLayout<NT, D, CONV>;
    using G = typename Lay::G;
    constexpr int S = Lay::S;
    constexpr int TOK = Lay::TOK;
    constexpr uint32_t TC = Lay::TILE_COLS;
    constexpr float kLn2 = 0.69314718055994530942f;
    constexpr float kLazyRescale = 8.f;
    // P is scaled by 2^kPShift so that small p stay normal in f16; l carries the
    // same factor and the stored max drops by kPShift.  For a 16-token slice whose V
    // is f16 (an f16 cache, or a bf16 slice the conversion warps rewrote) P is one
    // f16 value per token (11 significant bits) and P V one product.  For a bf16
    // slice P = hi + lo, both bf16 (hi = p truncated to bf16, lo = the residual
    // truncated), ~15 significant bits, and P V two products; the split uses shifts,
    // logic ops and FMAs only (see pack_upper_halves).
    constexpr bool kSplit = BF16;
    constexpr int kParts = kSplit ? 2 : 1;
    constexpr float kPShift = 7.f;

    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* q_tiles = smem + Lay::OFF_Q;
    uint8_t* stages = smem + Lay::OFF_STAGES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::OFF_BARS);
    uint64_t* full = bars;            // 2S
    uint64_t* empty = bars + 2 * S;   // S
    uint64_t* s_full = bars + 3 * S;  // [NT][2]
    uint64_t* p_full = s_full + 2 * NT;  // [NT][2]
    uint64_t* o_done = p_full + 2 * NT;  // [NT]
    uint64_t* o_final = o_done + NT;     // [NT]
    uint64_t* mma_fin = o_final + NT;
    uint64_t* conv_full = mma_fin + 1;  // [S]: the stage's V slices are converted (bf16)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(conv_full + (CONV ? S : 0));
    uint32_t* vmode = tmem_slot + 2;    // [S]: byte w = 1 when V slice w of the stage is f16

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Row tiles vary fastest over the launch, so the CTAs resident at one time
    // share a few (sequence, KV head) streams and re-read them from L2.
    const unsigned lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const int cta_tile = static_cast<int>(lin % gridDim.z);
    const int kvh = static_cast<int>((lin / gridDim.z) % gridDim.y);
    const WorkItem it = p.items[lin / (gridDim.z * gridDim.y)];
    const int b = it.seq;
    const int row0 = cta_tile * Lay::ROWS;

    // Launched as a programmatic dependent of the kernel before it in the stream: read
    // and write nothing but plan data before that kernel has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    ItemRange ir = item_range<TOK>(p, it);
    if (p.causal) {  // no row of this CTA sees past L - Q + (its last q position)
        const int last_row = min(row0 + Lay::ROWS, p.rows) - 1;
        const int lim_max = ir.L - p.q_len + last_row / p.group;
        ir.tok_end = min(ir.tok_end, lim_max + 1);
        ir.n_stage = ir.tok_end > ir.tok_begin ? (ir.tok_end - ir.tok_begin + TOK - 1) / TOK : 0;
    }
    const int n_tiles = ir.n_stage;
    const bool tma_mode = p.page_shift >= 3;

    if (threadIdx.x == 0) {
        init_stage_barriers<S>(full, empty, tma_mode);
#pragma unroll
        for (int i = 0; i < 2 * NT; ++i) {
            mbar_init(smem_addr(&s_full[i]), 1);
            mbar_init(smem_addr(&p_full[i]), 4);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            mbar_init(smem_addr(&o_done[t]), 1);
            mbar_init(smem_addr(&o_final[t]), 1);
        }
        mbar_init(smem_addr(mma_fin), 1);
        if constexpr (CONV) {
#pragma unroll
            for (int x = 0; x < S; ++x) mbar_init(smem_addr(&conv_full[x]), 4);  // one arrival per conversion warp
        }
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0 && tma_mode) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), Lay::TMEM_COLS);
        tmem_relinquish();
    }
    // Q tiles: K-major, 128B-swizzled (two 64-dim regions per tile); absent rows are zero.
    {
        QChunks<Lay::ROWS, D, Lay::THREADS> qc;
        qc.load(p, b, kvh, row0, threadIdx.x);
#pragma unroll
        for (int i = 0; i < qc.PER; ++i) {
            const int idx = qc.chunk(threadIdx.x, i);
            if (idx < qc.CH) {
                const int r = idx / (D / 8);
                const int c = idx - r * (D / 8);  // 16-byte chunk of the row
                const int t = r / Lay::TM, rt = r - t * Lay::TM;
                *reinterpret_cast<uint4*>(q_tiles + t * Lay::Q_BYTES + (c >> 3) * (Lay::TM * 128) +
                                          sw128_offset(rt, c & 7)) = qc.v[i];
            }
        }
    }
    fence_proxy_async_shared();  // generic writes of Q, read by the tensor cores
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if constexpr (Lay::QTM) {
        // Q into tensor memory: softmax thread r copies row r of its tile (lane r; dims
        // 2k, 2k + 1 in column Q_COL + k, the lower dim in the low half).
        if (warp >= 2 && warp < 2 + 4 * NT) {
            const int t = (warp - 2) >> 2, wq = warp & 3, r = wq * 32 + lane;
            const uint8_t* qt = q_tiles + t * Lay::Q_BYTES;
            const uint32_t dst = tmem + TC * t + (static_cast<uint32_t>(wq * 32) << 16) + Lay::Q_COL;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {  // one 64-dim region: 32 columns
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4*>(qt + h * (Lay::TM * 128) + sw128_offset(r, c));
                    w[4 * c] = v.x;
                    w[4 * c + 1] = v.y;
                    w[4 * c + 2] = v.z;
                    w[4 * c + 3] = v.w;
                }
                tmem_st32_u(dst + 32 * h, w);
            }
            tmem_wait_st();
        }
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        produce_stages<D, S, TOK>(p, &tmk, &tmv, full, empty, stages, b, kvh, ir, tma_mode);
        if (lane == 0) report_item_range(p, ir);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_tiles > 0) {
            bool ok = true;
            const uint32_t i_qk = idesc_f16(128, TOK, BF16, false, false);
            const uint32_t i_pv = idesc_f16(128, D, BF16, false, true);
            const uint32_t i_pv16 = idesc_f16(128, D, false, false, true);  // f16 P times an f16 V slice
            // Descriptors are built once; a byte offset x within shared memory is
            // x >> 4 added to the start-address field (the sum stays below 2^14).
            const uint64_t qd0 = smem_desc_sw128(smem_addr(q_tiles), 16, 1024);
            const uint64_t kd0 = smem_desc_sw128(smem_addr(stages), 16, 1024);
            const uint64_t vd0 = smem_desc_sw128(smem_addr(stages + G::HALF_BYTES), G::REGION_BYTES, 1024);
            constexpr uint32_t kQTile = Lay::Q_BYTES >> 4, kQRegion = (Lay::TM * 128) >> 4;
            constexpr uint32_t kStage = G::STAGE_BYTES >> 4, kKRegion = G::REGION_BYTES >> 4;
            auto issue_qk = [&](int t, int slot, int buf) {
                const uint64_t qd = qd0 + t * kQTile;
                const uint64_t kd = kd0 + static_cast<uint32_t>(slot) * kStage;
                const uint32_t d = tmem + TC * t + 64 * buf;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    if constexpr (Lay::QTM)  // A = Q from tensor memory: 16 dims = 8 columns per step
                        tc_mma_f16_ts(d, tmem + TC * t + Lay::Q_COL + 8 * ks, kd + (ks >> 2) * kKRegion + (ks & 3) * 2,
                                      i_qk, ks > 0);
                    else
                        tc_mma_f16(d, qd + (ks >> 2) * kQRegion + (ks & 3) * 2, kd + (ks >> 2) * kKRegion + (ks & 3) * 2,
                                   i_qk, ks > 0);
                }
                tc_commit(smem_addr(&s_full[2 * t + buf]));
            };
            // P V of one block, 16 tokens (128 rows of V) per step: one f16 product for a
            // slice whose mode bit is set, else one product per part of P.
            auto issue_pv = [&](int t, int slot, int buf, bool acc, uint32_t modes) {
                const uint64_t vd = vd0 + static_cast<uint32_t>(slot) * kStage;
                const uint32_t p_tm = tmem + TC * t + 64 * buf;
                const uint32_t o_tm = tmem + TC * t + Lay::O_COL;
                bool a = acc;
                if (CONV && modes == 0x01010101u) {
#pragma unroll
                    for (int ks = 0; ks < TOK / 16; ++ks) tc_mma_f16_ts(o_tm, p_tm + 8 * ks, vd + ks * 128, i_pv16, ks > 0 || acc);
                    tc_commit(smem_addr(&o_done[t]));
                    return;
                }
#pragma unroll
                for (int ks = 0; ks < TOK / 16; ++ks) {
                    if (CONV && ((modes >> (8 * ks)) & 1u)) {
                        tc_mma_f16_ts(o_tm, p_tm + 8 * ks, vd + ks * 128, i_pv16, a);
                        a = true;
                    } else {
#pragma unroll
                        for (int part = 0; part < kParts; ++part) {
                            tc_mma_f16_ts(o_tm, p_tm + 32 * part + 8 * ks, vd + ks * 128, i_pv, a);
                            a = true;
                        }
                    }
                }
                tc_commit(smem_addr(&o_done[t]));
            };
            // Stage j landed?  (this thread is the only consumer of the stages, in order)
            auto wait_full = [&](int j) { return mbar_wait_bounded(smem_addr(&full[j % (2 * S)]), (j / (2 * S)) & 1); };
            ok = wait_full(0);
            if (ok) {
                tc_fence_after_sync();
#pragma unroll
                for (int t = 0; t < NT; ++t) issue_qk(t, 0, 0);
            }
            int slot = 0;  // stage slot of block j
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int next_slot = slot + 1 == S ? 0 : slot + 1;
                if constexpr (Lay::QTM) {
                    // One S / P buffer per tile: S_t(j + 1) is issued right after the P V
                    // products of block j, which read P_t(j) from that buffer first (in-order
                    // execution); the commit on s_full_t then also covers those products, so a
                    // row of O_t may be rescaled once S_t(j + 1) has landed.
                    uint32_t modes = 0;
                    if constexpr (CONV) {
                        if (!(ok = mbar_wait_bounded(smem_addr(&conv_full[slot]), (j / S) & 1))) break;
                        modes = vmode[slot];
                    }
                    for (int t = 0; t < NT; ++t) {
                        if (!(ok = mbar_wait_bounded(smem_addr(&p_full[2 * t]), j & 1))) break;
                        tc_fence_after_sync();
                        issue_pv(t, slot, 0, j > 0, modes);
                        if (j + 1 == n_tiles) {
                            tc_commit(smem_addr(&o_final[t]));
                            continue;
                        }
                        if (t == 0) {
                            if (!(ok = wait_full(j + 1))) break;
                            tc_fence_after_sync();
                        }
                        issue_qk(t, next_slot, 0);
                    }
                    if (!ok) break;
                    tc_commit(smem_addr(&empty[slot]));  // the stage is free once these MMAs completed
                    slot = next_slot;
                    continue;
                }
                if (j + 1 < n_tiles) {
                    // S_t(j + 1) goes to the other buffer, whose P_t(j - 1) the P V
                    // products issued before have consumed by then (in-order execution).
                    if (!(ok = wait_full(j + 1))) break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int t = 0; t < NT; ++t) issue_qk(t, next_slot, (j + 1) & 1);
                }
                uint32_t modes = 0;
                if constexpr (CONV) {  // the stage's V slices are final (converted or left bf16)
                    if (!(ok = mbar_wait_bounded(smem_addr(&conv_full[slot]), (j / S) & 1))) break;
                    modes = vmode[slot];
                }
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (!(ok = mbar_wait_bounded(smem_addr(&p_full[2 * t + (j & 1)]), (j >> 1) & 1))) break;
                    tc_fence_after_sync();
                    issue_pv(t, slot, j & 1, j > 0, modes);
                    if (j + 1 == n_tiles) tc_commit(smem_addr(&o_final[t]));
                }
                if (!ok) break;
                tc_commit(smem_addr(&empty[slot]));  // the stage is free once these MMAs completed
                slot = next_slot;
            }
            // Tensor memory is freed below: first let every MMA issued here complete.
            tc_commit(smem_addr(mma_fin));
            if (!mbar_wait_bounded(smem_addr(mma_fin), 0)) ok = false;
            if (!ok) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);
        }
    } else if (warp >= 2 + 4 * NT) {
        // ------------------------------------------------------------ V conversion (bf16 caches)
        // Warp w owns token slice w (rows 16w .. 16w + 15 of every V region) of each
        // stage.  When the slice's largest |v| is 0 or lies in [2^-10, 65504] it is
        // rewritten in place as f16: exact for |v| >= 2^-17, and below that rounded to
        // the f16 grid (spacing 2^-24, under 2^-14 of the slice's largest value); its
        // P V product then runs once, with an f16 P.  Otherwise (larger or only tiny
        // values, inf, NaN) the slice stays bf16 and takes the two products of P's
        // parts.  Rows past the sequence's end are zeroed either way: their P is 0,
        // and 0 x NaN would poison O.
        if constexpr (CONV) {
            const int w = warp - (2 + 4 * NT);
            constexpr int CPL = D / 16;  // 16-byte chunks per lane: 16 rows x D / 8 chunks over 32 lanes
            constexpr uint32_t kLo = 0x3a80u;  // |v| bits of 2^-10 (bf16)
            constexpr uint32_t kHi = 0x477fu;  // 65280, the largest bf16 below the f16 maximum 65504
            bool ok = true;
            for (int j = 0; j < n_tiles; ++j) {
                if (!(ok = mbar_wait_bounded(smem_addr(&full[j % (2 * S)]), (j / (2 * S)) & 1))) break;
                const int slot = j % S;
                uint8_t* vrows = stages + slot * G::STAGE_BYTES + G::HALF_BYTES;
                const int nv = min(TOK, ir.tok_end - (ir.tok_begin + j * TOK));
                uint4 x[CPL];
                uint32_t m2 = 0u;  // per 16-bit half: the largest |v| bits seen (inf and NaN above every finite value)
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    // chunk idx: 8 per 128-byte row, 16 rows per region (consecutive lanes
                    // take consecutive 16 bytes of a row: conflict-free)
                    const int idx = lane + 32 * i;
                    const int row = 16 * w + ((idx >> 3) & 15);
                    uint4* ptr = reinterpret_cast<uint4*>(vrows + (idx >> 7) * G::REGION_BYTES + row * 128 + (idx & 7) * 16);
                    x[i] = row < nv ? *ptr : make_uint4(0u, 0u, 0u, 0u);
                    m2 = max_u16x2(m2, x[i].x & 0x7fff7fffu);
                    m2 = max_u16x2(m2, x[i].y & 0x7fff7fffu);
                    m2 = max_u16x2(m2, x[i].z & 0x7fff7fffu);
                    m2 = max_u16x2(m2, x[i].w & 0x7fff7fffu);
                }
                const uint32_t wm = __reduce_max_sync(0xffffffffu, max(m2 & 0xffffu, m2 >> 16));
                const bool f16 = wm == 0u || (wm >= kLo && wm <= kHi);
#pragma unroll
                for (int i = 0; i < CPL; ++i) {
                    const int idx = lane + 32 * i;
                    const int row = 16 * w + ((idx >> 3) & 15);
                    uint4* ptr = reinterpret_cast<uint4*>(vrows + (idx >> 7) * G::REGION_BYTES + row * 128 + (idx & 7) * 16);
                    if (f16) {
                        uint32_t u[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const __half2 h = __floats2half2_rn(__uint_as_float(u[k] << 16), __uint_as_float(u[k] & 0xffff0000u));
                            u[k] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                        *ptr = make_uint4(u[0], u[1], u[2], u[3]);
                    } else if (row >= nv) {
                        *ptr = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_shared();  // read by the tensor cores
                __syncwarp();
                if (lane == 0) {
                    reinterpret_cast<uint8_t*>(&vmode[slot])[w] = f16 ? 1 : 0;
                    mbar_arrive(smem_addr(&conv_full[slot]));
                }
            }
            if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = (warp - 2) >> 2;       // tile of this warpgroup
        const int wq = warp & 3;             // tensor-memory lane quarter of this warp
        const int r = wq * 32 + lane;        // row within the tile = tensor-memory lane
        const int row = row0 + t * Lay::TM + r;
        const int qi = row / p.group;
        const int lim = p.causal ? (ir.L - p.q_len + qi) : (ir.L - 1);
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tmem_t = tmem + TC * t + lane_base;
        const uint32_t tmem_o = tmem_t + Lay::O_COL;
        const float c_log2 = p.scale_log2;
        // Every row of this warp past the CTA's query rows (a tile of few rows): its rows of
        // P are never used for a stored row (row m of O depends on row m of P alone), so the
        // warp only keeps the barriers in step.  Its issue slots go to the other warps.
        const bool idle = row0 + t * Lay::TM + wq * 32 >= p.rows;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            constexpr int NSB = Lay::NSB;
            const uint32_t buf = tmem_t + 64 * (j % NSB);
            if (!mbar_wait_bounded(smem_addr(&s_full[2 * t + (j % NSB)]), (j / NSB) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            if (idle) {
                if (!CONV && t == 0 && ir.tok_end - (ir.tok_begin + j * TOK) < TOK) {  // the tail rows, as below
                    zero_v_tail<D, TOK>(stages + (j % S) * G::STAGE_BYTES, ir.tok_end - (ir.tok_begin + j * TOK),
                                        threadIdx.x - 64, 128);
                    fence_proxy_async_shared();
                    named_barrier(2, 128);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&p_full[2 * t + (j % NSB)]));
                continue;
            }
            float sv[TOK];
            {
                float a[32];
                tmem_ld32(buf + 0, a);
#pragma unroll
                for (int c = 0; c < 32; ++c) sv[c] = a[c];
                tmem_ld32(buf + 32, a);
#pragma unroll
                for (int c = 0; c < 32; ++c) sv[32 + c] = a[c];
                tmem_wait_ld();
            }

            const int t0 = ir.tok_begin + j * TOK;
            const int nv = min(TOK, ir.tok_end - t0);
            const int vis = min(nv, lim - t0 + 1);  // tokens of this block the row may see
            // Row max of the logits in log2 units.  Blocks that some row of the
            // warp sees only in part take the masked form; the others scale the
            // raw maximum (minimum for a negative scale) and fold the scale into
            // the exponent below.  Eight independent chains, then a tree.
            float mx, cs;
            if (__any_sync(0xffffffffu, vis < TOK)) {
#pragma unroll
                for (int c = 0; c < TOK; ++c) sv[c] = c < vis ? sv[c] * c_log2 : -INFINITY;
                float q8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) q8[k] = sv[k];
#pragma unroll
                for (int c = 8; c < TOK; ++c) q8[c & 7] = fmaxf(q8[c & 7], sv[c]);
                mx = fmaxf(fmaxf(fmaxf(q8[0], q8[1]), fmaxf(q8[2], q8[3])), fmaxf(fmaxf(q8[4], q8[5]), fmaxf(q8[6], q8[7])));
                cs = 1.f;
            } else {
                float q8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) q8[k] = sv[k];
                if (c_log2 >= 0.f) {
#pragma unroll
                    for (int c = 8; c < TOK; ++c) q8[c & 7] = fmaxf(q8[c & 7], sv[c]);
                    mx = fmaxf(fmaxf(fmaxf(q8[0], q8[1]), fmaxf(q8[2], q8[3])), fmaxf(fmaxf(q8[4], q8[5]), fmaxf(q8[6], q8[7])));
                } else {
#pragma unroll
                    for (int c = 8; c < TOK; ++c) q8[c & 7] = fminf(q8[c & 7], sv[c]);
                    mx = fminf(fminf(fminf(q8[0], q8[1]), fminf(q8[2], q8[3])), fminf(fminf(q8[4], q8[5]), fminf(q8[6], q8[7])));
                }
                mx *= c_log2;
                cs = c_log2;
            }
            const bool grow = mx > m + kLazyRescale;
            const bool rescale = __any_sync(0xffffffffu, grow);
            // 1 for rows that keep their max (also while it is still -inf), 0 when m was -inf
            const float alpha = grow ? exp2_approx(m - mx) : 1.f;
            if (grow) m = mx;
            if (rescale && j > 0) {
                // O_t holds blocks 0 .. j-1: wait for the last of their P V products,
                // then rescale this row of O_t in tensor memory.  o_done_t is in
                // phase j - 1 or j here: S_t(j) has landed, so the products of
                // block j - 2 (issued before it) have completed, and those of
                // block j wait for this warp's P_t(j).  The parity test is exact.
                // (One S / P buffer: S_t(j) was committed after the products of block
                // j - 1, so they have completed.)
                if (!Lay::QTM && !mbar_wait_bounded(smem_addr(&o_done[t]), (j - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 16) {  // 16 columns at a time: few registers beside the row of S
                    float a[16];
                    tmem_ld16(tmem_o + c0, a);
                    tmem_wait_ld();
                    uint32_t u[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) u[c] = __float_as_uint(a[c] * alpha);
                    tmem_st16_u(tmem_o + c0, u);
                }
                tmem_wait_st();
            }
            const float mu = m == -INFINITY ? 0.f : m;
            // Which 16-token V slices of this block are f16 (bf16 caches: set by the
            // conversion warps; the stage's slot is not refilled before P_t(j) is consumed).
            uint32_t modes = 0x01010101u;
            if constexpr (CONV) {
                if (!mbar_wait_bounded(smem_addr(&conv_full[j % S]), (j / S) & 1)) {
                    ok = false;
                    break;
                }
                modes = vmode[j % S];
            }
            // p = exp2(s * cs - mu), its row sum, and P packed per slice: one f16 value
            // per token, or (bf16 slices) the bf16 high part and residual.  P_t(j) goes
            // over S_t(j) (f16 values or high parts in columns 0..31, residuals in
            // 32..63), 32 tokens at a time: the row of S is already in registers.
            float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            const float2 cs2 = make_float2(cs, cs), nmu2 = make_float2(kPShift - mu, kPShift - mu);
            if (modes == 0x01010101u) {
                // every slice f16 (the common case): one straight-line pass, no per-slice branches
#pragma unroll
                for (int h = 0; h < TOK / 32; ++h) {
                    uint32_t hv[16];
#pragma unroll
                    for (int c = 32 * h; c < 32 * h + 32; c += 2) {
                        const float2 z = __ffma2_rn(make_float2(sv[c], sv[c + 1]), cs2, nmu2);
                        const float2 e = make_float2(exp2_approx(z.x), exp2_approx(z.y));
                        ls[(c >> 1) & 3] = __fadd2_rn(ls[(c >> 1) & 3], e);
                        hv[(c - 32 * h) / 2] = pack2<false>(e.x, e.y);
                    }
                    tmem_st16_u(buf + 16 * h, hv);
                }
            } else {
#pragma unroll
            for (int h = 0; h < TOK / 32; ++h) {
                uint32_t hi[16], lo[kSplit ? 16 : 1];
#pragma unroll
                for (int ks = 2 * h; ks < 2 * h + 2; ++ks) {
                    const bool half_p = (modes >> (8 * ks)) & 1u;
#pragma unroll
                    for (int c = 16 * ks; c < 16 * ks + 16; c += 2) {
                        const int x = (c - 32 * h) / 2;  // word of this half
                        const float2 z = __ffma2_rn(make_float2(sv[c], sv[c + 1]), cs2, nmu2);
                        const float2 e = make_float2(exp2_approx(z.x), exp2_approx(z.y));
                        ls[(c >> 1) & 3] = __fadd2_rn(ls[(c >> 1) & 3], e);
                        if (!kSplit || half_p) {
                            hi[x] = pack2<false>(e.x, e.y);
                            if constexpr (kSplit) lo[x] = 0u;  // not read: this slice takes one product
                        } else {
                            const uint32_t bx = __float_as_uint(e.x), by = __float_as_uint(e.y);
                            hi[x] = pack_upper_halves(bx, by);  // truncation to bf16
                            const float2 hf = make_float2(__uint_as_float(bx & 0xffff0000u),
                                                          __uint_as_float(by & 0xffff0000u));
                            const float2 rs = __ffma2_rn(hf, make_float2(-1.f, -1.f), e);  // exact residual
                            if constexpr (kSplit) lo[x] = pack_upper_halves(__float_as_uint(rs.x), __float_as_uint(rs.y));
                        }
                    }
                }
                tmem_st16_u(buf + 16 * h, hi);
                if constexpr (kSplit) {
                    if (((modes >> (16 * h)) & 0x0101u) != 0x0101u) tmem_st16_u(buf + 32 + 16 * h, lo);
                }
            }
            }
            const float2 l01 = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
            l = l * alpha + (l01.x + l01.y);
            tmem_wait_st();
            if (!CONV && t == 0 && nv < TOK) {
                // A partial stage: zero V rows past the sequence end (0 * NaN would
                // poison O).  Tile 0's P V products come first for every stage.
                zero_v_tail<D, TOK>(stages + (j % S) * G::STAGE_BYTES, nv, threadIdx.x - 64, 128);
                fence_proxy_async_shared();  // read by the tensor cores
                named_barrier(2, 128);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&p_full[2 * t + (j % NSB)]));
        }
        // The last P V products: o_done_t may be anywhere from phase n - 2 to n
        // here, so the MMA thread signals them on a barrier of their own.
        if (ok && n_tiles > 0 && !mbar_wait_bounded(smem_addr(&o_final[t]), 0)) ok = false;
        tc_fence_after_sync();
        if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);

        const int h = kvh * p.group + (row - qi * p.group);
        const int64_t orow = static_cast<int64_t>(b * p.q_len + qi) * p.hq + h;
        const int64_t prow = (static_cast<int64_t>(it.slot) * p.hk + kvh) * p.rows + row;
        if (n_tiles > 0 && ok) {
            // O row from tensor memory -> partial (unnormalised) or final output
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float a[32];
                tmem_ld32(tmem_o + c0, a);
                tmem_wait_ld();
                if (row < p.rows) {
                    float* dst = it.slot < 0 ? p.out + orow * D + c0 : p.part_o + prow * D + c0;
                    const float f = (it.slot < 0 ? inv : 1.f) * p.v_scale;
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4*>(dst + c) =
                            make_float4(a[c] * f, a[c + 1] * f, a[c + 2] * f, a[c + 3] * f);
                }
            }
        } else {
            // nothing visible (or a failed wait): an empty state
            if (row < p.rows) {
                float* dst = it.slot < 0 ? p.out + orow * D : p.part_o + prow * D;
                for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            m = -INFINITY;
            l = 0.f;
        }
        if (row < p.rows) {
            if (it.slot < 0) {
                if (p.lse != nullptr) p.lse[orow] = l > 0.f ? (m - kPShift + log2f(l)) * kLn2 : -INFINITY;
            } else {
                p.part_ml[prow] = make_float2(l > 0.f ? m - kPShift : -INFINITY, l);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, Lay::TMEM_COLS);
    }
}

template <int NT, int D, bool BF16>
cudaError_t launch_split_tc_one(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                                cudaStream_t stream, bool launch) {
    static unsigned long long attr_done = 0;  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(split_tc_kernel<NT, D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcLayout<NT, D, BF16>::SMEM);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&attr_done, 1ull << dev, __ATOMIC_RELEASE);
    }
    if (!launch) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(TcLayout<NT, D, BF16>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = TcLayout<NT, D, BF16>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait in the kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_tc_kernel<NT, D, BF16>, p, tk, tv);
}

}  // namespace fdec
