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
//
// Quantised caches (KV8: K and V stored as 8-bit E4M3 codes, head_dim 128 and
// 256): the producer stages the codes (half the bytes of a 16-bit cache) and the
// consumers build f16 MMA fragments straight from them (every E4M3 value is
// exact in f16; one hardware conversion per pair of codes):
//   K: ldmatrix on the code rows hands lane l four consecutive codes of token
//      l / 4 (dims 16c + 4 (l % 4) .. + 3 of chunk c).  The k order inside each
//      16-dim step is permuted so that these are exactly the lane's B fragment
//      (k slots 2t, 2t+1 <- dims 4t, 4t+1 and 2t+8, 2t+9 <- 4t+2, 4t+3), and Q's A
//      fragments are read from shared memory in the same order.  A dot product
//      does not depend on the order of its terms.
//   V: ldmatrix.trans on the code rows hands lane l the codes of tokens 2t, 2t+1
//      for dims 2g, 2g+1 (g = l / 4); one byte permutation pairs them by dim, so
//      each register yields the B fragments of two n-tiles: the even dims and the
//      odd dims of a 16-dim chunk.  The epilogue puts O's columns back in order.
// A bf16 query is brought to f16 by scaling each query row by a power of two
// that puts its largest magnitude in f16's top binade [2^14, 2^15): exact for
// every element within 2^38 of the row's largest, and the factor is taken back
// out of the row's logit scale.  P is one f16 value scaled by 2^7.  The cache's
// k_scale is folded into the logit scale and v_scale into the epilogue.
#pragma once

#include <type_traits>

#include <cuda_fp8.h>

#include "split_common.cuh"

namespace fdec {

template <int D, bool KV8 = false, bool Q8 = false>
struct MmaLayout {
    using G = StageGeom<D>;                                   // 16-bit tile: what the consumers read
    using GS = StageGeom<D, kStageTokens, KV8 ? 1 : 2>;       // what the producer stages
    static constexpr int RC = 16;                 // query rows per M tile
    static constexpr int BAR_BYTES = 512;
    static constexpr int Q_BYTES = RC * D * 2;    // 16-bit q rows
    static constexpr int ALIGN_SLACK = 1024;
    // Two CTAs per SM (measured: 103 us against 131 us with one CTA of 7
    // consumers for 537 MB at 262144 tokens): each CTA gets half the shared
    // memory and four warps (3 consumers + the producer), 255 registers each.
    // head_dim 256 fits three stages and two consumers per CTA; head_dim 512
    // runs one CTA per SM (stages of 64 KB).
    static constexpr int CTAS_PER_SM = (KV8 && !Q8 && D <= 128) ? 3 : (D <= 256 ? 2 : 1);
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
    static constexpr int NP_MAX = 3;
    static constexpr int FIXED = BAR_BYTES + Q_BYTES + ALIGN_SLACK;
    // q8_0 caches: each slot also holds its tokens' K and V block-scale rows
    // (head_dim / 32 binary16 values each), after the S stages.
    static constexpr int SCB = Q8 ? D / 16 : 0;              // bytes of one token's scale row
    static constexpr int SC_STAGE = 2 * kStageTokens * SCB;  // per slot: K rows, then V rows
    static constexpr int S_FIT = (BUDGET - FIXED) / (GS::STAGE_BYTES + SC_STAGE);
    static constexpr int S = S_FIT > 16 ? 16 : S_FIT;
    static constexpr int NP = (S - 1) < NP_MAX ? (S - 1) : NP_MAX;  // consumer groups (stages in flight at once)
    static constexpr int NW = NP * DSPLIT;                 // consumer warps
    static constexpr int THREADS = (NW + 1) * 32;
    static constexpr int SMEM = FIXED + S * (GS::STAGE_BYTES + SC_STAGE);
    static_assert(!Q8 || KV8, "q8_0 codes are staged as bytes");
    static_assert(S >= NP + 1, "stage ring too small");
    static_assert(!KV8 || DSPLIT == 1, "E4M3 caches: one warp per stage");
    // Pages smaller than a stage land one box per page (all regions; see produce_stages)
    // except at head_dim 512 over 16-bit caches, whose warp pairs split each stage's V by
    // regions.
    static constexpr bool BOXMAJ = DSPLIT == 1;
    static constexpr int QMAX_OFFSET = BAR_BYTES - RC * 4;  // E4M3 caches: query row maxima
    static_assert(3 * S * 8 <= QMAX_OFFSET, "barrier area too small");
    static_assert(NP * RC * (D + 2) * 4 <= S * GS::STAGE_BYTES, "merge scratch must fit the stage area");
};

// Four E4M3 codes (w's bytes, lowest first) -> two packed f16 pairs (exact; the
// lower code of each pair lands in the lower half).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& p01, uint32_t& p23) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(p01), "=r"(p23)
        : "r"(w));
}

// Four signed 8-bit codes (w's bytes, lowest first) -> two packed f16 pairs, exact:
// the f16 with bits 0x6400 | u is 1024 + u for a byte u, so code c (u = c + 128,
// the byte with its top bit flipped) is that value minus 1152.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& p01, uint32_t& p23) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __half2half2(__ushort_as_half(static_cast<unsigned short>(0x6480u)));  // 1152
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u), b = __byte_perm(u, 0x64646464u, 0x4342u);
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    p01 = *reinterpret_cast<const uint32_t*>(&ha);
    p23 = *reinterpret_cast<const uint32_t*>(&hb);
}

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

// (x, y) rounded to a packed f16 pair, x in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float x, float y) {
    const __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<const uint32_t*>(&h);
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

// A bf16 query row with largest magnitude bits `mbits` (bf16 pattern without the
// sign) is scaled by 2^sh, sh = 14 - floor(log2 max), so that the largest lands in
// [2^14, 2^15) (f16's top binade); sh is kept in [-126, 126] so 2^sh and 2^-sh are
// normal floats.  forward: 2^sh (applied to q), else 2^-sh (applied to its logits).
__device__ __forceinline__ float q_row_factor(uint32_t mbits, bool forward) {
    int sh = 0;
    if (mbits != 0) sh = 14 - (static_cast<int>((mbits >> 7) & 0xFF) - 127);
    sh = max(-126, min(126, sh));
    return __int_as_float((127 + (forward ? sh : -sh)) << 23);
}

// q8_0: the NB binary16 block scales of tokens t and t + 1 (rows of NB values, consecutive
// in shared memory) as NB 32-bit words: token t's in words 0 .. NB/2 - 1, t + 1's after.
template <int NB>
__device__ __forceinline__ void load_scale_pair(const __half* rows, int t, uint32_t (&w)[NB]) {
    static_assert(NB % 4 == 0, "two rows of NB binary16 values: whole 16-byte chunks");
    const uint4* src = reinterpret_cast<const uint4*>(rows + t * NB);
#pragma unroll
    for (int i = 0; i < NB / 4; ++i) {
        const uint4 x = src[i];
        w[4 * i] = x.x;
        w[4 * i + 1] = x.y;
        w[4 * i + 2] = x.z;
        w[4 * i + 3] = x.w;
    }
}

// Scale of block blk of the first (u = 0) or second (u = 1) token of a pair from load_scale_pair.
template <int NB>
__device__ __forceinline__ float pair_scale(const uint32_t (&w)[NB], int u, int blk) {
    const uint32_t word = w[u * (NB / 2) + (blk >> 1)];
    return __half2float(__ushort_as_half(static_cast<unsigned short>((blk & 1) ? (word >> 16) : (word & 0xFFFFu))));
}

// One consumer warp of the tensor-core split kernels: its lane addressing into
// the swizzled stages, its query fragments, its running state (O accumulators
// of this warp's DH columns; row max m and sum l of rows g and g + 8, in log2
// units) and the work of one 32-token stage.
// BM: the stages are box-major (see stage_row_offset) with boxes of fewer rows than a
// stage possible; false: region-major only, with the row addresses fixed at compile time.
template <int D, bool BF16, bool KV8, bool Q8 = false, bool BM = MmaLayout<D, KV8, Q8>::BOXMAJ>
struct MmaWarp {
    using Lay = MmaLayout<D, KV8, Q8>;
    using G = StageGeom<D>;
    using GS = typename Lay::GS;
    static constexpr int RC = Lay::RC;
    static constexpr int DH = Lay::DH;
    static constexpr int KSTEPS = D / 16;    // k-steps of S = Q K^T
    static constexpr int NT = DH / 8;        // n-tiles of this warp's O
    static constexpr bool MB = KV8 ? false : BF16;  // operand type of the MMAs (f16 over E4M3 caches)
    static constexpr bool P1 = KV8;                 // one f16 P (11 bits) instead of a 16-bit hi + lo pair
    static constexpr float kP1Scale = 128.f;        // 2^7
    static constexpr int QREGS = Lay::Q_IN_REGS ? KSTEPS : 1;

    int lane, g, tq, mi;  // g: fragment row (and row + 8); tq: column pair; mi: ldmatrix matrix
    uint32_t rs_;         // box-major stages: bytes between two 128-byte regions of a row
    // 16-bit stages: ldmatrix row addresses within a stage (chunk c of row r at c ^ (r & 7)).
    uint32_t kb_row[2], kb_x[4], vb_row[2], vb_x[4];
    // KV8 ldmatrix addresses in a code stage (32 token rows of D/128 regions of 128 bytes).
    // K: lane l addresses token l (matrix = n-tile l / 8).  V: lane l addresses token
    // 16 k2 + 8 ((l >> 3) & 1) + (l & 7) of chunk c + (l >> 4).
    uint32_t k8_row, k8_x, v8_row[2], v8_x;
    uint32_t qa[QREGS][4];
    float o[NT][4];
    float mrow[2], lrow[2];

    // Bytes between two 128-byte regions of a token row in the stage.
    __device__ __forceinline__ uint32_t rs() const {
        if constexpr (BM)
            return rs_;
        else
            return GS::REGION_BYTES;
    }

    // br: token rows per staged box (kStageTokens: the region-major layout; see
    // stage_row_offset); only box-major kernels stage boxes of fewer rows.
    __device__ __forceinline__ explicit MmaWarp(int lane_, int br = kStageTokens)
        : lane(lane_), g(lane_ >> 2), tq(lane_ & 3), mi(lane_ >> 3), rs_(static_cast<uint32_t>(br * 128)) {
        auto row_off = [&](int t) -> uint32_t {
            if constexpr (BM)
                return stage_row_offset<GS::ROW_BYTES>(t, br);
            else
                return static_cast<uint32_t>(t * 128);
        };
        k8_row = row_off(lane);
        k8_x = static_cast<uint32_t>((lane & 7) << 4);
#pragma unroll
        for (int j = 0; j < 2; ++j) v8_row[j] = row_off(16 * j + 8 * ((lane >> 3) & 1) + (lane & 7));
        v8_x = static_cast<uint32_t>((((lane >> 4) & 1) ^ (lane & 7)) << 4);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            kb_row[j] = row_off(8 * (2 * j + (mi >> 1)) + (lane & 7));
            vb_row[j] = row_off(16 * j + 8 * (mi & 1) + (lane & 7));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            kb_x[j] = static_cast<uint32_t>(((2 * j + (mi & 1)) ^ (lane & 7)) << 4);
            vb_x[j] = static_cast<uint32_t>(((2 * j + (mi >> 1)) ^ (lane & 7)) << 4);
        }
        reset();
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        mrow[0] = mrow[1] = -INFINITY;
        lrow[0] = lrow[1] = 0.f;
    }

    // ldmatrix address of this lane in the query rows q_s ([RC][D] 16-bit, row-major).
    __device__ __forceinline__ uint32_t q_lane(const uint16_t* q_s) const {
        return smem_addr(q_s) + ((mi & 1) * 8 + (lane & 7)) * (D * 2) + (mi >> 1) * 16;
    }

    // KV8: A fragments in the permuted k order of the code fragments (dims 16 kk + 4 tq .. + 3
    // of rows g and g + 8: k slots 2tq, 2tq+1 and 2tq+8, 2tq+9).
    __device__ __forceinline__ void load_q8(const uint16_t* q_s, int kk, uint32_t (&a)[4]) const {
        const uint2 r0 = *reinterpret_cast<const uint2*>(q_s + g * D + 16 * kk + 4 * tq);
        const uint2 r1 = *reinterpret_cast<const uint2*>(q_s + (g + 8) * D + 16 * kk + 4 * tq);
        a[0] = r0.x;
        a[1] = r1.x;
        a[2] = r0.y;
        a[3] = r1.y;
    }

    // Q's A fragments into registers (when they stay there for the whole run).
    __device__ __forceinline__ void load_q(const uint16_t* q_s) {
        if constexpr (Lay::Q_IN_REGS) {
            const uint32_t ql = q_lane(q_s);
            static_for<0, KSTEPS>([&](auto kk_) {
                constexpr int kk = decltype(kk_)::value;
                if constexpr (KV8)
                    load_q8(q_s, kk, qa[kk]);
                else
                    ldmatrix_x4(ql + 2 * kk * 16, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            });
        }
    }

    // One 32-token stage: S = Q K^T, masked online softmax in log2 units, O += P V.
    // nv: tokens of the stage that exist (the V rows past them are zeroed here);
    // vis0 / vis1: tokens rows g / g + 8 may see; sl: their logit scales; v_half:
    // byte offset of this warp's DH columns of V; scl (q8_0): the stage's block-scale
    // rows, [32 tokens][D / 32] binary16 for K, then the same for V.
    __device__ __forceinline__ void stage(const uint16_t* q_s, uint8_t* stage_ptr, int nv, int vis0, int vis1,
                                          const float (&sl)[2], uint32_t v_half, uint8_t* scl = nullptr) {
        constexpr int NB = D / 32;  // q8_0 blocks per row
        const uint32_t kbase = smem_addr(stage_ptr);
        const uint32_t vbase = kbase + GS::HALF_BYTES;
        if (nv < kStageTokens) {
            if constexpr (Q8) {  // V scale rows past the end: 0 (their P is 0, and 0 x NaN is NaN)
                if (lane >= nv) {
                    if constexpr (Lay::SCB == 16)
                        *reinterpret_cast<uint4*>(scl + (kStageTokens + lane) * 16) = make_uint4(0u, 0u, 0u, 0u);
                    else
                        *reinterpret_cast<uint2*>(scl + (kStageTokens + lane) * 8) = make_uint2(0u, 0u);
                }
            }
            if constexpr (BM)
                zero_v_tail<D, kStageTokens, KV8 ? 1 : 2>(stage_ptr, nv, lane, 32, static_cast<int>(rs_ >> 7));
            else
                zero_v_tail<D, kStageTokens, KV8 ? 1 : 2>(stage_ptr, nv);
        }
        const uint32_t ql = Lay::Q_IN_REGS ? 0u : q_lane(q_s);
        const __half* sck = reinterpret_cast<const __half*>(scl);  // q8_0: K scales [32][NB], V scales after
        const __half* scv = sck + kStageTokens * NB;

        // S = Q K^T for the stage's 32 tokens (4 n-tiles of 8)
        float sc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        if constexpr (Q8) {
            // q8_0: each 32-dim block (k-steps 2 blk, 2 blk + 1) into an accumulator of its
            // own, then times the block scale of each token column (exact products: the
            // codes and the query are exact in f16) and added to S
            uint32_t ksc[4][NB];  // n-tile n: scales of tokens 8 n + 2 tq and 8 n + 2 tq + 1
#pragma unroll
            for (int n = 0; n < 4; ++n) load_scale_pair<NB>(sck, 8 * n + 2 * tq, ksc[n]);
            static_for<0, NB>([&](auto b_) {
                constexpr int blk = decltype(b_)::value;
                float acc[4][4];
#pragma unroll
                for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
                static_for<0, 2>([&](auto h_) {
                    constexpr int kk = 2 * blk + decltype(h_)::value;
                    constexpr int qk = Lay::Q_IN_REGS ? kk : 0;
                    if constexpr (!Lay::Q_IN_REGS) load_q8(q_s, kk, qa[0]);
                    uint32_t r[4];
                    ldmatrix_x4(kbase + (kk >> 3) * rs() + k8_row + ((static_cast<uint32_t>(kk & 7) << 4) ^ k8_x),
                                r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t b0, b1;
                        i8x4_to_f16(r[j], b0, b1);
                        mma_16816<false>(acc[j], qa[qk], b0, b1);
                    }
                });
#pragma unroll
                for (int n = 0; n < 4; ++n) {  // columns: tokens 8 n + 2 tq and 8 n + 2 tq + 1
                    const float d0 = pair_scale<NB>(ksc[n], 0, blk);
                    const float d1 = pair_scale<NB>(ksc[n], 1, blk);
                    sc[n][0] = fmaf(acc[n][0], d0, sc[n][0]);
                    sc[n][1] = fmaf(acc[n][1], d1, sc[n][1]);
                    sc[n][2] = fmaf(acc[n][2], d0, sc[n][2]);
                    sc[n][3] = fmaf(acc[n][3], d1, sc[n][3]);
                }
            });
        } else static_for<0, KSTEPS>([&](auto kk_) {
            constexpr int kk = decltype(kk_)::value;
            constexpr int qk = Lay::Q_IN_REGS ? kk : 0;
            if constexpr (KV8) {
                if constexpr (!Lay::Q_IN_REGS) load_q8(q_s, kk, qa[0]);
                uint32_t r[4];
                ldmatrix_x4(kbase + (kk >> 3) * rs() + k8_row + ((static_cast<uint32_t>(kk & 7) << 4) ^ k8_x),
                            r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t b0, b1;
                    e4m3x4_to_f16(r[j], b0, b1);
                    mma_16816<false>(sc[j], qa[qk], b0, b1);
                }
            } else {
                if constexpr (!Lay::Q_IN_REGS)
                    ldmatrix_x4(ql + 2 * kk * 16, qa[0][0], qa[0][1], qa[0][2], qa[0][3]);
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(kbase + (kk >> 2) * rs() + kb_row[pr] + kb_x[kk & 3], b0, b1, b2, b3);
                    mma_16816<MB>(sc[2 * pr], qa[qk], b0, b1);
                    mma_16816<MB>(sc[2 * pr + 1], qa[qk], b2, b3);
                }
            }
        });

        // softmax in log2 units on the fragments: element e of n-tile n is
        // row g + 8 * (e >> 1), token 8 n + 2 tq + (e & 1)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = 8 * n + 2 * tq + (e & 1);
                float z = sc[n][e] * sl[e >> 1];
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
            // 0 when m was -inf and the row now sees a token; 1 for a row that still has seen
            // nothing (the branch is taken for the whole warp when any row grows, and
            // -inf - -inf would be NaN and poison its l)
            const float a0 = n0 == -INFINITY ? 1.f : exp2_approx(mrow[0] - n0);
            const float a1 = n1 == -INFINITY ? 1.f : exp2_approx(mrow[1] - n1);
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
        // P as A fragments of two k-steps of 16 tokens: split into high and residual
        // parts, or (P1) one f16 value scaled by 2^7 (p <= 2^8 by the lazy rescale, so
        // p 2^7 <= 2^15 fits f16, and small p stay normal); O then carries 2^7.
        uint32_t ph[2][4], pl[2][4];
#pragma unroll
        for (int k2 = 0; k2 < 2 && !Q8; ++k2) {
            if constexpr (P1) {
                ph[k2][0] = pack_f16x2(sc[2 * k2][0] * kP1Scale, sc[2 * k2][1] * kP1Scale);
                ph[k2][1] = pack_f16x2(sc[2 * k2][2] * kP1Scale, sc[2 * k2][3] * kP1Scale);
                ph[k2][2] = pack_f16x2(sc[2 * k2 + 1][0] * kP1Scale, sc[2 * k2 + 1][1] * kP1Scale);
                ph[k2][3] = pack_f16x2(sc[2 * k2 + 1][2] * kP1Scale, sc[2 * k2 + 1][3] * kP1Scale);
            } else {
                split_pair<MB>(sc[2 * k2][0], sc[2 * k2][1], ph[k2][0], pl[k2][0]);
                split_pair<MB>(sc[2 * k2][2], sc[2 * k2][3], ph[k2][1], pl[k2][1]);
                split_pair<MB>(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1], ph[k2][2], pl[k2][2]);
                split_pair<MB>(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3], ph[k2][3], pl[k2][3]);
            }
        }
        // O += P V
        if constexpr (Q8) {
            // q8_0: output block blk (dims 32 blk .. + 31, chunks c = 2 blk and c + 1) takes
            // P' = p x (V scale of the token's block blk) x 2^(7 - ex), ex such that the
            // stage's largest |scale| of that block is below 2^ex (so |P'| <= p 2^7 <=
            // 2^15 fits f16; the quad's lanes cover all 32 tokens), into an accumulator of
            // its own that is added to O times 2^ex.  This lane's tokens of k-step k2:
            // 16 k2 + 2 tq, + 1 (A registers 0, 1) and 16 k2 + 8 + 2 tq, + 1 (2, 3).
            uint32_t vsc[2][2][NB];  // [k2][h]: scales of tokens 16 k2 + 8 h + 2 tq and + 1
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
                for (int h = 0; h < 2; ++h) load_scale_pair<NB>(scv, 16 * k2 + 8 * h + 2 * tq, vsc[k2][h]);
            static_for<0, NB>([&](auto b_) {
                constexpr int blk = decltype(b_)::value;
                constexpr int c = 2 * blk;
                float dv[2][4];
                float mx = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        dv[k2][j] = pair_scale<NB>(vsc[k2][j >> 1], j & 1, blk);
                        mx = fmaxf(mx, fabsf(dv[k2][j]));
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const int ex = mx > 0.f ? ((__float_as_int(mx) >> 23) & 0xff) - 126 : 0;  // mx < 2^ex
                const float down = __int_as_float((127 - ex) << 23) * kP1Scale;
                const float up = __int_as_float((127 + ex) << 23);
                float acc[4][4];
#pragma unroll
                for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2) {
                    const float w0 = dv[k2][0] * down, w1 = dv[k2][1] * down;
                    const float w2 = dv[k2][2] * down, w3 = dv[k2][3] * down;
                    uint32_t a[4];
                    a[0] = pack_f16x2(sc[2 * k2][0] * w0, sc[2 * k2][1] * w1);
                    a[1] = pack_f16x2(sc[2 * k2][2] * w0, sc[2 * k2][3] * w1);
                    a[2] = pack_f16x2(sc[2 * k2 + 1][0] * w2, sc[2 * k2 + 1][1] * w3);
                    a[3] = pack_f16x2(sc[2 * k2 + 1][2] * w2, sc[2 * k2 + 1][3] * w3);
                    uint32_t r[4];
                    ldmatrix_x4_trans(vbase + (c >> 3) * rs() + v8_row[k2] +
                                          ((static_cast<uint32_t>(c & 7) << 4) ^ v8_x),
                                      r[0], r[1], r[2], r[3]);
                    uint32_t ev[4], od[4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) i8x4_to_f16(__byte_perm(r[m], 0u, 0x3120u), ev[m], od[m]);
                    mma_16816<false>(acc[0], a, ev[0], ev[1]);
                    mma_16816<false>(acc[1], a, od[0], od[1]);
                    mma_16816<false>(acc[2], a, ev[2], ev[3]);
                    mma_16816<false>(acc[3], a, od[2], od[3]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[2 * c + i][e] = fmaf(acc[i][e], up, o[2 * c + i][e]);
            });
        } else
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            if constexpr (KV8) {
                // chunks c, c + 1 (16 dims each): o[2c] / o[2c+1] hold the even / odd dims of chunk c
                static_for<0, D / 32>([&](auto cp_) {
                    constexpr int c = 2 * decltype(cp_)::value;
                    uint32_t r[4];
                    ldmatrix_x4_trans(vbase + (c >> 3) * rs() + v8_row[k2] +
                                          ((static_cast<uint32_t>(c & 7) << 4) ^ v8_x),
                                      r[0], r[1], r[2], r[3]);
                    uint32_t ev[4], od[4];  // by matrix: (tokens 0-7 | 8-15) x (chunk c | c + 1)
#pragma unroll
                    for (int m = 0; m < 4; ++m) e4m3x4_to_f16(__byte_perm(r[m], 0u, 0x3120u), ev[m], od[m]);
                    mma_16816<false>(o[2 * c], ph[k2], ev[0], ev[1]);
                    mma_16816<false>(o[2 * c + 1], ph[k2], od[0], od[1]);
                    mma_16816<false>(o[2 * c + 2], ph[k2], ev[2], ev[3]);
                    mma_16816<false>(o[2 * c + 3], ph[k2], od[2], od[3]);
                });
            } else {
                static_for<0, DH / 16>([&](auto jp_) {
                    constexpr int jp = decltype(jp_)::value;  // 16-column group of this warp's half
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(vbase + v_half + (jp >> 2) * rs() + vb_row[k2] + vb_x[jp & 3], b0, b1,
                                      b2, b3);
                    mma_16816<MB>(o[2 * jp], ph[k2], b0, b1);
                    if constexpr (!P1) mma_16816<MB>(o[2 * jp], pl[k2], b0, b1);
                    mma_16816<MB>(o[2 * jp + 1], ph[k2], b2, b3);
                    if constexpr (!P1) mma_16816<MB>(o[2 * jp + 1], pl[k2], b2, b3);
                });
            }
        }
    }

    // Row sums of the lane quad (after the last stage).
    __device__ __forceinline__ void finish_l() {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
            lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
        }
    }
};

template <int D, bool BF16, bool KV8, bool Q8 = false>
__global__ void __launch_bounds__(MmaLayout<D, KV8, Q8>::THREADS, MmaLayout<D, KV8, Q8>::CTAS_PER_SM)
split_mma_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
    using Lay = MmaLayout<D, KV8, Q8>;
    using W = MmaWarp<D, BF16, KV8, Q8>;
    using G = StageGeom<D>;
    using GS = typename Lay::GS;
    constexpr int NW = Lay::NW;
    constexpr int S = Lay::S;
    constexpr int RC = Lay::RC;
    constexpr int NP = Lay::NP;          // consumer groups, one stage each
    constexpr int DSPLIT = Lay::DSPLIT;  // warps per group (each owns DH columns of O)
    constexpr int DH = Lay::DH;
    constexpr int NT = W::NT;
    constexpr bool QSCALE = KV8 && BF16;     // bf16 query rows rescaled into f16
    const float o_out = W::P1 ? 1.f / W::kP1Scale : 1.f;

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
    uint8_t* sc_ring = stages + S * GS::STAGE_BYTES;  // q8_0: [S][SC_STAGE] block-scale rows

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WorkItem it = p.items[blockIdx.x];
    const int b = it.seq;
    const int kvh = blockIdx.y;
    const int row0 = blockIdx.z * RC;
    const bool tma_mode = p.page_shift >= 3;
    if (threadIdx.x == 0) init_stage_barriers<S>(full, empty, tma_mode, DSPLIT, Q8 ? 33u : 1u);
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
        produce_stages<D, S, kStageTokens, KV8 ? 1 : 2, Lay::SCB, Lay::BOXMAJ>(p, &tmk, &tmv, full, empty, stages, b,
                                                                              kvh, ir, tma_mode, sc_ring);
        return;
    }
    if (threadIdx.x == 0) report_item_range(p, ir);
    // The group's query rows, as stored (16-bit, [RC][D]); rows past the group are zero.
    // QSCALE: bf16 rows -> f16 rows times 2^sh(row), sh from the row's largest magnitude.
    uint32_t* q_rmax = reinterpret_cast<uint32_t*>(smem + Lay::QMAX_OFFSET);  // [RC] largest |q| (bf16 bits)
    {
        QChunks<RC, D, NW * 32> qc;
        qc.load(p, b, kvh, row0, threadIdx.x);
        if constexpr (QSCALE) {
            if (threadIdx.x < RC) q_rmax[threadIdx.x] = 0u;
            named_barrier(1, NW * 32);
#pragma unroll
            for (int i = 0; i < qc.PER; ++i) {
                const int idx = qc.chunk(threadIdx.x, i);
                if (idx < qc.CH) {
                    const uint32_t w[4] = {qc.v[i].x, qc.v[i].y, qc.v[i].z, qc.v[i].w};
                    uint32_t mx = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) mx = max(mx, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
                    atomicMax(&q_rmax[idx / (D / 8)], mx);  // bf16 magnitudes order as integers
                }
            }
            named_barrier(1, NW * 32);
#pragma unroll
            for (int i = 0; i < qc.PER; ++i) {
                const int idx = qc.chunk(threadIdx.x, i);
                if (idx < qc.CH) {
                    const float f = q_row_factor(q_rmax[idx / (D / 8)], true);
                    const uint32_t w[4] = {qc.v[i].x, qc.v[i].y, qc.v[i].z, qc.v[i].w};
                    uint32_t h[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 v = unpack2<true>(w[e]);
                        const __half2 hv = __floats2half2_rn(v.x * f, v.y * f);
                        h[e] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                    *reinterpret_cast<uint4*>(q_s + idx * 8) = make_uint4(h[0], h[1], h[2], h[3]);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < qc.PER; ++i) {
                const int idx = qc.chunk(threadIdx.x, i);
                if (idx < qc.CH) *reinterpret_cast<uint4*>(q_s + idx * 8) = qc.v[i];
            }
        }
    }
    named_barrier(1, NW * 32);

    // ---------------------------------------------------------------------- consumers
    W cw(lane, staged_box_rows(p.page_shift, Lay::BOXMAJ));
    const int g = cw.g, tq = cw.tq;
    cw.load_q(q_s);
    int lim[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int qi = (row0 + g + 8 * h) / p.group;
        lim[h] = p.causal ? (ir.L - p.q_len + qi) : (ir.L - 1);
    }
    // Logit scale of rows g and g + 8 (QSCALE: the row factor taken back out).
    float sl[2] = {p.scale_log2, p.scale_log2};
    if constexpr (QSCALE) {
        sl[0] = p.scale_log2 * q_row_factor(q_rmax[g], false);
        sl[1] = p.scale_log2 * q_row_factor(q_rmax[g + 8], false);
    }
    bool ok = true;

    const int grp = warp / DSPLIT;             // consumer group: stages grp, grp + NP, ...
    const int half = warp - grp * DSPLIT;      // which DH columns of O this warp accumulates
    static_assert(DSPLIT == 1 || !Lay::BOXMAJ, "warp pairs split V by regions of the region-major layout");
    const uint32_t v_half = static_cast<uint32_t>(half * (DH / 64) * G::REGION_BYTES);
    for (int i = grp; i < ir.n_stage; i += NP) {
        const int s = i % S;
        if (!wait_stage<S>(full, i)) {
            ok = false;
            break;
        }
        const int t0 = ir.tok_begin + i * kStageTokens;
        const int nv = min(kStageTokens, ir.tok_end - t0);
        cw.stage(q_s, stages + s * GS::STAGE_BYTES, nv, min(nv, lim[0] - t0 + 1), min(nv, lim[1] - t0 + 1), sl,
                 v_half, Q8 ? sc_ring + s * Lay::SC_STAGE : nullptr);
        if (nv < kStageTokens) fence_proxy_async_shared();  // generic zeroing before the slot's next TMA write
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
    cw.finish_l();
    if (!ok && lane == 0) atomicOr(p.err, FDEC_DEVERR_TIMEOUT);

    // ---------------------------------------------------------------------- epilogue
    named_barrier(1, NW * 32);  // every consumer is done with the stage buffers
    // The reduction (launched as a programmatic dependent) may start its launch now.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float* sm_m = reinterpret_cast<float*>(stages);  // [NP][RC]
    float* sm_l = sm_m + NP * RC;                     // [NP][RC]
    float* sm_o = sm_l + NP * RC;                     // [NP][RC][D]
    if (tq == 0 && half == 0) {  // the warps of a group hold the same m and l
        sm_m[grp * RC + g] = cw.mrow[0];
        sm_m[grp * RC + g + 8] = cw.mrow[1];
        sm_l[grp * RC + g] = cw.lrow[0];
        sm_l[grp * RC + g + 8] = cw.lrow[1];
    }
    if constexpr (KV8) {
        // o[2c] / o[2c+1]: dims 16c + 2n / 16c + 2n + 1 of column n: this lane's columns 2tq, 2tq+1
        // are dims 16c + 4tq + {0, 2} / {1, 3}
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
            *reinterpret_cast<float4*>(sm_o + (grp * RC + g) * D + 16 * c + 4 * tq) =
                make_float4(cw.o[2 * c][0] * o_out, cw.o[2 * c + 1][0] * o_out, cw.o[2 * c][1] * o_out,
                            cw.o[2 * c + 1][1] * o_out);
            *reinterpret_cast<float4*>(sm_o + (grp * RC + g + 8) * D + 16 * c + 4 * tq) =
                make_float4(cw.o[2 * c][2] * o_out, cw.o[2 * c + 1][2] * o_out, cw.o[2 * c][3] * o_out,
                            cw.o[2 * c + 1][3] * o_out);
        }
    }
#pragma unroll
    for (int n = 0; n < (KV8 ? 0 : NT); ++n) {
        *reinterpret_cast<float2*>(sm_o + (grp * RC + g) * D + half * DH + 8 * n + 2 * tq) =
            make_float2(cw.o[n][0] * o_out, cw.o[n][1] * o_out);
        *reinterpret_cast<float2*>(sm_o + (grp * RC + g + 8) * D + half * DH + 8 * n + 2 * tq) =
            make_float2(cw.o[n][2] * o_out, cw.o[n][3] * o_out);
    }
    named_barrier(1, NW * 32);
    merge_and_store<NP, RC, D, NW * 32>(p, it, kvh, row0, sm_m, sm_l, sm_o);
}

template <int D, bool BF16, bool KV8 = false, bool Q8 = false>
cudaError_t launch_split_mma_one(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, dim3 grid,
                                 cudaStream_t stream, bool launch) {
    using Lay = MmaLayout<D, KV8, Q8>;
    static unsigned long long attr_done = 0;  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !(__atomic_load_n(&attr_done, __ATOMIC_ACQUIRE) & (1ull << dev))) {
        e = cudaFuncSetAttribute(split_mma_kernel<D, BF16, KV8, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    return cudaLaunchKernelEx(&cfg, split_mma_kernel<D, BF16, KV8, Q8>, p, tk, tv);
}

}  // namespace fdec
