// fdec_internal.h -- kernel parameter blocks and launcher declarations shared by
// the C-ABI layer (fdec_api.cu) and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace fdec {

// The split granularity: every split is a run of whole 64-token blocks (the HRX
// decode_split producer runs one workgroup per 64-token KV block).
constexpr int kBlockTokens = 64;
// One pipeline stage carries 32 consecutive tokens of K and V (one per lane).
constexpr int kStageTokens = 32;

// Work item of the split kernel: sequence, [block_begin, block_end) in 64-token
// blocks, and the partial slot (-1: the item covers its whole sequence and
// writes out/lse directly).
struct WorkItem {
    int32_t seq;
    int32_t block_begin;
    int32_t block_end;
    int32_t slot;
};

// Reduction task: merge partial slots [src, src + count) of one sequence into
// slot dst of the next level, or into out/lse when dst < 0.
struct ReduceTask {
    int32_t seq;
    int32_t src;
    int32_t count;
    int32_t dst;
};

struct SplitParams {
    const uint16_t* q;
    int64_t q_stride_tok;
    int64_t q_stride_head;
    const uint8_t* k_base;   // byte strides below
    int64_t k_pages, k_sp, k_sh, k_st;
    const uint8_t* v_base;
    int64_t v_pages, v_sp, v_sh, v_st;
    // q8_0 caches: the binary16 block-scale rows (head_dim / 32 per token), byte strides
    const uint8_t* ks_base;
    int64_t ks_sp, ks_sh, ks_st;
    const uint8_t* vs_base;
    int64_t vs_sp, vs_sh, vs_st;
    const int32_t* page_table;
    int64_t pt_stride;
    const int32_t* seq_lens;
    const int32_t* capacity;   // planned capacity per sequence (workspace copy)
    const WorkItem* items;
    float* part_o;             // [slot][Hk][rows][D]
    float2* part_ml;           // [slot][Hk][rows]  (m in log2 units, l)
    float* out;                // [B*Q*Hq][D]
    float* lse;                // [B*Q*Hq] or null
    unsigned* err;
    int q_len, hq, hk, group, rows, page_shift, causal;
    float scale_log2;          // scale * k_scale * log2(e): logits are kept in log2 units
    float v_scale;             // value scale (quantised caches; 1 otherwise), applied to O
    // Persistent split kernel: work units = items x KV heads x row groups, in item
    // order; CTA c starts with unit c and takes the units past the grid from the
    // ticket counter (advanced by exactly n_units per launch).
    int n_units;
    unsigned long long* ticket;
    // One sequence (batch 1): its work items are runs of seq1_bps blocks in order, so
    // a unit's item follows from its index with no table read (0: read the table).
    int seq1_bps, seq1_blocks, seq1_capacity;
};

struct ReduceParams {
    const ReduceTask* tasks;
    const float* src_o;        // [slot][Hk][rows][D]
    const float2* src_ml;      // (m in log2 units, l) per source row
    const float* src_lse;      // natural-log lse per source row when normalized_input
    float* dst_o;
    float2* dst_ml;
    float* out;                // final: [B*Q*Hq][D]
    float* lse;                // final: [B*Q*Hq] or null
    int hk, rows, group, q_len, hq, head_dim;
    int normalized_input;      // 1: sources are normalised (o, lse) states (merge_states)
    int src_rows_stride;       // rows per (slot, kv head) in the source arrays
    int warps_per_unit;        // 1, 2 or 4 (reduce_warps_per_unit of the largest task)
};

// Launch the split kernel for head_dim D (defined in split_d<D>.cu); rc is the
// compile-time query-row group.  With launch == false only the kernel's
// shared-memory attribute is set (done at upload, outside any capture).
cudaError_t launch_split_d64(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc,
                               bool bf16, dim3 grid, cudaStream_t s, bool launch);
cudaError_t launch_split_d128(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc,
                               bool bf16, dim3 grid, cudaStream_t s, bool launch);
cudaError_t launch_split_d192(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc,
                               bool bf16, dim3 grid, cudaStream_t s, bool launch);
cudaError_t launch_split_d256(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc,
                               bool bf16, dim3 grid, cudaStream_t s, bool launch);
cudaError_t launch_split_d512(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc,
                               bool bf16, dim3 grid, cudaStream_t s, bool launch);

// The tensor-core split kernel (head_dim 64, 128, 192, 256, 512; query rows in
// groups of 16).  kv8: K/V stored as E4M3 codes (head_dim 128 and 256).
cudaError_t launch_split_mma(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                             bool bf16, bool kv8, dim3 grid, cudaStream_t s, bool launch);
size_t split_mma_smem_bytes(int head_dim, bool kv8);
// The persistent form of the tensor-core split kernel (16-bit caches, every head_dim;
// q rows 16-byte aligned): CTAs stay resident and take work units until none is left,
// so a unit's pipeline fill is paid once per CTA and not once per work item.
cudaError_t launch_split_mma_persist(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                                     bool bf16, dim3 grid, cudaStream_t s, bool launch);
inline bool split_mma_persist_supported(int head_dim) {
    return head_dim == 64 || head_dim == 128 || head_dim == 192 || head_dim == 256 || head_dim == 512;
}
inline int split_mma_persist_ctas_per_sm(int head_dim) { return head_dim > 256 ? 1 : 2; }
int split_mma_threads(int head_dim, bool kv8);
inline bool split_mma_kv8_supported(int head_dim) { return head_dim == 128 || head_dim == 256; }
// Whether the tensor-core split kernels stage pages smaller than a stage one box per
// page ([box][region][rows][128 B]) rather than region-major: all but 16-bit head_dim
// 512 (MmaLayout / PersistLayout BOXMAJ); their tensor maps then take every region.
inline bool split_mma_box_major(int head_dim, bool kv8) { return kv8 || head_dim <= 256; }
// q8_0 caches (int8 codes in blocks of 32 with one binary16 scale each) on the
// one-CTA-per-item tensor-core kernel, head_dim 128 and 256.
cudaError_t launch_split_mma_q8(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                                bool bf16, dim3 grid, cudaStream_t s, bool launch);
size_t split_mma_q8_smem_bytes(int head_dim);
int split_mma_q8_threads(int head_dim);
constexpr int kMmaRows = 16;

// The tcgen05 dense-query split kernel (head_dim 64, 128, 192, 256; `tiles` 128-row
// query tiles per CTA: 1 or 2 for head_dim 64 and 128, 1 above; 64-token stages: its
// tensor maps use boxes of min(page_size, 64) token rows).
cudaError_t launch_split_tc(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int tiles, int head_dim,
                            bool bf16, dim3 grid, cudaStream_t s, bool launch);
size_t split_tc_smem_bytes(int tiles, int head_dim);
int split_tc_threads(int tiles, bool bf16);
inline bool split_tc_supported(int head_dim) {
    return head_dim == 64 || head_dim == 128 || head_dim == 192 || head_dim == 256;
}
inline int split_tc_max_tiles(int head_dim) { return head_dim <= 128 ? 2 : 1; }
constexpr int kTcRows = 128;
constexpr int kTcStageTokens = 64;

// Shared-memory bytes and threads of the split kernel for (D, RC); 0 if not built.
size_t split_smem_bytes(int head_dim, int rc);
int split_threads(int head_dim);
int split_max_rc(int head_dim);

int reduce_warps_per_unit(int max_count);
cudaError_t launch_reduce(const ReduceParams& p, int num_tasks, cudaStream_t s);

// Paged KV append (fdec_append, fdec_append_e4m3).  Strides in bytes; every row
// is row_bytes long (a multiple of 16) and starts on a 16-byte boundary.
struct AppendParams {
    const uint8_t* k_new;
    const uint8_t* v_new;
    int64_t new_st, new_sh;
    const int32_t* batch_indices;
    const int32_t* positions;
    const int32_t* page_table;
    int64_t pt_stride;
    uint8_t* k_base;
    int64_t k_pages, k_sp, k_sh, k_st;
    uint8_t* v_base;
    int64_t v_pages, v_sp, v_sh, v_st;
    unsigned* err;
    int n_tokens, batch, hk, row_bytes, page_shift;
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
// One task given by value (p.tasks must be null): used by fdec_merge_states.
cudaError_t launch_reduce_single(const ReduceParams& p, ReduceTask task, cudaStream_t s);

}  // namespace fdec
