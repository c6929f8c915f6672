/*
 * fdec.h -- paged split-KV flash-decoding for GB300 (sm_103a): C ABI.
 *
 * Attention of a (multi-token) query over a paged KV cache:
 *
 *   out[b,i,h,:] = sum_t softmax_t(z) V_t,   lse[b,i,h] = ln sum_t exp(z_t),
 *   z_t = scale * q[b,i,h,:] . K_t,  t over the visible tokens of sequence b,
 *   K_t / V_t gathered through the page table (page table[b][t / P], slot t % P),
 *   query head h reading KV head h / (Hq / Hk).
 *
 * The KV range of every sequence is cut into 64-token blocks; a run of blocks
 * (a "split") yields one partial (running max m, sum l, unnormalised o), and a
 * log-sum-exp merge with as many passes as needed combines any number of
 * partials, so the split path serves every context length.  This is the
 * decode_split producer / reduce_fused reducer structure of the HRX issue
 * "flash-attention decode-split template resolution fails ("all_rejected") at
 * longer context" (root cause: 64-token producer blocks, a 32-block reducer
 * scratch; follow-up: the multipass reducer that lane-strides over the block
 * dimension), without its fixed 32-block cap.
 *
 * Conventions for every entry point:
 *   - Return codes only: nothing aborts and no exception crosses the ABI.  On a
 *     non-FDEC_OK return, fdec_last_error() holds a message for this thread.
 *   - The library allocates no device memory, ever.  The caller owns q, K, V,
 *     the page table, seq_lens, out, lse and the workspace.  (The FlashInfer PR
 *     "Stop declaring the paged KV cache mutated on read-only attention ops",
 *     first commit: a lazily allocated untracked tensor broke CUDA-graph pools.)
 *   - K, V and q are only read, never written (same PR, second commit: the
 *     read-only ops must not declare or perform writes to the cache).
 *   - Element strides are in elements of the storage type (16-bit, or one
 *     byte for E4M3 caches); the innermost (head_dim) stride is always 1.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - A plan is not thread-safe: fdec_run caches the tensor maps of the last
 *     K/V descriptors in the plan, so calls on one plan from several host threads
 *     must be serialised by the caller (calls on different plans need not be).
 *     Calls on one plan and workspace from one thread may go to any streams only
 *     if the caller orders them (they share the workspace's partials).
 */
#ifndef FDEC_H
#define FDEC_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FDEC_OK = 0,
    FDEC_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad option */
    FDEC_ERR_LAYOUT = 2,       /* a K/V/q layout the kernels cannot address (alignment, strides) */
    FDEC_ERR_UNSUPPORTED = 3,  /* head_dim / page_size / path not built */
    FDEC_ERR_CAPACITY = 4,     /* a length above the planned capacity */
    FDEC_ERR_CAPTURING = 5,    /* plan upload attempted on a capturing stream */
    FDEC_ERR_WORKSPACE = 6,    /* workspace missing, misaligned, or not the one uploaded */
    FDEC_ERR_CUDA = 7,         /* a CUDA runtime call or kernel launch failed */
    FDEC_ERR_DEVICE = 8        /* a device-side check fired (fdec_read_device_errors) */
} fdec_status;

typedef enum { FDEC_F16 = 0, FDEC_BF16 = 1 } fdec_dtype;

/* Device-side error bits, accumulated in the workspace by the kernels. */
#define FDEC_DEVERR_PAGE_ID 0x1u       /* a page id outside [0, num_pages): that row was skipped */
#define FDEC_DEVERR_SEQ_LEN 0x2u       /* seq_lens[b] above the planned capacity (clamped) or < 0 */
#define FDEC_DEVERR_TIMEOUT 0x4u       /* a bounded pipeline wait gave up; results are invalid */

/*
 * One K or V pool.  Element (page, kv_head, slot, dim) is at
 *   base + page*stride_page + kv_head*stride_head + slot*stride_token + dim.
 * This covers separate K/V pools (HND [pages,Hk,P,D] or NHD [pages,P,Hk,D]),
 * one interleaved [pages,2,Hk,P,D] tensor (K = kv, V = kv + Hk*P*D,
 * stride_page = 2*Hk*P*D), and [2,pages,...] views (K = kv[0], V = kv[1]):
 * the K/V forms of the FlashInfer PR's "Architecture / design notes" table.
 * K and V may differ in strides and page count; only indexed pages are read
 * (same PR, first commit: a shorter V pool).  base must be 16-byte aligned and
 * every stride a multiple of 16 bytes (8 elements of a 16-bit cache, 16 of an
 * E4M3 cache), so that each token row starts on a 16-byte boundary; otherwise
 * fdec_run returns FDEC_ERR_LAYOUT.
 */
typedef struct {
    const void* base;
    int64_t num_pages;
    int64_t stride_page;
    int64_t stride_head;
    int64_t stride_token;
} fdec_kv_desc;

typedef struct fdec_plan_s* fdec_plan_t;

/*
 * Split-kernel paths.  SIMT: fp32 FMA (every head_dim).  MMA: warp-level
 * tensor-core MMA on 16-row query groups (every head_dim), the decode
 * default.  TC: 5th-generation tensor cores (tcgen05, accumulators in tensor
 * memory) on 128-row query tiles, head_dim 64, 128, 192 and 256 (at 512 the
 * output accumulator alone would fill tensor memory); chosen by AUTO when q_len
 * x group > 16 (> 32 at head_dim 256), where attention over the gathered pages
 * turns into a dense contraction (speculative-decode and prefill chunks) and the
 * 16-row kernel would stream K/V once per 16-row group.  Up to 16 rows the work
 * is bound by streaming K/V and the 16-row kernel wastes no tensor-core tile
 * (measured crossover: the 16-row kernel is faster at 16 rows for every head_dim
 * the TC path is built for, and at 32 rows for head_dim 256; slower above).
 */
enum { FDEC_PATH_AUTO = 0, FDEC_PATH_SIMT = 1, FDEC_PATH_MMA = 2, FDEC_PATH_TC = 3 };

/*
 * K/V storage types.  SAME: K and V are 16-bit, of the query's dtype.  E4M3:
 * quantised caches of 8-bit OCP E4M3 codes (the fp8 caches of the FlashInfer
 * PR's AITER paged-attention notes, with a k_scale and a v_scale): the key and
 * value of a token are k_scale x the decoded K code and v_scale x the decoded V
 * code (scales given to fdec_run_scaled).  E4M3 caches run on the MMA path with
 * head_dim 128 or 256; the codes are staged as they are stored and widened to
 * 16 bits in shared memory, so no dequantised copy of the cache exists anywhere.
 * Q8_0: the llama.cpp block format the turboquant PR's caches use ("q8_0-K"; the
 * HRX issue lists "KV cache types (q8_0 / q4_0)" as open); the pages name it and
 * do not print it, so this is its public definition: each K/V row of head_dim
 * elements is head_dim / 32 blocks of 32 signed 8-bit codes, one binary16 scale
 * per block, and element e is scale[e / 32] x code[e].  Codes and scales live in
 * separate pools (fdec_run_q8_0); MMA path, head_dim 128 or 256.
 */
enum { FDEC_KV_SAME = 0, FDEC_KV_E4M3 = 1, FDEC_KV_Q8_0 = 2 };

/* Plan options; pass NULL for the defaults (all fields 0). */
typedef struct {
    int blocks_per_split;  /* 64-token blocks per split; 0 = auto; 1 = one partial per block */
    int reducer_fanin;     /* partials merged per reduction task; 0 = auto (1024); >= 2 */
    int path;              /* FDEC_PATH_AUTO (TC when head_dim <= 256 and q_len x group > 16, > 32 at 256, else
                              MMA), _SIMT, _MMA (every head_dim), _TC (head_dim 64, 128, 192, 256) */
    int num_sms;           /* 0 = query the current device; > 0 plans without a device */
    int kv_dtype;          /* FDEC_KV_SAME (0), FDEC_KV_E4M3 or FDEC_KV_Q8_0 (head_dim 128 / 256; path AUTO
                              or MMA) */
} fdec_plan_opts;

/* What a plan decided (for logging, tests and benchmarks). */
typedef struct {
    int path;              /* FDEC_PATH_SIMT, FDEC_PATH_MMA or FDEC_PATH_TC */
    int blocks_per_split;
    int num_items;         /* split work items (each runs for every KV head and row group) */
    int num_split_ctas;    /* CTAs of the split launch */
    int row_groups;        /* query-row groups per (sequence, KV head) */
    int rows_per_group;
    int max_splits;        /* largest split count of any sequence */
    int reduce_passes;     /* 0 when every sequence has a single split */
    int launches;          /* kernel launches per fdec_run */
    int num_sms;
    size_t workspace_bytes;
} fdec_plan_info;

/*
 * Plan a run (host only; no device memory is touched).
 *   seq_lens_host[batch]: the capacity of each sequence, i.e. the largest KV
 *     length fdec_run will be given for it.  The 64-token block count is
 *     ceil(capacity / 64) (the HRX issue's key_value_capacity =
 *     ceil_div(n, 64) * 64).  The launch grid and workspace strides are fixed
 *     from these capacities; the loop bounds come from the device seq_lens at
 *     run time, so one plan serves a decode loop whose lengths grow up to the
 *     capacity (the HRX issue's SGPR-exhaustion fix: loop bound at run time,
 *     partial stride fixed from capacity).
 *   q_len >= 1 (query tokens per sequence); causal applies only when q_len > 1
 *     (query i sees tokens t <= L - q_len + i, bottom-right aligned).
 *   page_size: a power of two in [1, 256].  head_dim: 64, 128, 192, 256 or 512.
 *   num_qo_heads must be a multiple of num_kv_heads.
 * On success *out_plan owns host memory released by fdec_plan_destroy and
 * *workspace_bytes is the device workspace fdec_plan_upload / fdec_run need.
 * The only CUDA calls are device attribute queries (skipped when opts->num_sms > 0).
 */
fdec_status fdec_plan(const int32_t* seq_lens_host, int batch, int q_len, int page_size,
                      int num_qo_heads, int num_kv_heads, int head_dim, fdec_dtype dtype,
                      int causal, const fdec_plan_opts* opts, fdec_plan_t* out_plan,
                      size_t* workspace_bytes);

/*
 * Copy the plan's work lists into `workspace` (>= workspace_bytes, 256-byte
 * aligned, device memory) and clear its device error word.  Must not be called
 * while `stream` is capturing (FDEC_ERR_CAPTURING).  Blocks until the copy is done.
 */
fdec_status fdec_plan_upload(fdec_plan_t plan, void* workspace, cudaStream_t stream);

/*
 * Run the planned attention.  Kernel launches only (no allocation, no copy, no
 * synchronisation), so it may be captured in a CUDA graph once the plan is
 * uploaded.  The decode kernel (16-bit caches, up to 16 rows per KV head) is a
 * programmatic dependent of the kernel before it on `stream`: its CTAs may start
 * while that kernel finishes, but it reads and writes nothing (inputs, outputs,
 * workspace) until that kernel has completed, so stream order holds as for an
 * ordinary launch.
 *   q: [batch, q_len, Hq, head_dim] 16-bit, element (b, i, h, d) at
 *      q + (b*q_len + i)*q_stride_tok + h*q_stride_head + d.  Covers a packed q,
 *      a head slice of a fused QKV tensor, and a head-major q (FlashInfer PR,
 *      first commit, q layouts).
 *   k, v: the pools (see fdec_kv_desc).  Read only.
 *   page_table: int32 device [batch][page_table_stride]; row b lists the
 *      physical pages of sequence b in token order; page_table_stride must be
 *      >= ceil(capacity_b / page_size) for every b.
 *   seq_lens_dev: int32 device [batch], each in [0, capacity_b].
 *   scale: logit scale (1/sqrt(head_dim) for standard attention).
 *   out: float32 device [batch, q_len, Hq, head_dim], contiguous (written densely).
 *   lse: float32 device [batch, q_len, Hq] natural-log LSE of the scaled logits,
 *      or NULL.  An empty row gives out = 0 and lse = -inf.
 *   workspace: the buffer passed to fdec_plan_upload for this plan.
 */
fdec_status fdec_run(fdec_plan_t plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                     fdec_kv_desc k, fdec_kv_desc v, const int32_t* page_table,
                     int64_t page_table_stride, const int32_t* seq_lens_dev, float scale,
                     float* out, float* lse, void* workspace, cudaStream_t stream);

/*
 * fdec_run for scaled caches: K_t = k_scale x stored K_t and V_t = v_scale x
 * stored V_t (E4M3 caches, see FDEC_KV_E4M3; any cache may carry scales).  So
 * z_t = scale x k_scale x q . K_stored_t and out = v_scale x (the attention of
 * the stored values); lse does not depend on v_scale.  The scales are host
 * values: nothing is read from or allocated on the device for them, so a
 * captured graph holds them as launch arguments (the FlashInfer PR's first
 * commit: a lazily allocated unit-scale tensor broke graph pools).  Both must
 * be finite (FDEC_ERR_INVALID_ARG).  fdec_run is this call with 1 and 1.
 */
fdec_status fdec_run_scaled(fdec_plan_t plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                            fdec_kv_desc k, fdec_kv_desc v, const int32_t* page_table,
                            int64_t page_table_stride, const int32_t* seq_lens_dev, float scale,
                            float k_scale, float v_scale, float* out, float* lse, void* workspace,
                            cudaStream_t stream);

/*
 * fdec_run for q8_0 caches (plans made with kv_dtype FDEC_KV_Q8_0; fdec_run and
 * fdec_run_scaled refuse them with FDEC_ERR_INVALID_ARG).  k and v describe the
 * code pools as for E4M3 caches: one signed byte per element, strides in
 * elements (bytes), 16-byte aligned base and strides.  k_scales and v_scales
 * describe the block-scale pools: binary16, scale j of (page, head, slot) at
 * base + page*stride_page + head*stride_head + slot*stride_token + j (elements),
 * j < head_dim / 32; base aligned to head_dim / 16 bytes and strides multiples
 * of head_dim / 32 (FDEC_ERR_LAYOUT otherwise); a page id must be below every
 * pool's num_pages.  Neither codes nor scales are written; the scales are staged
 * with their tokens' codes and applied in the kernel, so no dequantised copy
 * exists.  Otherwise as fdec_run (k_scale = v_scale = 1).
 */
fdec_status fdec_run_q8_0(fdec_plan_t plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                          fdec_kv_desc k, fdec_kv_desc k_scales, fdec_kv_desc v, fdec_kv_desc v_scales,
                          const int32_t* page_table, int64_t page_table_stride, const int32_t* seq_lens_dev,
                          float scale, float* out, float* lse, void* workspace, cudaStream_t stream);

/*
 * Merge n_states normalised attention states (as fdec_run writes them) over
 * disjoint KV ranges: lse_out = ln sum_i exp(lse_i), o_out = sum_i
 * exp(lse_i - lse_out) o_i; a state with lse = -inf contributes nothing, and
 * rows where every state is empty give o_out = 0, lse_out = -inf.  This is the
 * merge/cascade operation of the FlashInfer test plan (test_cascade).
 *   o: float32 device [n_states][rows][head_dim]; lse: float32 device [n_states][rows].
 *   o_out: [rows][head_dim]; lse_out: [rows] (may be NULL).  head_dim: 1..512.
 * One kernel launch; lanes stride over any number of states.
 */
fdec_status fdec_merge_states(const float* o, const float* lse, int n_states, int rows,
                              int head_dim, float* o_out, float* lse_out, cudaStream_t stream);

/*
 * Paged KV append, the write side of the cache (FlashInfer PR "Stop declaring
 * the paged KV cache mutated on read-only attention ops", append notes: the
 * append op genuinely writes the cache; K and V are best given as separate
 * storage).  For each new token i of n_tokens, with b = batch_indices[i] and
 * position t = positions[i] (its index within sequence b):
 *   page = page_table[b * page_table_stride + t / page_size], slot = t % page_size,
 *   K[page, h, slot, :] = k_new[i, h, :] and V[page, h, slot, :] = v_new[i, h, :]
 * for every KV head h.  Nothing else of K or V is written.
 *   k_new, v_new: 16-bit device [n_tokens][num_kv_heads][head_dim] with token
 *      stride new_stride_tok and head stride new_stride_head (elements; unit
 *      dim stride; 16-byte aligned rows).
 *   batch_indices, positions: int32 device [n_tokens].
 *   k, v: the cache pools (fdec_kv_desc, same rules as fdec_run).
 *   page_table: int32 device [batch][page_table_stride], as for fdec_run.
 *   device_errors: optional uint32 device word; a page id outside the pool sets
 *      FDEC_DEVERR_PAGE_ID, and a position outside [0, page_table_stride *
 *      page_size) or a sequence outside [0, batch) sets FDEC_DEVERR_SEQ_LEN;
 *      that token is skipped.
 * Errors: FDEC_ERR_INVALID_ARG (null pointers, counts), FDEC_ERR_UNSUPPORTED
 * (head_dim, page_size), FDEC_ERR_LAYOUT (alignment and stride rules).
 * Tokens must not repeat a (sequence, position) (the order of two writes to
 * one slot is unspecified).  One kernel launch, no allocation; capturable.
 */
fdec_status fdec_append(const void* k_new, const void* v_new, int64_t new_stride_tok, int64_t new_stride_head,
                        const int32_t* batch_indices, const int32_t* positions, int n_tokens, int num_kv_heads,
                        int head_dim, int page_size, fdec_kv_desc k, fdec_kv_desc v, const int32_t* page_table,
                        int batch, int64_t page_table_stride, uint32_t* device_errors, cudaStream_t stream);

/*
 * fdec_append for E4M3 caches (FDEC_KV_E4M3): k_new / v_new hold E4M3 codes,
 * one byte per element, and are copied into the code pools unchanged (the
 * caller quantises with its k_scale / v_scale; the library never re-rounds).
 * Strides are in bytes and must be multiples of 16; otherwise as fdec_append.
 */
fdec_status fdec_append_e4m3(const void* k_new, const void* v_new, int64_t new_stride_tok, int64_t new_stride_head,
                             const int32_t* batch_indices, const int32_t* positions, int n_tokens, int num_kv_heads,
                             int head_dim, int page_size, fdec_kv_desc k, fdec_kv_desc v, const int32_t* page_table,
                             int batch, int64_t page_table_stride, uint32_t* device_errors, cudaStream_t stream);

/* Release a plan (NULL is a no-op). */
fdec_status fdec_plan_destroy(fdec_plan_t plan);

/* Report what the plan decided. */
fdec_status fdec_plan_get_info(fdec_plan_t plan, fdec_plan_info* info);

/* Per-sequence split counts (batch entries). */
fdec_status fdec_plan_get_splits(fdec_plan_t plan, int32_t* splits, int batch);

/*
 * Timing hook: when `event` is non-NULL every later fdec_run records it on its
 * stream right after the split launch, before the reduction launches, so the
 * caller can time the split kernel alone.  NULL turns it off.
 */
fdec_status fdec_plan_set_split_event(fdec_plan_t plan, cudaEvent_t event);

/*
 * Read (synchronously, on `stream`) the device error bits FDEC_DEVERR_* that
 * the kernels accumulated in `workspace` since the last upload or clear; clear
 * them when `clear` is non-zero.  Not capturable.
 */
fdec_status fdec_read_device_errors(fdec_plan_t plan, void* workspace, uint32_t* flags, int clear,
                                    cudaStream_t stream);

/*
 * fdec_run without any workspace from the caller (the pages have no
 * counterpart: this is a convenience of this library).  For callers that
 * cannot allocate device memory at all, e.g. a plug-in inside a program whose
 * memory pool owns the whole device, or a loop that must never call
 * cudaMalloc because it may synchronise the device.  Inputs and outputs are
 * as for fdec_run, and so is the result: the cache is read unscaled
 * (k_scale = v_scale = 1), as fdec_run reads it; scaled caches go through
 * fdec_run_scaled with a workspace, and q8_0 plans are refused as fdec_run
 * refuses them (they need fdec_run_q8_0 with a workspace).  The partials and work lists live in a
 * 16 MiB array built into the library, which every GPU that loads the library
 * keeps until the process exits.  A plan whose workspace_bytes exceeds 16 MiB
 * is rejected with FDEC_ERR_WORKSPACE (use fdec_run with your own workspace).
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The plan needs no fdec_plan_upload: every call copies the plan's work
 *     lists (host memory) into the array with cudaMemcpyAsync on `stream`,
 *     which also clears the device error word, then launches the kernels.
 *   - Not for CUDA graph capture: every call copies the work lists from the
 *     plan's pageable host memory, which stream capture does not accept.  A
 *     captured decode loop uses fdec_run with an uploaded workspace.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for the
 *     process.  The address belongs to the device's primary context: do not
 *     call this entry point again on a device after cudaDeviceReset of that
 *     device.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race and corrupt each other's results.
 *   - Device error bits land in the array and are not reported; use fdec_run
 *     and fdec_read_device_errors where they matter.
 */
fdec_status fdec_run_static_workspace(fdec_plan_t plan, const void* q, int64_t q_stride_tok,
                                      int64_t q_stride_head, fdec_kv_desc k, fdec_kv_desc v,
                                      const int32_t* page_table, int64_t page_table_stride,
                                      const int32_t* seq_lens_dev, float scale, float* out, float* lse,
                                      cudaStream_t stream);

/* Message of the last failure on this thread ("" if none). */
const char* fdec_last_error(void);

/* Library version string. */
const char* fdec_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FDEC_H */
