// fdec_api.cu -- the C ABI: planning, validation, upload, launch and errors.
//
// Planning follows the dispatch lesson of the HRX decode-split issue: the
// split path must be chosen at every context length (its matcher once stopped
// at a capacity of 2048 = 32 blocks x 64 tokens and handed longer contexts to
// a serial fallback, -32% at depth 2100).  Here every sequence is cut into
// splits of whole 64-token blocks, the split count follows the machine (SM
// count) and the batch, and the reduction takes as many passes as needed.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/fdec.h"
#include "fdec_internal.h"
#include "split_kernel.cuh"

using namespace fdec;

namespace {

thread_local std::string g_last_error;

fdec_status fail(fdec_status st, const std::string& msg) {
    g_last_error = msg;
    return st;
}

fdec_status fail_cuda(cudaError_t e, const char* what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return FDEC_ERR_CUDA;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int ilog2_exact(int x) {
    int s = 0;
    while ((1 << s) < x) ++s;
    return (1 << s) == x ? s : -1;
}

int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

bool head_dim_supported(int d) { return d == 64 || d == 128 || d == 192 || d == 256 || d == 512; }

template <int D>
size_t smem_for_rc(int rc) {
    switch (rc) {
        case 1: return SplitLayout<D, 1>::SMEM;
        case 2: return SplitLayout<D, 2>::SMEM;
        case 4: return SplitLayout<D, 4>::SMEM;
        case 8:
            if constexpr (SplitShape<D>::RCMAX >= 8) return SplitLayout<D, 8>::SMEM;
            return 0;
        case 16:
            if constexpr (SplitShape<D>::RCMAX >= 16) return SplitLayout<D, 16>::SMEM;
            return 0;
        default: return 0;
    }
}

}  // namespace

namespace fdec {

size_t split_smem_bytes(int d, int rc) {
    switch (d) {
        case 64: return smem_for_rc<64>(rc);
        case 128: return smem_for_rc<128>(rc);
        case 192: return smem_for_rc<192>(rc);
        case 256: return smem_for_rc<256>(rc);
        case 512: return smem_for_rc<512>(rc);
        default: return 0;
    }
}

int split_threads(int d) {
    switch (d) {
        case 64: return SplitLayout<64, SplitShape<64>::RCMAX>::THREADS;
        case 128: return SplitLayout<128, SplitShape<128>::RCMAX>::THREADS;
        case 192: return SplitLayout<192, SplitShape<192>::RCMAX>::THREADS;
        case 256: return SplitLayout<256, SplitShape<256>::RCMAX>::THREADS;
        case 512: return SplitLayout<512, SplitShape<512>::RCMAX>::THREADS;
        default: return 0;
    }
}

int split_max_rc(int d) {
    switch (d) {
        case 64: return SplitShape<64>::RCMAX;
        case 128: return SplitShape<128>::RCMAX;
        case 192: return SplitShape<192>::RCMAX;
        case 256: return SplitShape<256>::RCMAX;
        case 512: return SplitShape<512>::RCMAX;
        default: return 0;
    }
}

}  // namespace fdec

struct fdec_plan_s {
    int batch = 0, q_len = 1, page_size = 1, page_shift = 0;
    int hq = 0, hk = 0, head_dim = 0, group = 1, rows = 1;
    fdec_dtype dtype = FDEC_BF16;
    bool kv8 = false;  // K/V stored as 8-bit codes (E4M3, or q8_0 with q8 set)
    bool q8 = false;   // q8_0: int8 codes in blocks of 32 with a binary16 scale each
    int causal = 0;
    int path = FDEC_PATH_SIMT;
    bool persistent = false;  // MMA path over 16-bit caches: resident CTAs take work units
    int n_units = 0, persist_grid = 0;
    int rc = 1, row_groups = 1;
    int blocks_per_split = 1, fanin = 64, num_sms = 0, ctas_per_sm = 1;
    int max_pages_needed = 0;  // max_b ceil(capacity_b / page_size)
    std::vector<int32_t> capacity;
    std::vector<int32_t> splits;  // per sequence
    std::vector<WorkItem> items;
    std::vector<std::vector<ReduceTask>> passes;
    // workspace layout
    size_t off_err = 0, off_ticket = 0, off_cap = 0, off_items = 0;
    std::vector<size_t> off_tasks;
    size_t off_a_o = 0, off_a_ml = 0, off_b_o = 0, off_b_ml = 0;
    size_t slots_a = 0, slots_b = 0;
    size_t meta_bytes = 0, ws_bytes = 0;
    std::vector<uint8_t> meta;  // host image of [0, meta_bytes)
    void* uploaded = nullptr;
    cudaEvent_t split_event = nullptr;
    // Tensor maps of the last K/V descriptors seen by fdec_run (re-encoded on change).
    bool maps_valid = false;
    fdec_kv_desc map_k{}, map_v{};
    CUtensorMap tmap_k{};
    CUtensorMap tmap_v{};
};

namespace {

// Longest-processing-time makespan of `sizes` (each repeated `copies` times)
// on `slots` identical CTA slots, plus a fixed cost per item.
double lpt_makespan(std::vector<int> sizes, int copies, int slots, double per_item) {
    std::sort(sizes.begin(), sizes.end(), std::greater<int>());
    std::priority_queue<double, std::vector<double>, std::greater<double>> load;
    for (int i = 0; i < slots; ++i) load.push(0.0);
    double worst = 0.0;
    for (int s : sizes) {
        for (int c = 0; c < copies; ++c) {
            double l = load.top();
            load.pop();
            l += s + per_item;
            worst = std::max(worst, l);
            load.push(l);
        }
    }
    return worst;
}

std::vector<int> item_sizes(const std::vector<int>& nblocks, int C) {
    std::vector<int> out;
    for (int nb : nblocks) {
        int left = nb;
        do {
            out.push_back(std::min(C, std::max(left, 0)));
            left -= C;
        } while (left > 0);
    }
    return out;
}

// partial_cost: the cost of one partial slot (written by the split kernel and
// read back by the reduction: 2 x Hk x rows x (4 D + 8) bytes) in the same units.
int choose_blocks_per_split(const std::vector<int>& nblocks, int copies, int slots, double partial_cost) {
    const int max_nb = std::max(1, *std::max_element(nblocks.begin(), nblocks.end()));
    long long total = 0;
    for (int nb : nblocks) total += std::max(nb, 1);
    // Cost model in units of one 64-token block streamed by one CTA slot: the
    // LPT makespan of the items, a fixed cost per item (a CTA's start-up and
    // epilogue, or a persistent CTA's unit switch: both measured at a few blocks'
    // worth), the extra reduction launch when any sequence is split, and the
    // partials' traffic.
    const double per_item = 2.0;
    const double reduce_cost = 4.0;
    std::vector<int> cands;
    const long long lo = std::max<long long>(1, (total * copies) / (8LL * slots));
    if (max_nb - lo <= 512) {
        for (long long c = lo; c <= max_nb; ++c) cands.push_back(static_cast<int>(c));
    } else {
        for (double c = static_cast<double>(lo); c < max_nb; c *= 1.02) cands.push_back(static_cast<int>(c));
        cands.push_back(max_nb);
    }
    int best = max_nb;
    double best_cost = 1e300;
    for (int C : cands) {
        const std::vector<int> sizes = item_sizes(nblocks, C);
        const bool split = sizes.size() > nblocks.size();
        size_t partials = 0;
        for (int nb : nblocks) {
            const int n = (std::max(nb, 1) + C - 1) / C;
            if (n > 1) partials += n;
        }
        const double cost = lpt_makespan(sizes, copies, slots, per_item) +
                            (split ? reduce_cost + partial_cost * static_cast<double>(partials) : 0.0);
        if (cost < best_cost - 1e-9 || (std::fabs(cost - best_cost) <= 1e-9 && C > best)) {
            best_cost = cost;
            best = C;
        }
    }
    return best;
}

cudaError_t dispatch_split(const fdec_plan_s* p, const SplitParams& sp, dim3 grid, cudaStream_t stream, bool launch,
                           bool persist = false) {
    const bool bf16 = p->dtype == FDEC_BF16;
    const CUtensorMap& tk = p->tmap_k;
    const CUtensorMap& tv = p->tmap_v;
    if (persist)
        return launch_split_mma_persist(sp, tk, tv, p->head_dim, bf16, dim3(static_cast<unsigned>(p->persist_grid), 1, 1),
                                        stream, launch);
    if (p->path == FDEC_PATH_TC)
        return launch_split_tc(sp, tk, tv, p->rc / kTcRows, p->head_dim, bf16, grid, stream, launch);
    if (p->path == FDEC_PATH_MMA)
        return p->q8 ? launch_split_mma_q8(sp, tk, tv, p->head_dim, bf16, grid, stream, launch)
                     : launch_split_mma(sp, tk, tv, p->head_dim, bf16, p->kv8, grid, stream, launch);
    switch (p->head_dim) {
        case 64: return launch_split_d64(sp, tk, tv, p->rc, bf16, grid, stream, launch);
        case 128: return launch_split_d128(sp, tk, tv, p->rc, bf16, grid, stream, launch);
        case 192: return launch_split_d192(sp, tk, tv, p->rc, bf16, grid, stream, launch);
        case 256: return launch_split_d256(sp, tk, tv, p->rc, bf16, grid, stream, launch);
        case 512: return launch_split_d512(sp, tk, tv, p->rc, bf16, grid, stream, launch);
        default: return cudaErrorInvalidValue;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// A 5-D tensor map over one K or V pool, dims (128 bytes of a row: 64 16-bit
// elements or 128 E4M3 codes; eb = element bytes), slot, 128-byte region of the
// row, KV head, page), 128-byte swizzle; box (128 bytes, box_rows slots, R, 1, 1)
// with R = every region when a box spans a whole stage (box_rows == the stage's
// token rows) or the kernel stages small pages box-major (all_regions), else 1.
// With the region dim after the slot dim a box of every region lands region-major
// in shared memory, [region][slot][128 B]: a whole-stage box is the stage layout
// every split kernel reads; a box-major stage is a run of such boxes, one per page.
// The strides need not increase with the dim index (the region stride is 128 bytes,
// the slot stride a whole row); dims of one index take any stride.
fdec_status encode_kv_map(CUtensorMap* map, const fdec_kv_desc& d, int head_dim, int page_size, int hk,
                          int box_rows, int stage_rows, int eb, bool all_regions) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return fail(FDEC_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int regions = head_dim * eb / 128;
    auto stride_of = [](uint64_t size, int64_t stride_bytes) -> cuuint64_t {
        return (size == 1 && stride_bytes == 0) ? 16 : static_cast<cuuint64_t>(stride_bytes);
    };
    cuuint64_t gdim[5] = {static_cast<cuuint64_t>(128 / eb), static_cast<cuuint64_t>(page_size),
                          static_cast<cuuint64_t>(regions), static_cast<cuuint64_t>(hk),
                          static_cast<cuuint64_t>(d.num_pages)};
    cuuint64_t gstride[4] = {stride_of(page_size, d.stride_token * eb), 128,
                             stride_of(hk, d.stride_head * eb), stride_of(d.num_pages, d.stride_page * eb)};
    if (regions == 1) gstride[1] = 16;  // a single region: any stride
    cuuint32_t box[5] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows),
                         static_cast<cuuint32_t>((box_rows == stage_rows || all_regions) ? regions : 1), 1, 1};
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 5,
                     const_cast<void*>(d.base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FDEC_ERR_LAYOUT, "cuTensorMapEncodeTiled rejected the K/V layout (error " + std::to_string(r) + ")");
    return FDEC_OK;
}

bool same_desc(const fdec_kv_desc& a, const fdec_kv_desc& b) {
    return a.base == b.base && a.num_pages == b.num_pages && a.stride_page == b.stride_page &&
           a.stride_head == b.stride_head && a.stride_token == b.stride_token;
}

void log_plan(const fdec_plan_s* p) {
    const char* env = std::getenv("FDEC_LOG");
    if (env == nullptr || env[0] == '0') return;
    int max_s = 0;
    for (int s : p->splits) max_s = std::max(max_s, s);
    std::fprintf(stderr,
                 "[fdec] plan: batch=%d q_len=%d Hq=%d Hk=%d D=%d P=%d rows=%d path=%s rc=%d row_groups=%d "
                 "blocks_per_split=%d items=%zu max_splits=%d reduce_passes=%zu sms=%d ctas/sm=%d "
                 "workspace=%zu B\n",
                 p->batch, p->q_len, p->hq, p->hk, p->head_dim, p->page_size, p->rows,
                 p->path == FDEC_PATH_TC ? "tc" : (p->path == FDEC_PATH_MMA ? "mma" : "simt"), p->rc, p->row_groups, p->blocks_per_split,
                 p->items.size(), max_s, p->passes.size(), p->num_sms, p->ctas_per_sm, p->ws_bytes);
}

}  // namespace

// AUTO takes the tcgen05 kernel above this many rows (q_len x group): measured per
// head_dim, the 16-row kernel is faster at 16 rows everywhere and, at head_dim 256,
// still at 32 rows (102 against 120 us); the tcgen05 kernel from 32 rows below 256
// and from 64 at 256.
static int tc_min_rows(int head_dim) { return head_dim >= 256 ? 32 : kMmaRows; }

// A tiny decode: one query token, at most 4 query rows per KV head, head_dim up to
// 128, every sequence within 5 blocks of 64 tokens and at most one (sequence, KV
// head) pair per SM.  Measured on GB300 (f16, page 16; graph-replayed µs per call
// after an L2 eviction, the SIMT kernel against the tensor-core one): 4.3-8.8
// against 6.4-9.9 at head_dim 64 and 6.6-10.6 against 7.8-12.0 at head_dim 128
// over 64 and 300 tokens, batches 1 and 4, 1 and 8 KV heads; at 1000 tokens and
// more, or 8 rows, the tensor-core kernel wins or ties.
static bool tiny_decode(const int32_t* seq_lens_host, int batch, int q_len, int rows, int num_kv_heads,
                        int head_dim, int num_sms) {
    if (q_len != 1 || rows > 4 || head_dim > 128 || static_cast<long long>(batch) * num_kv_heads > num_sms)
        return false;
    for (int b = 0; b < batch; ++b)
        if (seq_lens_host[b] > 5 * kBlockTokens) return false;
    return true;
}

extern "C" {

const char* fdec_last_error(void) { return g_last_error.c_str(); }

const char* fdec_version(void) { return "fdec 0.1.0 (sm_103a)"; }

fdec_status fdec_plan(const int32_t* seq_lens_host, int batch, int q_len, int page_size, int num_qo_heads,
                      int num_kv_heads, int head_dim, fdec_dtype dtype, int causal, const fdec_plan_opts* opts,
                      fdec_plan_t* out_plan, size_t* workspace_bytes) {
    g_last_error.clear();
    if (out_plan == nullptr || workspace_bytes == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null output pointer");
    *out_plan = nullptr;
    *workspace_bytes = 0;
    if (batch < 1 || seq_lens_host == nullptr) return fail(FDEC_ERR_INVALID_ARG, "batch must be >= 1 with seq_lens");
    if (q_len < 1) return fail(FDEC_ERR_INVALID_ARG, "q_len must be >= 1");
    if (num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0)
        return fail(FDEC_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads");
    if (dtype != FDEC_F16 && dtype != FDEC_BF16) return fail(FDEC_ERR_INVALID_ARG, "dtype must be FDEC_F16 or FDEC_BF16");
    if (!head_dim_supported(head_dim))
        return fail(FDEC_ERR_UNSUPPORTED, "head_dim must be one of 64, 128, 192, 256, 512");
    const int pshift = ilog2_exact(page_size);
    if (page_size < 1 || page_size > 256 || pshift < 0)
        return fail(FDEC_ERR_UNSUPPORTED, "page_size must be a power of two in [1, 256]");
    fdec_plan_opts o{};
    if (opts != nullptr) o = *opts;
    if (o.blocks_per_split < 0 || o.reducer_fanin < 0 || o.num_sms < 0 || (o.reducer_fanin == 1))
        return fail(FDEC_ERR_INVALID_ARG, "invalid plan options");
    if (o.path != FDEC_PATH_AUTO && o.path != FDEC_PATH_SIMT && o.path != FDEC_PATH_MMA && o.path != FDEC_PATH_TC)
        return fail(FDEC_ERR_INVALID_ARG, "invalid path option");
    if (o.kv_dtype != FDEC_KV_SAME && o.kv_dtype != FDEC_KV_E4M3 && o.kv_dtype != FDEC_KV_Q8_0)
        return fail(FDEC_ERR_INVALID_ARG, "kv_dtype must be FDEC_KV_SAME, FDEC_KV_E4M3 or FDEC_KV_Q8_0");
    const bool q8 = o.kv_dtype == FDEC_KV_Q8_0;
    const bool kv8 = o.kv_dtype == FDEC_KV_E4M3 || q8;
    if (kv8 && !split_mma_kv8_supported(head_dim))
        return fail(FDEC_ERR_UNSUPPORTED, "E4M3 and q8_0 caches support head_dim 128 and 256");
    if (kv8 && o.path != FDEC_PATH_AUTO && o.path != FDEC_PATH_MMA)
        return fail(FDEC_ERR_UNSUPPORTED, "E4M3 and q8_0 caches run on the MMA path only");
    const bool mma_ok = head_dim_supported(head_dim);  // every supported head_dim
    const bool tc_ok = split_tc_supported(head_dim);
    if (o.path == FDEC_PATH_MMA && !mma_ok)
        return fail(FDEC_ERR_UNSUPPORTED, "the tensor-core path supports head_dim 64, 128, 192, 256 and 512");
    if (o.path == FDEC_PATH_TC && !tc_ok)
        return fail(FDEC_ERR_UNSUPPORTED, "the tcgen05 path supports head_dim 64, 128, 192 and 256");
    const long long rows_ll = static_cast<long long>(q_len) * (num_qo_heads / num_kv_heads);
    if (rows_ll > (1 << 24)) return fail(FDEC_ERR_UNSUPPORTED, "q_len x group too large");
    for (int b = 0; b < batch; ++b)
        if (seq_lens_host[b] < 0) return fail(FDEC_ERR_INVALID_ARG, "negative sequence capacity");

    int num_sms = o.num_sms;
    if (num_sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail_cuda(e, "querying the SM count (pass opts.num_sms to plan without a device)");
        }
    }

    fdec_plan_s* p = new (std::nothrow) fdec_plan_s();
    if (p == nullptr) return fail(FDEC_ERR_INVALID_ARG, "out of host memory");
    p->batch = batch;
    p->q_len = q_len;
    p->page_size = page_size;
    p->page_shift = pshift;
    p->hq = num_qo_heads;
    p->hk = num_kv_heads;
    p->head_dim = head_dim;
    p->group = num_qo_heads / num_kv_heads;
    p->rows = static_cast<int>(rows_ll);
    p->dtype = dtype;
    p->kv8 = kv8;
    p->q8 = q8;
    p->causal = (causal != 0 && q_len > 1) ? 1 : 0;
    // The warp-level tensor-core kernel by default (every head_dim; see
    // split_mma_kernel.cuh for why tensor cores pay off even when bandwidth-bound);
    // the tcgen05 kernel once the rows need more than one 16-row group (the 16-row
    // kernel would stream K/V once per group); E4M3 and q8_0 caches always on the
    // former.  The fp32 SIMT kernel on request, and for tiny decodes (see
    // tiny_decode): its shorter prologue (no tensor maps, stage barriers or unit
    // counter) wins while a call is one short pass over a few pages.
    if (kv8)
        p->path = FDEC_PATH_MMA;
    else if (o.path == FDEC_PATH_AUTO)
        p->path = tiny_decode(seq_lens_host, batch, q_len, static_cast<int>(rows_ll), num_kv_heads, head_dim, num_sms)
                      ? FDEC_PATH_SIMT
                      : (tc_ok && p->rows > tc_min_rows(head_dim)) ? FDEC_PATH_TC
                                                                    : (mma_ok ? FDEC_PATH_MMA : FDEC_PATH_SIMT);
    else
        p->path = o.path;
    p->persistent = p->path == FDEC_PATH_MMA && !kv8 && split_mma_persist_supported(head_dim);
    p->num_sms = num_sms;
    p->fanin = o.reducer_fanin > 0 ? o.reducer_fanin : 1024;
    size_t smem = 0;
    int threads = 0;
    if (p->path == FDEC_PATH_TC) {
        // Two 128-row tiles per CTA share each staged K/V block once there are more than 128 rows
        // (where tensor memory holds two tiles' S/P buffers and O: head_dim up to 128).
        const int tiles = (p->rows > kTcRows && split_tc_max_tiles(head_dim) == 2) ? 2 : 1;
        p->rc = kTcRows * tiles;
        smem = split_tc_smem_bytes(tiles, head_dim);
        threads = split_tc_threads(tiles, dtype == FDEC_BF16);
    } else if (p->path == FDEC_PATH_MMA) {
        p->rc = kMmaRows;
        smem = q8 ? split_mma_q8_smem_bytes(head_dim) : split_mma_smem_bytes(head_dim, kv8);
        threads = q8 ? split_mma_q8_threads(head_dim) : split_mma_threads(head_dim, kv8);
    } else {
        p->rc = std::min(next_pow2(p->rows), split_max_rc(head_dim));
        smem = split_smem_bytes(head_dim, p->rc);
        threads = split_threads(head_dim);
    }
    p->row_groups = (p->rows + p->rc - 1) / p->rc;
    if (p->row_groups > 65535 || num_kv_heads > 65535) {
        delete p;
        return fail(FDEC_ERR_UNSUPPORTED, "q_len x group / rows per CTA or num_kv_heads above 65535");
    }
    p->ctas_per_sm = p->persistent ? split_mma_persist_ctas_per_sm(head_dim)
                                   : std::max(1, std::min(static_cast<int>(233472 / (smem + 1024)), 2048 / threads));

    p->capacity.assign(seq_lens_host, seq_lens_host + batch);
    std::vector<int> nblocks(batch);
    for (int b = 0; b < batch; ++b) {
        nblocks[b] = std::max(1, (p->capacity[b] + kBlockTokens - 1) / kBlockTokens);
        p->max_pages_needed = std::max(p->max_pages_needed, (p->capacity[b] + page_size - 1) / page_size);
    }
    const int copies = p->hk * p->row_groups;
    const int slots = num_sms * p->ctas_per_sm;
    // A block unit streams 64 tokens of K and V (64 x D x 2 x element bytes) at 1/slots of the
    // machine's bandwidth.
    const double kv_bytes_per_token = head_dim * 2.0 * (kv8 ? 1.0 : 2.0);
    const double partial_cost = 2.0 * p->hk * static_cast<double>(p->rows) * (4.0 * head_dim + 8.0) /
                                (64.0 * kv_bytes_per_token * slots);
    p->blocks_per_split = o.blocks_per_split > 0 ? o.blocks_per_split
                                                 : choose_blocks_per_split(nblocks, copies, slots, partial_cost);
    const int C = p->blocks_per_split;

    // Work items and level-0 partial slots: runs of C blocks.
    p->splits.resize(batch);
    std::vector<int> slot_base(batch, -1);
    size_t next_slot = 0;
    for (int b = 0; b < batch; ++b) {
        const int ns = (nblocks[b] + C - 1) / C;
        p->splits[b] = ns;
        if (ns > 1) {
            slot_base[b] = static_cast<int>(next_slot);
            next_slot += ns;
        }
        for (int k = 0; k < ns; ++k) {
            WorkItem it;
            it.seq = b;
            it.block_begin = k * C;
            it.block_end = std::min((k + 1) * C, nblocks[b]);
            it.slot = ns > 1 ? slot_base[b] + k : -1;
            p->items.push_back(it);
        }
    }
    // Longest items first: the hardware hands out CTAs roughly in index order.
    std::stable_sort(p->items.begin(), p->items.end(), [](const WorkItem& a, const WorkItem& b) {
        return (a.block_end - a.block_begin) > (b.block_end - b.block_begin);
    });
    p->slots_a = next_slot;
    p->n_units = static_cast<int>(p->items.size()) * p->hk * p->row_groups;
    p->persist_grid = std::min(p->n_units, num_sms * p->ctas_per_sm);

    // Reduction passes: level l merges groups of `fanin` slots; levels alternate
    // between region A (even) and region B (odd).
    std::vector<int> n_cur(batch), base_cur(slot_base);
    for (int b = 0; b < batch; ++b) n_cur[b] = p->splits[b] > 1 ? p->splits[b] : 1;
    size_t max_b = 0;
    for (int level = 0;; ++level) {
        std::vector<ReduceTask> tasks;
        size_t next_base = 0;
        std::vector<int> n_next(batch, 1), base_next(batch, -1);
        for (int b = 0; b < batch; ++b) {
            if (n_cur[b] <= 1) continue;
            const int groups = (n_cur[b] + p->fanin - 1) / p->fanin;
            if (groups > 1) {
                base_next[b] = static_cast<int>(next_base);
                next_base += groups;
            }
            n_next[b] = groups;
            for (int gi = 0; gi < groups; ++gi) {
                ReduceTask t;
                t.seq = b;
                t.src = base_cur[b] + gi * p->fanin;
                t.count = std::min(p->fanin, n_cur[b] - gi * p->fanin);
                t.dst = groups > 1 ? base_next[b] + gi : -1;
                tasks.push_back(t);
            }
        }
        if (tasks.empty()) break;
        if (level % 2 == 0)
            max_b = std::max(max_b, next_base);
        else
            p->slots_a = std::max(p->slots_a, next_base);
        p->passes.push_back(std::move(tasks));
        n_cur = n_next;
        base_cur = base_next;
    }
    p->slots_b = max_b;

    // Workspace layout: metadata first (uploaded), partial regions after.
    size_t off = 0;
    p->off_err = off;
    p->off_ticket = off + 8;  // the persistent kernel's unit counter (uint64)
    off = align_up(off + 16);
    p->off_cap = off;
    off = align_up(off + sizeof(int32_t) * batch);
    p->off_items = off;
    off = align_up(off + sizeof(WorkItem) * p->items.size());
    for (const auto& t : p->passes) {
        p->off_tasks.push_back(off);
        off = align_up(off + sizeof(ReduceTask) * t.size());
    }
    p->meta_bytes = off;
    const size_t per_slot_o = static_cast<size_t>(p->hk) * p->rows * head_dim * sizeof(float);
    const size_t per_slot_ml = static_cast<size_t>(p->hk) * p->rows * sizeof(float2);
    p->off_a_o = off;
    off = align_up(off + per_slot_o * p->slots_a);
    p->off_a_ml = off;
    off = align_up(off + per_slot_ml * p->slots_a);
    p->off_b_o = off;
    off = align_up(off + per_slot_o * p->slots_b);
    p->off_b_ml = off;
    off = align_up(off + per_slot_ml * p->slots_b);
    p->ws_bytes = off;

    p->meta.assign(p->meta_bytes, 0);
    std::memcpy(p->meta.data() + p->off_cap, p->capacity.data(), sizeof(int32_t) * batch);
    std::memcpy(p->meta.data() + p->off_items, p->items.data(), sizeof(WorkItem) * p->items.size());
    for (size_t i = 0; i < p->passes.size(); ++i)
        std::memcpy(p->meta.data() + p->off_tasks[i], p->passes[i].data(), sizeof(ReduceTask) * p->passes[i].size());

    log_plan(p);
    *out_plan = p;
    *workspace_bytes = p->ws_bytes;
    return FDEC_OK;
}

fdec_status fdec_plan_destroy(fdec_plan_t plan) {
    delete plan;
    return FDEC_OK;
}

fdec_status fdec_plan_get_info(fdec_plan_t p, fdec_plan_info* info) {
    if (p == nullptr || info == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null argument");
    std::memset(info, 0, sizeof(*info));
    info->path = p->path;
    info->blocks_per_split = p->blocks_per_split;
    info->num_items = static_cast<int>(p->items.size());
    info->num_split_ctas = p->persistent ? p->persist_grid : static_cast<int>(p->items.size()) * p->hk * p->row_groups;
    info->row_groups = p->row_groups;
    info->rows_per_group = p->rc;
    for (int s : p->splits) info->max_splits = std::max(info->max_splits, s);
    info->reduce_passes = static_cast<int>(p->passes.size());
    info->launches = 1 + static_cast<int>(p->passes.size());
    info->num_sms = p->num_sms;
    info->workspace_bytes = p->ws_bytes;
    return FDEC_OK;
}

fdec_status fdec_plan_get_splits(fdec_plan_t p, int32_t* splits, int batch) {
    if (p == nullptr || splits == nullptr || batch != p->batch) return fail(FDEC_ERR_INVALID_ARG, "bad arguments");
    std::memcpy(splits, p->splits.data(), sizeof(int32_t) * batch);
    return FDEC_OK;
}

fdec_status fdec_plan_set_split_event(fdec_plan_t p, cudaEvent_t event) {
    if (p == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null plan");
    p->split_event = event;
    return FDEC_OK;
}

fdec_status fdec_plan_upload(fdec_plan_t p, void* workspace, cudaStream_t stream) {
    g_last_error.clear();
    if (p == nullptr || workspace == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null plan or workspace");
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0)
        return fail(FDEC_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone)
        return fail(FDEC_ERR_CAPTURING, "fdec_plan_upload must not run while the stream is capturing");
    // Set the split kernel's shared-memory attribute here, outside any capture.
    SplitParams none{};
    e = dispatch_split(p, none, dim3(1, 1, 1), stream, false);
    if (e == cudaSuccess && p->persistent) e = dispatch_split(p, none, dim3(1, 1, 1), stream, false, true);
    if (e != cudaSuccess) return fail_cuda(e, "preparing the split kernel");
    e = cudaMemcpyAsync(workspace, p->meta.data(), p->meta_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return fail_cuda(e, "uploading the plan");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail_cuda(e, "uploading the plan");
    p->uploaded = workspace;
    return FDEC_OK;
}

fdec_status fdec_read_device_errors(fdec_plan_t p, void* workspace, uint32_t* flags, int clear, cudaStream_t stream) {
    if (p == nullptr || workspace == nullptr || flags == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null argument");
    uint32_t v = 0;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaError_t e = cudaMemcpyAsync(&v, ws + p->off_err, sizeof(v), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws + p->off_err, 0, sizeof(v), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail_cuda(e, "reading the device error word");
    *flags = v;
    return FDEC_OK;
}

fdec_status fdec_run(fdec_plan_t p, const void* q, int64_t q_stride_tok, int64_t q_stride_head, fdec_kv_desc k,
                     fdec_kv_desc v, const int32_t* page_table, int64_t page_table_stride,
                     const int32_t* seq_lens_dev, float scale, float* out, float* lse, void* workspace,
                     cudaStream_t stream) {
    return fdec_run_scaled(p, q, q_stride_tok, q_stride_head, k, v, page_table, page_table_stride, seq_lens_dev, scale,
                           1.f, 1.f, out, lse, workspace, stream);
}

// fdec_run_scaled and fdec_run_q8_0 (ks / vs: the q8_0 block-scale pools, else null).
static fdec_status run_impl(fdec_plan_t p, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                            const fdec_kv_desc& k, const fdec_kv_desc& v, const fdec_kv_desc* ks,
                            const fdec_kv_desc* vs, const int32_t* page_table, int64_t page_table_stride,
                            const int32_t* seq_lens_dev, float scale, float k_scale, float v_scale, float* out,
                            float* lse, void* workspace, cudaStream_t stream) {
    if (q == nullptr || k.base == nullptr || v.base == nullptr || page_table == nullptr || seq_lens_dev == nullptr ||
        out == nullptr)
        return fail(FDEC_ERR_INVALID_ARG, "null q, K, V, page_table, seq_lens or out");
    if (k.num_pages < 1 || v.num_pages < 1) return fail(FDEC_ERR_INVALID_ARG, "K and V pools need at least one page");
    if (k.num_pages > INT32_MAX || v.num_pages > INT32_MAX) return fail(FDEC_ERR_INVALID_ARG, "too many pages");
    if (page_table_stride < p->max_pages_needed)
        return fail(FDEC_ERR_CAPACITY, "page_table_stride is smaller than ceil(capacity / page_size)");
    if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale) ||
        !std::isfinite(scale * k_scale * 1.4426950408889634074f))
        return fail(FDEC_ERR_INVALID_ARG, "scale, k_scale and v_scale must be finite");
    const int eb = p->kv8 ? 1 : 2;  // bytes per stored K/V element
    const int64_t stride_unit = 16 / eb;
    const fdec_kv_desc* descs[2] = {&k, &v};
    for (const fdec_kv_desc* d : descs) {
        if (reinterpret_cast<uintptr_t>(d->base) % 16 != 0)
            return fail(FDEC_ERR_LAYOUT, "K/V base must be 16-byte aligned");
        if (d->stride_page % stride_unit != 0 || d->stride_head % stride_unit != 0 ||
            d->stride_token % stride_unit != 0)
            return fail(FDEC_ERR_LAYOUT, "K/V strides must be multiples of 16 bytes");
        if (d->stride_page < 0 || d->stride_head < 0 || d->stride_token < 0)
            return fail(FDEC_ERR_LAYOUT, "negative K/V stride");
    }
    if (reinterpret_cast<uintptr_t>(q) % 2 != 0 || reinterpret_cast<uintptr_t>(out) % 4 != 0 ||
        (lse != nullptr && reinterpret_cast<uintptr_t>(lse) % 4 != 0))
        return fail(FDEC_ERR_LAYOUT, "misaligned q, out or lse");
    if (workspace == nullptr || workspace != p->uploaded)
        return fail(FDEC_ERR_WORKSPACE, "workspace is not the buffer this plan was uploaded to");

    if (p->page_size >= 8 && !(p->maps_valid && same_desc(p->map_k, k) && same_desc(p->map_v, v))) {
        const int stage_rows = p->path == FDEC_PATH_TC ? kTcStageTokens : kStageTokens;
        const int box_rows = std::min(p->page_size, stage_rows);
        const bool all_regions = p->path == FDEC_PATH_MMA && split_mma_box_major(p->head_dim, p->kv8);
        fdec_status st =
            encode_kv_map(&p->tmap_k, k, p->head_dim, p->page_size, p->hk, box_rows, stage_rows, eb, all_regions);
        if (st == FDEC_OK)
            st = encode_kv_map(&p->tmap_v, v, p->head_dim, p->page_size, p->hk, box_rows, stage_rows, eb, all_regions);
        if (st != FDEC_OK) {
            p->maps_valid = false;
            return st;
        }
        p->map_k = k;
        p->map_v = v;
        p->maps_valid = true;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    SplitParams sp;
    sp.q = static_cast<const uint16_t*>(q);
    sp.q_stride_tok = q_stride_tok;
    sp.q_stride_head = q_stride_head;
    sp.k_base = static_cast<const uint8_t*>(k.base);
    sp.k_pages = k.num_pages;
    sp.k_sp = k.stride_page * eb;
    sp.k_sh = k.stride_head * eb;
    sp.k_st = k.stride_token * eb;
    sp.v_base = static_cast<const uint8_t*>(v.base);
    sp.v_pages = v.num_pages;
    sp.v_sp = v.stride_page * eb;
    sp.v_sh = v.stride_head * eb;
    sp.v_st = v.stride_token * eb;
    sp.ks_base = sp.vs_base = nullptr;
    sp.ks_sp = sp.ks_sh = sp.ks_st = sp.vs_sp = sp.vs_sh = sp.vs_st = 0;
    if (ks != nullptr && vs != nullptr) {  // binary16 elements -> bytes; page ids must fit every pool
        sp.ks_base = static_cast<const uint8_t*>(ks->base);
        sp.ks_sp = ks->stride_page * 2;
        sp.ks_sh = ks->stride_head * 2;
        sp.ks_st = ks->stride_token * 2;
        sp.vs_base = static_cast<const uint8_t*>(vs->base);
        sp.vs_sp = vs->stride_page * 2;
        sp.vs_sh = vs->stride_head * 2;
        sp.vs_st = vs->stride_token * 2;
        sp.k_pages = std::min(sp.k_pages, ks->num_pages);
        sp.v_pages = std::min(sp.v_pages, vs->num_pages);
    }
    sp.page_table = page_table;
    sp.pt_stride = page_table_stride;
    sp.seq_lens = seq_lens_dev;
    sp.capacity = reinterpret_cast<const int32_t*>(ws + p->off_cap);
    sp.items = reinterpret_cast<const WorkItem*>(ws + p->off_items);
    sp.part_o = reinterpret_cast<float*>(ws + p->off_a_o);
    sp.part_ml = reinterpret_cast<float2*>(ws + p->off_a_ml);
    sp.out = out;
    sp.lse = lse;
    sp.err = reinterpret_cast<unsigned*>(ws + p->off_err);
    sp.q_len = p->q_len;
    sp.hq = p->hq;
    sp.hk = p->hk;
    sp.group = p->group;
    sp.rows = p->rows;
    sp.page_shift = p->page_shift;
    sp.causal = p->causal;
    sp.scale_log2 = scale * k_scale * 1.4426950408889634074f;
    sp.v_scale = v_scale;
    sp.n_units = p->n_units;
    sp.ticket = reinterpret_cast<unsigned long long*>(ws + p->off_ticket);
    sp.seq1_bps = p->batch == 1 ? p->blocks_per_split : 0;
    sp.seq1_blocks = std::max(1, (p->capacity[0] + kBlockTokens - 1) / kBlockTokens);
    sp.seq1_capacity = p->capacity[0];

    // The persistent kernel copies each unit's query rows with 16-byte bulk copies.
    const bool q_rows_aligned = reinterpret_cast<uintptr_t>(q) % 16 == 0 && (q_stride_tok * 2) % 16 == 0 &&
                                (q_stride_head * 2) % 16 == 0;
    const dim3 grid(static_cast<unsigned>(p->items.size()), static_cast<unsigned>(p->hk),
                    static_cast<unsigned>(p->row_groups));
    cudaError_t e = dispatch_split(p, sp, grid, stream, true, p->persistent && q_rows_aligned);
    if (e != cudaSuccess) return fail_cuda(e, "launching the split kernel");
    if (p->split_event != nullptr) {
        e = cudaEventRecord(p->split_event, stream);
        if (e != cudaSuccess) return fail_cuda(e, "recording the split event");
    }

    for (size_t level = 0; level < p->passes.size(); ++level) {
        ReduceParams rp;
        const bool from_a = (level % 2 == 0);
        rp.tasks = reinterpret_cast<const ReduceTask*>(ws + p->off_tasks[level]);
        rp.src_o = reinterpret_cast<const float*>(ws + (from_a ? p->off_a_o : p->off_b_o));
        rp.src_ml = reinterpret_cast<const float2*>(ws + (from_a ? p->off_a_ml : p->off_b_ml));
        rp.src_lse = nullptr;
        rp.dst_o = reinterpret_cast<float*>(ws + (from_a ? p->off_b_o : p->off_a_o));
        rp.dst_ml = reinterpret_cast<float2*>(ws + (from_a ? p->off_b_ml : p->off_a_ml));
        rp.out = out;
        rp.lse = lse;
        rp.hk = p->hk;
        rp.rows = p->rows;
        rp.group = p->group;
        rp.q_len = p->q_len;
        rp.hq = p->hq;
        rp.head_dim = p->head_dim;
        rp.normalized_input = 0;
        rp.src_rows_stride = p->rows;
        int max_count = 1;
        for (const ReduceTask& t : p->passes[level]) max_count = std::max(max_count, t.count);
        rp.warps_per_unit = reduce_warps_per_unit(max_count);
        e = launch_reduce(rp, static_cast<int>(p->passes[level].size()), stream);
        if (e != cudaSuccess) return fail_cuda(e, "launching the reduction");
    }
    return FDEC_OK;
}

fdec_status fdec_run_scaled(fdec_plan_t p, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                            fdec_kv_desc k, fdec_kv_desc v, const int32_t* page_table, int64_t page_table_stride,
                            const int32_t* seq_lens_dev, float scale, float k_scale, float v_scale, float* out,
                            float* lse, void* workspace, cudaStream_t stream) {
    g_last_error.clear();
    if (p == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null plan");
    if (p->q8) return fail(FDEC_ERR_INVALID_ARG, "q8_0 plans run through fdec_run_q8_0 (it takes the block scales)");
    return run_impl(p, q, q_stride_tok, q_stride_head, k, v, nullptr, nullptr, page_table, page_table_stride,
                    seq_lens_dev, scale, k_scale, v_scale, out, lse, workspace, stream);
}

fdec_status fdec_run_q8_0(fdec_plan_t p, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                          fdec_kv_desc k, fdec_kv_desc k_scales, fdec_kv_desc v, fdec_kv_desc v_scales,
                          const int32_t* page_table, int64_t page_table_stride, const int32_t* seq_lens_dev,
                          float scale, float* out, float* lse, void* workspace, cudaStream_t stream) {
    g_last_error.clear();
    if (p == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null plan");
    if (!p->q8) return fail(FDEC_ERR_INVALID_ARG, "fdec_run_q8_0 needs a plan made with kv_dtype FDEC_KV_Q8_0");
    const int64_t row = p->head_dim / 32;  // binary16 scales per (page, head, slot)
    const fdec_kv_desc* descs[2] = {&k_scales, &v_scales};
    for (const fdec_kv_desc* d : descs) {
        if (d->base == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null q8_0 scale pool");
        if (d->num_pages < 1 || d->num_pages > INT32_MAX)
            return fail(FDEC_ERR_INVALID_ARG, "q8_0 scale pools need 1 .. 2^31 - 1 pages");
        if (reinterpret_cast<uintptr_t>(d->base) % (2 * row) != 0)
            return fail(FDEC_ERR_LAYOUT, "q8_0 scale pool base must be aligned to head_dim / 16 bytes");
        if (d->stride_page < 0 || d->stride_head < 0 || d->stride_token < 0 || d->stride_page % row != 0 ||
            d->stride_head % row != 0 || d->stride_token % row != 0)
            return fail(FDEC_ERR_LAYOUT, "q8_0 scale strides must be non-negative multiples of head_dim / 32");
    }
    return run_impl(p, q, q_stride_tok, q_stride_head, k, v, &k_scales, &v_scales, page_table, page_table_stride,
                    seq_lens_dev, scale, 1.f, 1.f, out, lse, workspace, stream);
}

}  // extern "C"

namespace {

// Both appends: K/V elements of eb bytes (2: the 16-bit cache types, 1: E4M3 codes).
fdec_status append_impl(const void* k_new, const void* v_new, int64_t new_stride_tok, int64_t new_stride_head,
                        const int32_t* batch_indices, const int32_t* positions, int n_tokens, int num_kv_heads,
                        int head_dim, int page_size, const fdec_kv_desc& k, const fdec_kv_desc& v,
                        const int32_t* page_table, int batch, int64_t page_table_stride, uint32_t* device_errors,
                        cudaStream_t stream, int eb) {
    g_last_error.clear();
    if (n_tokens < 0 || num_kv_heads < 1 || batch < 1 || page_table_stride < 1)
        return fail(FDEC_ERR_INVALID_ARG, "need n_tokens >= 0, num_kv_heads >= 1, batch >= 1, page_table_stride >= 1");
    if (!head_dim_supported(head_dim))
        return fail(FDEC_ERR_UNSUPPORTED, "head_dim must be one of 64, 128, 192, 256, 512");
    const int pshift = ilog2_exact(page_size);
    if (page_size < 1 || page_size > 256 || pshift < 0)
        return fail(FDEC_ERR_UNSUPPORTED, "page_size must be a power of two in [1, 256]");
    if (n_tokens == 0) return FDEC_OK;
    if (k_new == nullptr || v_new == nullptr || batch_indices == nullptr || positions == nullptr ||
        page_table == nullptr || k.base == nullptr || v.base == nullptr)
        return fail(FDEC_ERR_INVALID_ARG, "null pointer");
    if (k.num_pages < 1 || v.num_pages < 1 || k.num_pages > INT32_MAX || v.num_pages > INT32_MAX)
        return fail(FDEC_ERR_INVALID_ARG, "K and V pools need 1 .. 2^31-1 pages");
    const int64_t unit = 16 / eb;  // elements per 16 bytes
    const fdec_kv_desc* descs[2] = {&k, &v};
    for (const fdec_kv_desc* d : descs) {
        if (reinterpret_cast<uintptr_t>(d->base) % 16 != 0)
            return fail(FDEC_ERR_LAYOUT, "K/V base must be 16-byte aligned");
        if (d->stride_page % unit != 0 || d->stride_head % unit != 0 || d->stride_token % unit != 0 ||
            d->stride_page < 0 || d->stride_head < 0 || d->stride_token < 0)
            return fail(FDEC_ERR_LAYOUT, "K/V strides must be non-negative multiples of 16 bytes");
    }
    if (reinterpret_cast<uintptr_t>(k_new) % 16 != 0 || reinterpret_cast<uintptr_t>(v_new) % 16 != 0 ||
        new_stride_tok % unit != 0 || new_stride_head % unit != 0 || new_stride_tok < 0 || new_stride_head < 0)
        return fail(FDEC_ERR_LAYOUT, "new K/V rows must start on 16-byte boundaries");
    AppendParams ap;
    ap.k_new = static_cast<const uint8_t*>(k_new);
    ap.v_new = static_cast<const uint8_t*>(v_new);
    ap.new_st = new_stride_tok * eb;
    ap.new_sh = new_stride_head * eb;
    ap.batch_indices = batch_indices;
    ap.positions = positions;
    ap.page_table = page_table;
    ap.pt_stride = page_table_stride;
    ap.k_base = static_cast<uint8_t*>(const_cast<void*>(k.base));
    ap.k_pages = k.num_pages;
    ap.k_sp = k.stride_page * eb;
    ap.k_sh = k.stride_head * eb;
    ap.k_st = k.stride_token * eb;
    ap.v_base = static_cast<uint8_t*>(const_cast<void*>(v.base));
    ap.v_pages = v.num_pages;
    ap.v_sp = v.stride_page * eb;
    ap.v_sh = v.stride_head * eb;
    ap.v_st = v.stride_token * eb;
    ap.err = device_errors;
    ap.n_tokens = n_tokens;
    ap.batch = batch;
    ap.hk = num_kv_heads;
    ap.row_bytes = head_dim * eb;
    ap.page_shift = pshift;
    const cudaError_t e = launch_append(ap, stream);
    if (e != cudaSuccess) return fail_cuda(e, "launching the append");
    return FDEC_OK;
}

}  // namespace

extern "C" {

fdec_status fdec_append(const void* k_new, const void* v_new, int64_t new_stride_tok, int64_t new_stride_head,
                        const int32_t* batch_indices, const int32_t* positions, int n_tokens, int num_kv_heads,
                        int head_dim, int page_size, fdec_kv_desc k, fdec_kv_desc v, const int32_t* page_table,
                        int batch, int64_t page_table_stride, uint32_t* device_errors, cudaStream_t stream) {
    return append_impl(k_new, v_new, new_stride_tok, new_stride_head, batch_indices, positions, n_tokens,
                       num_kv_heads, head_dim, page_size, k, v, page_table, batch, page_table_stride, device_errors,
                       stream, 2);
}

fdec_status fdec_append_e4m3(const void* k_new, const void* v_new, int64_t new_stride_tok, int64_t new_stride_head,
                             const int32_t* batch_indices, const int32_t* positions, int n_tokens, int num_kv_heads,
                             int head_dim, int page_size, fdec_kv_desc k, fdec_kv_desc v, const int32_t* page_table,
                             int batch, int64_t page_table_stride, uint32_t* device_errors, cudaStream_t stream) {
    return append_impl(k_new, v_new, new_stride_tok, new_stride_head, batch_indices, positions, n_tokens,
                       num_kv_heads, head_dim, page_size, k, v, page_table, batch, page_table_stride, device_errors,
                       stream, 1);
}

fdec_status fdec_merge_states(const float* o, const float* lse, int n_states, int rows, int head_dim, float* o_out,
                              float* lse_out, cudaStream_t stream) {
    if (o == nullptr || lse == nullptr || o_out == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null pointer");
    if (n_states < 1 || rows < 1 || head_dim < 1 || head_dim > 512)
        return fail(FDEC_ERR_INVALID_ARG, "need n_states >= 1, rows >= 1, 1 <= head_dim <= 512");
    if (reinterpret_cast<uintptr_t>(o) % 4 != 0 || reinterpret_cast<uintptr_t>(lse) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(o_out) % 4 != 0 || (lse_out != nullptr && reinterpret_cast<uintptr_t>(lse_out) % 4 != 0))
        return fail(FDEC_ERR_LAYOUT, "misaligned float arrays");
    // One task over all states; the rows are one "KV head" of `rows` rows, and
    // row r is written to output row r (group = rows, q_len = 1, Hq = rows).
    ReduceParams rp;
    rp.tasks = nullptr;
    rp.src_o = o;
    rp.src_ml = nullptr;
    rp.src_lse = lse;
    rp.dst_o = nullptr;
    rp.dst_ml = nullptr;
    rp.out = o_out;
    rp.lse = lse_out;
    rp.hk = 1;
    rp.rows = rows;
    rp.group = rows;
    rp.q_len = 1;
    rp.hq = rows;
    rp.head_dim = head_dim;
    rp.normalized_input = 1;
    rp.src_rows_stride = rows;
    rp.warps_per_unit = reduce_warps_per_unit(n_states);
    ReduceTask single;
    single.seq = 0;
    single.src = 0;
    single.count = n_states;
    single.dst = -1;
    cudaError_t e = launch_reduce_single(rp, single, stream);
    if (e != cudaSuccess) return fail_cuda(e, "launching the merge");
    return FDEC_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// A run that allocates nothing, not even a caller-owned workspace.
//
// Some callers cannot allocate device memory at all: a plug-in loaded into a
// host program whose memory pool owns the whole device, or a latency-critical
// loop where a cudaMalloc (which may synchronise the device) is not allowed.
// For them the partials and work lists live in one fixed array compiled into
// this library.  Every GPU that loads the library keeps the array until the
// process exits.
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;  // 16 MiB

__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_static_mutex;
void* g_static_address[64] = {};  // device address of the array, per device

}  // namespace

extern "C" fdec_status fdec_run_static_workspace(fdec_plan_t p, const void* q, int64_t q_stride_tok,
                                                 int64_t q_stride_head, fdec_kv_desc k, fdec_kv_desc v,
                                                 const int32_t* page_table, int64_t page_table_stride,
                                                 const int32_t* seq_lens_dev, float scale, float* out, float* lse,
                                                 cudaStream_t stream) {
    if (p == nullptr) return fail(FDEC_ERR_INVALID_ARG, "null plan");
    if (p->ws_bytes > kStaticWorkspaceBytes)
        return fail(FDEC_ERR_WORKSPACE, "this plan needs " + std::to_string(p->ws_bytes) +
                                            " bytes of workspace but the built-in array holds " +
                                            std::to_string(kStaticWorkspaceBytes) +
                                            "; use fdec_run with a workspace of your own");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(FDEC_ERR_UNSUPPORTED, "device index above 63");
    void* ws = nullptr;
    {
        // Once per device, with that device current: the array's device address.
        // In host code the array's name is only a host-side stand-in.
        std::lock_guard<std::mutex> lock(g_static_mutex);
        if (g_static_address[dev] == nullptr) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_static_workspace);
            if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress of the built-in workspace");
            g_static_address[dev] = addr;
        }
        ws = g_static_address[dev];
    }
    // The work lists and capacities go in front; the device error word at the
    // start of this image is zero, so every call starts with a clear word.
    // The partials need no clearing: each is written before it is read.
    e = cudaMemcpyAsync(ws, p->meta.data(), p->meta_bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return fail_cuda(e, "copying the plan into the built-in workspace");
    // fdec_run checks the workspace against the plan's uploaded buffer: point
    // that at the array for this call only, then give the caller's back.
    void* saved = p->uploaded;
    p->uploaded = ws;
    const fdec_status st = fdec_run(p, q, q_stride_tok, q_stride_head, k, v, page_table, page_table_stride,
                                    seq_lens_dev, scale, out, lse, ws, stream);
    p->uploaded = saved;
    return st;
}
