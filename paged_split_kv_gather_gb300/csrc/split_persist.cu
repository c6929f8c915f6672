// split_persist.cu -- instantiations of the persistent tensor-core split kernel
// (16-bit caches, every head_dim), each in two stage layouts: box-major for pages of
// 8 or 16 tokens (one TMA box per page), region-major for every other page size.
#include "split_persist_kernel.cuh"

namespace fdec {

template <int D>
static cudaError_t launch_persist_d(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, bool bf16,
                                   dim3 grid, cudaStream_t s, bool launch) {
    if (!launch) {  // set-up only (plan upload): both layouts' kernel attributes
        cudaError_t e = bf16 ? launch_split_mma_persist_one<D, true, true>(p, tk, tv, grid, s, false)
                             : launch_split_mma_persist_one<D, false, true>(p, tk, tv, grid, s, false);
        if (e != cudaSuccess) return e;
        return bf16 ? launch_split_mma_persist_one<D, true, false>(p, tk, tv, grid, s, false)
                    : launch_split_mma_persist_one<D, false, false>(p, tk, tv, grid, s, false);
    }
    const bool small_pages = p.page_shift == 3 || p.page_shift == 4;  // several TMA boxes per stage
    if (small_pages)
        return bf16 ? launch_split_mma_persist_one<D, true, true>(p, tk, tv, grid, s, true)
                    : launch_split_mma_persist_one<D, false, true>(p, tk, tv, grid, s, true);
    return bf16 ? launch_split_mma_persist_one<D, true, false>(p, tk, tv, grid, s, true)
                : launch_split_mma_persist_one<D, false, false>(p, tk, tv, grid, s, true);
}

cudaError_t launch_split_mma_persist(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                                     bool bf16, dim3 grid, cudaStream_t s, bool launch) {
    switch (head_dim) {
        case 64:
            return launch_persist_d<64>(p, tk, tv, bf16, grid, s, launch);
        case 128:
            return launch_persist_d<128>(p, tk, tv, bf16, grid, s, launch);
        case 192:
            return launch_persist_d<192>(p, tk, tv, bf16, grid, s, launch);
        case 256:
            return launch_persist_d<256>(p, tk, tv, bf16, grid, s, launch);
        case 512:
            return launch_persist_d<512>(p, tk, tv, bf16, grid, s, launch);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace fdec
