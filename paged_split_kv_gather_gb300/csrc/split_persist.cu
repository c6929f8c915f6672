// split_persist.cu -- instantiations of the persistent tensor-core split kernel
// (16-bit caches, every head_dim).
#include "split_persist_kernel.cuh"

namespace fdec {

cudaError_t launch_split_mma_persist(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                                     bool bf16, dim3 grid, cudaStream_t s, bool launch) {
    switch (head_dim) {
        case 64:
            return bf16 ? launch_split_mma_persist_one<64, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_persist_one<64, false>(p, tk, tv, grid, s, launch);
        case 128:
            return bf16 ? launch_split_mma_persist_one<128, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_persist_one<128, false>(p, tk, tv, grid, s, launch);
        case 192:
            return bf16 ? launch_split_mma_persist_one<192, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_persist_one<192, false>(p, tk, tv, grid, s, launch);
        case 256:
            return bf16 ? launch_split_mma_persist_one<256, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_persist_one<256, false>(p, tk, tv, grid, s, launch);
        case 512:
            return bf16 ? launch_split_mma_persist_one<512, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_persist_one<512, false>(p, tk, tv, grid, s, launch);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace fdec
