// split_d256.cu -- split-kernel instantiations for head_dim 256.
#include "split_kernel.cuh"

namespace fdec {

cudaError_t launch_split_d256(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rc,
                               bool bf16, dim3 grid, cudaStream_t s, bool launch) {
    return launch_split_d<256>(p, tk, tv, rc, bf16, grid, s, launch);
}

}  // namespace fdec
