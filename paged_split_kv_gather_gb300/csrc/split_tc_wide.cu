// split_tc_wide.cu -- instantiations of the tcgen05 dense-query split kernel for
// head_dim 192 and 256: one 128-row query tile per CTA (the S/P buffers and an O
// of 192 or 256 columns fill the 512 tensor-memory columns of one CTA).
#include "split_tc_kernel.cuh"

namespace fdec {

cudaError_t launch_split_tc_wide(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                                 bool bf16, dim3 grid, cudaStream_t s, bool launch) {
    if (head_dim == 192)
        return bf16 ? launch_split_tc_one<1, 192, true>(p, tk, tv, grid, s, launch)
                    : launch_split_tc_one<1, 192, false>(p, tk, tv, grid, s, launch);
    if (head_dim == 256)
        return bf16 ? launch_split_tc_one<1, 256, true>(p, tk, tv, grid, s, launch)
                    : launch_split_tc_one<1, 256, false>(p, tk, tv, grid, s, launch);
    return cudaErrorInvalidValue;
}

size_t split_tc_wide_smem_bytes(int head_dim) {
    return head_dim == 192 ? TcLayout<1, 192>::SMEM : TcLayout<1, 256>::SMEM;
}

}  // namespace fdec
