// split_tc.cu -- instantiations of the tcgen05 dense-query split kernel for
// head_dim 64 and 128 (one or two 128-row query tiles per CTA), and the dispatch
// over every head_dim it is built for.
#include "split_tc_kernel.cuh"

namespace fdec {

cudaError_t launch_split_tc_wide(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                                 bool bf16, dim3 grid, cudaStream_t s, bool launch);
size_t split_tc_wide_smem_bytes(int head_dim);

cudaError_t launch_split_tc(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int tiles, int head_dim,
                            bool bf16, dim3 grid, cudaStream_t s, bool launch) {
    if (head_dim == 192 || head_dim == 256) {
        if (tiles != 1) return cudaErrorInvalidValue;
        return launch_split_tc_wide(p, tk, tv, head_dim, bf16, grid, s, launch);
    }
    if (head_dim == 64) {
        if (tiles == 1)
            return bf16 ? launch_split_tc_one<1, 64, true>(p, tk, tv, grid, s, launch)
                        : launch_split_tc_one<1, 64, false>(p, tk, tv, grid, s, launch);
        if (tiles == 2)
            return bf16 ? launch_split_tc_one<2, 64, true>(p, tk, tv, grid, s, launch)
                        : launch_split_tc_one<2, 64, false>(p, tk, tv, grid, s, launch);
    }
    if (head_dim == 128) {
        if (tiles == 1)
            return bf16 ? launch_split_tc_one<1, 128, true>(p, tk, tv, grid, s, launch)
                        : launch_split_tc_one<1, 128, false>(p, tk, tv, grid, s, launch);
        if (tiles == 2)
            return bf16 ? launch_split_tc_one<2, 128, true>(p, tk, tv, grid, s, launch)
                        : launch_split_tc_one<2, 128, false>(p, tk, tv, grid, s, launch);
    }
    return cudaErrorInvalidValue;
}

size_t split_tc_smem_bytes(int tiles, int head_dim) {
    switch (head_dim) {
        case 64: return tiles == 1 ? TcLayout<1, 64>::SMEM : TcLayout<2, 64>::SMEM;
        case 128: return tiles == 1 ? TcLayout<1, 128>::SMEM : TcLayout<2, 128>::SMEM;
        case 192:
        case 256: return split_tc_wide_smem_bytes(head_dim);
        default: return 0;
    }
}

int split_tc_threads(int tiles, bool bf16) {
    if (bf16) return tiles == 1 ? TcLayout<1, 128, true>::THREADS : TcLayout<2, 128, true>::THREADS;
    return tiles == 1 ? TcLayout<1, 128>::THREADS : TcLayout<2, 128>::THREADS;
}

}  // namespace fdec
