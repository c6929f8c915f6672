// split_tc.cu -- instantiations of the tcgen05 dense-query split kernel (head_dim 128;
// one or two 128-row query tiles per CTA).
#include "split_tc_kernel.cuh"

namespace fdec {

cudaError_t launch_split_tc(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int tiles, bool bf16,
                            dim3 grid, cudaStream_t s, bool launch) {
    if (tiles == 1)
        return bf16 ? launch_split_tc_one<1, true>(p, tk, tv, grid, s, launch)
                    : launch_split_tc_one<1, false>(p, tk, tv, grid, s, launch);
    if (tiles == 2)
        return bf16 ? launch_split_tc_one<2, true>(p, tk, tv, grid, s, launch)
                    : launch_split_tc_one<2, false>(p, tk, tv, grid, s, launch);
    return cudaErrorInvalidValue;
}

size_t split_tc_smem_bytes(int tiles) { return tiles == 1 ? TcLayout<1>::SMEM : TcLayout<2>::SMEM; }
int split_tc_threads(int tiles) { return tiles == 1 ? TcLayout<1>::THREADS : TcLayout<2>::THREADS; }

}  // namespace fdec
