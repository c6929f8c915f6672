// split_mma_q8.cu -- instantiations of the tensor-core split kernel over q8_0
// caches (int8 codes in blocks of 32 along head_dim, one binary16 scale per block),
// head_dim 128 and 256.
#include "split_mma_kernel.cuh"

namespace fdec {

cudaError_t launch_split_mma_q8(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                                bool bf16, dim3 grid, cudaStream_t s, bool launch) {
    switch (head_dim) {
        case 128:
            return bf16 ? launch_split_mma_one<128, true, true, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_one<128, false, true, true>(p, tk, tv, grid, s, launch);
        case 256:
            return bf16 ? launch_split_mma_one<256, true, true, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_one<256, false, true, true>(p, tk, tv, grid, s, launch);
        default:
            return cudaErrorInvalidValue;
    }
}

size_t split_mma_q8_smem_bytes(int head_dim) {
    return head_dim == 128 ? MmaLayout<128, true, true>::SMEM : head_dim == 256 ? MmaLayout<256, true, true>::SMEM : 0;
}

int split_mma_q8_threads(int head_dim) {
    return head_dim == 128 ? MmaLayout<128, true, true>::THREADS : MmaLayout<256, true, true>::THREADS;
}

}  // namespace fdec
