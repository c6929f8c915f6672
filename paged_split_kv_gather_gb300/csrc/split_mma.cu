// split_mma.cu -- instantiations of the tensor-core split kernel (head_dim 64, 128,
// 192, 256, 512 over 16-bit caches; 128 and 256 over E4M3 caches).
#include "split_mma_kernel.cuh"

namespace fdec {

cudaError_t launch_split_mma(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int head_dim,
                             bool bf16, bool kv8, dim3 grid, cudaStream_t s, bool launch) {
    if (kv8) {
        switch (head_dim) {
            case 128:
                return bf16 ? launch_split_mma_one<128, true, true>(p, tk, tv, grid, s, launch)
                            : launch_split_mma_one<128, false, true>(p, tk, tv, grid, s, launch);
            case 256:
                return bf16 ? launch_split_mma_one<256, true, true>(p, tk, tv, grid, s, launch)
                            : launch_split_mma_one<256, false, true>(p, tk, tv, grid, s, launch);
            default:
                return cudaErrorInvalidValue;
        }
    }
    switch (head_dim) {
        case 64:
            return bf16 ? launch_split_mma_one<64, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_one<64, false>(p, tk, tv, grid, s, launch);
        case 128:
            return bf16 ? launch_split_mma_one<128, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_one<128, false>(p, tk, tv, grid, s, launch);
        case 192:
            return bf16 ? launch_split_mma_one<192, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_one<192, false>(p, tk, tv, grid, s, launch);
        case 256:
            return bf16 ? launch_split_mma_one<256, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_one<256, false>(p, tk, tv, grid, s, launch);
        case 512:
            return bf16 ? launch_split_mma_one<512, true>(p, tk, tv, grid, s, launch)
                        : launch_split_mma_one<512, false>(p, tk, tv, grid, s, launch);
        default:
            return cudaErrorInvalidValue;
    }
}

size_t split_mma_smem_bytes(int head_dim, bool kv8) {
    if (kv8) {
        switch (head_dim) {
            case 128: return MmaLayout<128, true>::SMEM;
            case 256: return MmaLayout<256, true>::SMEM;
            default: return 0;
        }
    }
    switch (head_dim) {
        case 64: return MmaLayout<64>::SMEM;
        case 128: return MmaLayout<128>::SMEM;
        case 192: return MmaLayout<192>::SMEM;
        case 256: return MmaLayout<256>::SMEM;
        case 512: return MmaLayout<512>::SMEM;
        default: return 0;
    }
}

int split_mma_threads(int head_dim, bool kv8) {
    if (kv8) {
        switch (head_dim) {
            case 128: return MmaLayout<128, true>::THREADS;
            case 256: return MmaLayout<256, true>::THREADS;
            default: return 0;
        }
    }
    switch (head_dim) {
        case 64: return MmaLayout<64>::THREADS;
        case 128: return MmaLayout<128>::THREADS;
        case 192: return MmaLayout<192>::THREADS;
        case 256: return MmaLayout<256>::THREADS;
        case 512: return MmaLayout<512>::THREADS;
        default: return 0;
    }
}

}  // namespace fdec
