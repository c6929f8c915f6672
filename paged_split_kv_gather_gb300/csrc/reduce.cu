// reduce.cu -- the log-sum-exp reduction of attention partials.
//
// One CTA of eight warps per (KV head, query row, 32 head_dim elements) and
// task; a task merges `count` consecutive partial slots of one sequence.  Every
// warp strides over the partials to find the running max M (so any number of
// partials works, unlike a reducer that gives one lane to each partial and
// stops at 32); warp w then accumulates partials w, w + 8, ... (weight
// exp2(m_k - M), one element per lane, eight loads in flight), and the eight
// warp sums are added in shared memory.  The result is either one partial of the next level
// (hierarchical passes when a sequence has more partials than the fan-in) or
// the final out = O / L and lse = ln 2 * (M + log2 L).
//
// The same kernel merges caller-given normalised (o, lse) states for
// fdec_merge_states: there m_k = lse_k * log2(e) and l_k = 1.
#include <cmath>

#include "device_utils.cuh"
#include "fdec_internal.h"

namespace fdec {

constexpr int kReduceWarps = 8;

// (m in log2 units, l) of source row idx.
__device__ __forceinline__ float2 source_ml(const ReduceParams& p, int64_t idx) {
    constexpr float kLog2e = 1.4426950408889634074f;
    if (p.normalized_input) return make_float2(p.src_lse[idx] * kLog2e, 1.f);
    return p.src_ml[idx];
}

__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(const ReduceParams p, int num_tasks,
                                                                   ReduceTask single) {
    constexpr float kLn2 = 0.69314718055994530942f;
    __shared__ float s_acc[kReduceWarps][32];
    __shared__ float s_l[kReduceWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int chunks = (p.head_dim + 31) / 32;
    const int unit = blockIdx.x / chunks;  // (kv head, row)
    const int d = (blockIdx.x - unit * chunks) * 32 + lane;  // this lane's head_dim element
    const int kvh = unit / p.rows;
    const int row = unit - kvh * p.rows;
    const int D = p.head_dim;
    // Launched as a programmatic dependent of the split kernel: everything above
    // overlaps its tail; wait here until its partials are complete and visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    for (int ti = blockIdx.y; ti < num_tasks; ti += gridDim.y) {
        const ReduceTask task = p.tasks != nullptr ? p.tasks[ti] : single;
        const int64_t base = (static_cast<int64_t>(task.src) * p.hk + kvh) * p.src_rows_stride + row;
        const int64_t step = static_cast<int64_t>(p.hk) * p.src_rows_stride;

        float M = -INFINITY;
        for (int k = lane; k < task.count; k += 32) M = fmaxf(M, source_ml(p, base + k * step).x);
        M = warp_max(M);

        float Lw = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll 8
            for (int k = warp; k < task.count; k += kReduceWarps) {
                const int64_t idx = base + k * step;
                const float2 ml = source_ml(p, idx);
                const float o = d < D ? p.src_o[idx * D + d] : 0.f;
                const float w = ml.x == -INFINITY ? 0.f : exp2_approx(ml.x - M);
                Lw += w * ml.y;
                acc += w * o;
            }
        }
        s_acc[warp][lane] = acc;
        if (lane == 0) s_l[warp] = Lw;
        __syncthreads();
        if (warp == 0 && d < D) {
            float Lsum = 0.f, o = 0.f;
#pragma unroll
            for (int w = 0; w < kReduceWarps; ++w) {
                Lsum += s_l[w];
                o += s_acc[w][lane];
            }
            if (task.dst < 0) {
                const int qi = row / p.group;
                const int h = kvh * p.group + (row - qi * p.group);
                const int64_t orow = static_cast<int64_t>(task.seq * p.q_len + qi) * p.hq + h;
                p.out[orow * D + d] = Lsum > 0.f ? o / Lsum : 0.f;
                if (d == 0 && p.lse != nullptr) p.lse[orow] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
            } else {
                const int64_t drow = (static_cast<int64_t>(task.dst) * p.hk + kvh) * p.rows + row;
                p.dst_o[drow * D + d] = o;
                if (d == 0) p.dst_ml[drow] = make_float2(M, Lsum);
            }
        }
        __syncthreads();  // s_acc and s_l are reused by the next task
    }
}

cudaError_t launch_reduce(const ReduceParams& p, int num_tasks, cudaStream_t s) {
    if (num_tasks <= 0) return cudaSuccess;
    const int units = p.hk * p.rows * ((p.head_dim + 31) / 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units, num_tasks < 65535 ? num_tasks : 65535, 1);
    cfg.blockDim = dim3(kReduceWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reduce_kernel, p, num_tasks, ReduceTask{0, 0, 0, -1});
}

cudaError_t launch_reduce_single(const ReduceParams& p, ReduceTask task, cudaStream_t s) {
    const int units = p.hk * p.rows * ((p.head_dim + 31) / 32);
    dim3 grid(units, 1, 1);
    reduce_kernel<<<grid, kReduceWarps * 32, 0, s>>>(p, 1, task);
    return cudaGetLastError();
}

}  // namespace fdec
