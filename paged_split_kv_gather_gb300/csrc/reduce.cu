// reduce.cu -- the log-sum-exp reduction of attention partials.
//
// One warp per (task, KV head, query row).  A task merges `count` consecutive
// partial slots of one sequence.  Lanes first stride over the partials to find
// the running max and the weighted sum of l (so any number of partials works,
// unlike a reducer that gives one lane to each partial and stops at 32), then
// stride over head_dim accumulating exp2(m_k - M) * o_k.  The result is either
// one partial of the next level (hierarchical passes when a sequence has more
// partials than the fan-in) or the final out = O / L and lse = ln 2 * (M + log2 L).
//
// The same kernel merges caller-given normalised (o, lse) states for
// fdec_merge_states: there m_k = lse_k * log2(e) and l_k = 1.
#include <cmath>

#include "device_utils.cuh"
#include "fdec_internal.h"

namespace fdec {

constexpr int kReduceWarps = 4;
constexpr int kMaxDimPerLane = 16;  // head_dim <= 512

// (m in log2 units, l) of source row idx.
__device__ __forceinline__ float2 source_ml(const ReduceParams& p, int64_t idx) {
    constexpr float kLog2e = 1.4426950408889634074f;
    if (p.normalized_input) return make_float2(p.src_lse[idx] * kLog2e, 1.f);
    return p.src_ml[idx];
}

__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(const ReduceParams p, int num_tasks, ReduceTask single) {
    constexpr float kLn2 = 0.69314718055994530942f;
    const int lane = threadIdx.x & 31;
    const int unit = blockIdx.x * kReduceWarps + (threadIdx.x >> 5);  // (kv head, row)
    if (unit >= p.hk * p.rows) return;
    const int kvh = unit / p.rows;
    const int row = unit - kvh * p.rows;
    const int D = p.head_dim;

    for (int ti = blockIdx.y; ti < num_tasks; ti += gridDim.y) {
        const ReduceTask task = p.tasks != nullptr ? p.tasks[ti] : single;
        const int64_t base = (static_cast<int64_t>(task.src) * p.hk + kvh) * p.src_rows_stride + row;
        const int64_t step = static_cast<int64_t>(p.hk) * p.src_rows_stride;

        float M = -INFINITY;
        for (int k = lane; k < task.count; k += 32) {
            M = fmaxf(M, source_ml(p, base + k * step).x);
        }
        M = warp_max(M);

        float Lsum = 0.f;
        float acc[kMaxDimPerLane];
#pragma unroll
        for (int j = 0; j < kMaxDimPerLane; ++j) acc[j] = 0.f;
        if (M != -INFINITY) {
            for (int k = lane; k < task.count; k += 32) {
                const float2 ml = source_ml(p, base + k * step);
                if (ml.x != -INFINITY) Lsum += ml.y * exp2_approx(ml.x - M);
            }
            for (int k = 0; k < task.count; ++k) {
                const int64_t idx = base + k * step;
                const float mk = source_ml(p, idx).x;
                if (mk == -INFINITY) continue;
                const float w = exp2_approx(mk - M);
                const float* src = p.src_o + idx * D;
#pragma unroll
                for (int j = 0; j < kMaxDimPerLane; ++j) {
                    const int d = lane + 32 * j;
                    if (d < D) acc[j] += w * src[d];
                }
            }
        }
        Lsum = warp_sum(Lsum);

        if (task.dst < 0) {
            const int qi = row / p.group;
            const int h = kvh * p.group + (row - qi * p.group);
            const int64_t orow = static_cast<int64_t>(task.seq * p.q_len + qi) * p.hq + h;
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
            for (int j = 0; j < kMaxDimPerLane; ++j) {
                const int d = lane + 32 * j;
                if (d < D) p.out[orow * D + d] = acc[j] * inv;
            }
            if (lane == 0 && p.lse != nullptr) p.lse[orow] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
        } else {
            const int64_t drow = (static_cast<int64_t>(task.dst) * p.hk + kvh) * p.rows + row;
#pragma unroll
            for (int j = 0; j < kMaxDimPerLane; ++j) {
                const int d = lane + 32 * j;
                if (d < D) p.dst_o[drow * D + d] = acc[j];
            }
            if (lane == 0) p.dst_ml[drow] = make_float2(M, Lsum);
        }
    }
}

cudaError_t launch_reduce(const ReduceParams& p, int num_tasks, cudaStream_t s) {
    if (num_tasks <= 0) return cudaSuccess;
    const int units = p.hk * p.rows;
    dim3 grid((units + kReduceWarps - 1) / kReduceWarps, num_tasks < 65535 ? num_tasks : 65535, 1);
    reduce_kernel<<<grid, kReduceWarps * 32, 0, s>>>(p, num_tasks, ReduceTask{0, 0, 0, -1});
    return cudaGetLastError();
}

cudaError_t launch_reduce_single(const ReduceParams& p, ReduceTask task, cudaStream_t s) {
    const int units = p.hk * p.rows;
    dim3 grid((units + kReduceWarps - 1) / kReduceWarps, 1, 1);
    reduce_kernel<<<grid, kReduceWarps * 32, 0, s>>>(p, 1, task);
    return cudaGetLastError();
}

}  // namespace fdec
