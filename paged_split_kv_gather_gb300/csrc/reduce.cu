// reduce.cu -- the log-sum-exp reduction of attention partials.
//
// One CTA of four warps; each (KV head, query row, 32 head_dim elements) unit
// of a task gets `warps_per_unit` (1, 2 or 4) of them, chosen by the host from
// the task's partial count, so that a few partials per row do not leave warps
// idle.  A task merges `count` consecutive partial slots of one sequence.  Warp
// w of a unit takes partials w, w + wpu, ... (any number: no fixed 32-block
// scratch), 20 at a time with all their loads in flight together (one element
// per lane), and keeps a running (max, sum, accumulator) merged by log-sum-exp,
// so one round trip to memory serves up to 20 x wpu partials.  The warp states
// of a unit are merged in shared memory.  The result is either one partial of
// the next level (hierarchical passes when a sequence has more partials than
// the fan-in) or the final out = O / L and lse = ln 2 * (M + log2 L).
//
// The CTA is sized to sit beside two CTAs of the persistent split kernel on one
// SM (128 threads at <= 96 registers: the 12,288 registers those two leave free),
// so that, launched as a programmatic dependent, every reduction CTA is resident
// and past its prologue when the split grid completes.  (Measured: with 256-thread
// CTAs of 78 registers, which do not fit there, the CTAs that had to wait for an
// SM to empty made a 61-partial reduction 1.6 us slower.)
//
// The same kernel merges caller-given normalised (o, lse) states for
// fdec_merge_states: there m_k = lse_k * log2(e) and l_k = 1.
#include <cmath>

#include "device_utils.cuh"
#include "fdec_internal.h"

namespace fdec {

constexpr int kReduceWarps = 4;
constexpr int kReducePerWarp = 20;

// (m in log2 units, l) of source row idx.
__device__ __forceinline__ float2 source_ml(const ReduceParams& p, int64_t idx) {
    constexpr float kLog2e = 1.4426950408889634074f;
    if (p.normalized_input) return make_float2(p.src_lse[idx] * kLog2e, 1.f);
    return p.src_ml[idx];
}

__global__ void __launch_bounds__(kReduceWarps * 32, 5) reduce_kernel(const ReduceParams p, int num_tasks,
                                                                   ReduceTask single) {
    constexpr float kLn2 = 0.69314718055994530942f;
    constexpr int U = kReducePerWarp;  // partials per warp per round trip
    __shared__ float s_acc[kReduceWarps][32];
    __shared__ float s_m[kReduceWarps];
    __shared__ float s_l[kReduceWarps];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int wpu = p.warps_per_unit;
    const int ww = warp % wpu;  // warp within its unit
    const int chunks = (p.head_dim + 31) / 32;
    const int64_t unit_lin = static_cast<int64_t>(blockIdx.x) * (kReduceWarps / wpu) + warp / wpu;
    const bool active = unit_lin < static_cast<int64_t>(p.hk) * p.rows * chunks;
    const int64_t unit = unit_lin / chunks;  // (kv head, row)
    const int d = static_cast<int>(unit_lin - unit * chunks) * 32 + lane;  // this lane's head_dim element
    const int kvh = static_cast<int>(unit / p.rows);
    const int row = static_cast<int>(unit - static_cast<int64_t>(kvh) * p.rows);
    const int D = p.head_dim;
    // The first task is plan data (not written by the split kernel): read it early.
    ReduceTask task = single;
    if (p.tasks != nullptr && static_cast<int>(blockIdx.y) < num_tasks) task = p.tasks[blockIdx.y];
    // The next kernel in the stream may be scheduled now (a split kernel of the next
    // decode step waits for this one's completion before it reads or writes anything).
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Launched as a programmatic dependent of the split kernel: everything above
    // overlaps its tail; wait here until its partials are complete and visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    for (int ti = blockIdx.y; ti < num_tasks; ti += gridDim.y) {
        if (ti != static_cast<int>(blockIdx.y) && p.tasks != nullptr) task = p.tasks[ti];
        const int64_t base = (static_cast<int64_t>(task.src) * p.hk + kvh) * p.src_rows_stride + row;
        const int64_t step = static_cast<int64_t>(p.hk) * p.src_rows_stride;

        float m_w = -INFINITY, l_w = 0.f, acc = 0.f;
        for (int k0 = ww; active && k0 < task.count; k0 += wpu * U) {
            float2 ml[U];
            float o[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = k0 + u * wpu;
                ml[u] = make_float2(-INFINITY, 0.f);
                o[u] = 0.f;
                if (k < task.count) {
                    const int64_t idx = base + k * step;
                    ml[u] = source_ml(p, idx);
                    if (d < D) o[u] = p.src_o[idx * D + d];
                }
            }
            float mx = m_w;
#pragma unroll
            for (int u = 0; u < U; ++u) mx = fmaxf(mx, ml[u].x);
            if (mx == -INFINITY) continue;  // nothing visible so far (uniform across the warp)
            const float a = exp2_approx(m_w - mx);  // 0 while m_w is -inf
            l_w *= a;
            acc *= a;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float w = ml[u].x == -INFINITY ? 0.f : exp2_approx(ml[u].x - mx);
                l_w += w * ml[u].y;
                acc += w * o[u];
            }
            m_w = mx;
        }
        s_acc[warp][lane] = acc;
        if (lane == 0) {
            s_m[warp] = m_w;
            s_l[warp] = l_w;
        }
        __syncthreads();
        if (active && ww == 0 && d < D) {
            float M = -INFINITY;
            for (int w = warp; w < warp + wpu; ++w) M = fmaxf(M, s_m[w]);
            float Lsum = 0.f, o = 0.f;
            if (M != -INFINITY) {
                for (int w = warp; w < warp + wpu; ++w) {
                    const float e = s_m[w] == -INFINITY ? 0.f : exp2_approx(s_m[w] - M);
                    Lsum += e * s_l[w];
                    o += e * s_acc[w][lane];
                }
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
        __syncthreads();  // the shared arrays are reused by the next task
    }
}

// Warps per unit for tasks of up to `max_count` partials: enough that each warp
// takes at most kReducePerWarp (one round trip), at most all of the CTA's.
int reduce_warps_per_unit(int max_count) {
    int w = 1;
    while (w < kReduceWarps && w * kReducePerWarp < max_count) w *= 2;
    return w;
}

static unsigned reduce_grid_x(const ReduceParams& p) {
    const int64_t units = static_cast<int64_t>(p.hk) * p.rows * ((p.head_dim + 31) / 32);
    const int upc = kReduceWarps / p.warps_per_unit;
    return static_cast<unsigned>((units + upc - 1) / upc);
}

cudaError_t launch_reduce(const ReduceParams& p, int num_tasks, cudaStream_t s) {
    if (num_tasks <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(reduce_grid_x(p), num_tasks < 65535 ? num_tasks : 65535, 1);
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
    dim3 grid(reduce_grid_x(p), 1, 1);
    reduce_kernel<<<grid, kReduceWarps * 32, 0, s>>>(p, 1, task);
    return cudaGetLastError();
}

}  // namespace fdec
