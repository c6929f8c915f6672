// e2e_loop.cu -- end-to-end timing of fdec_run from C, with no Python in the loop.
//
// One step is what a C caller of the library does per decode step: copy the
// step's inputs from pinned host memory to the device (q, the page table and
// the lengths; one cudaMemcpyAsync per buffer), call fdec_run, copy out and lse
// back to pinned host memory (one cudaMemcpyAsync each) and synchronise the
// stream.  The K/V cache stays resident on the device.  Host wall-clock time
// over `iters` steps (after `warmup` untimed ones) is returned in *seconds.
// This file is a benchmark helper, built next to the library; it is not part
// of the library's ABI.
#include <time.h>

#include <cuda_runtime.h>

#include "../../include/fdec.h"

namespace {

double now_s() {
    timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return static_cast<double>(ts.tv_sec) + 1e-9 * static_cast<double>(ts.tv_nsec);
}

}  // namespace

extern "C" int fdec_e2e_loop(fdec_plan_t plan, const void* h_q, void* d_q, size_t q_bytes, int64_t q_stride_tok,
                             int64_t q_stride_head, fdec_kv_desc k, fdec_kv_desc v, const int32_t* h_table,
                             int32_t* d_table, size_t table_bytes, int64_t table_stride, const int32_t* h_lens,
                             int32_t* d_lens, size_t lens_bytes, float scale, float* d_out, float* h_out,
                             size_t out_bytes, float* d_lse, float* h_lse, size_t lse_bytes, void* workspace,
                             cudaStream_t stream, int warmup, int iters, double* seconds) {
    double t0 = 0.0;
    for (int i = 0; i < warmup + iters; ++i) {
        if (i == warmup) {
            if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
            t0 = now_s();
        }
        if (cudaMemcpyAsync(d_q, h_q, q_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return -2;
        if (cudaMemcpyAsync(d_table, h_table, table_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return -2;
        if (cudaMemcpyAsync(d_lens, h_lens, lens_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return -2;
        const fdec_status st = fdec_run(plan, d_q, q_stride_tok, q_stride_head, k, v, d_table, table_stride, d_lens,
                                        scale, d_out, d_lse, workspace, stream);
        if (st != FDEC_OK) return static_cast<int>(st);
        if (cudaMemcpyAsync(h_out, d_out, out_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return -3;
        if (d_lse != nullptr && cudaMemcpyAsync(h_lse, d_lse, lse_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return -3;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return -4;
    }
    *seconds = (now_s() - t0) / (iters > 0 ? iters : 1);
    return 0;
}
