// e2e_loop.cu -- end-to-end timing of fdec_run from C, with no Python in the loop.
//
// One step is what a C caller of the library does per decode step: copy the
// step's inputs from pinned host memory to the device, call fdec_run, copy the
// results back to pinned host memory and synchronise the stream.  The caller
// stages the inputs (q, the page table, the lengths) in one pinned buffer laid
// out like one device buffer, so the inputs take one cudaMemcpyAsync, and
// fdec_run writes out and lse into one device buffer, so the results take one
// more: every copy has a fixed cost of its own, whatever its size.  The K/V
// cache stays resident on the device.  Host wall-clock time over `iters` steps
// (after `warmup` untimed ones) is returned in *seconds.  This file is a
// benchmark helper, built next to the library; it is not part of the library's
// ABI.
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

// h_in / d_in: in_bytes of staged inputs; d_q, d_table and d_lens point into d_in.
// d_res / h_res: res_bytes of results; d_out and d_lse point into d_res.
extern "C" int fdec_e2e_loop(fdec_plan_t plan, const void* h_in, void* d_in, size_t in_bytes, const void* d_q,
                             int64_t q_stride_tok, int64_t q_stride_head, fdec_kv_desc k, fdec_kv_desc v,
                             const int32_t* d_table, int64_t table_stride, const int32_t* d_lens, float scale,
                             float* d_out, float* d_lse, const void* d_res, void* h_res, size_t res_bytes,
                             void* workspace, cudaStream_t stream, int warmup, int iters, double* seconds) {
    double t0 = 0.0;
    for (int i = 0; i < warmup + iters; ++i) {
        if (i == warmup) {
            if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
            t0 = now_s();
        }
        if (cudaMemcpyAsync(d_in, h_in, in_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return -2;
        const fdec_status st = fdec_run(plan, d_q, q_stride_tok, q_stride_head, k, v, d_table, table_stride, d_lens,
                                        scale, d_out, d_lse, workspace, stream);
        if (st != FDEC_OK) return static_cast<int>(st);
        if (cudaMemcpyAsync(h_res, d_res, res_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return -3;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return -4;
    }
    *seconds = (now_s() - t0) / (iters > 0 ? iters : 1);
    return 0;
}
