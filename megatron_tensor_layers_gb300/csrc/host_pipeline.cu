// tp_mlp_forward_host: the tensor-parallel MLP for activations that live in
// (pinned) host memory, with the copies overlapped with the compute.
//
// The n tokens are cut into row blocks.  Block i is copied to the device on
// `copy_stream`, the MLP of block i runs on `stream` once its copy has landed
// (an event), and its output is copied back on `copy_stream` once the MLP is
// done (another event).  All input copies are queued first in order, so the
// copy of block i+1 runs under the compute of block i and the read-back of
// block i under the compute of block i+1; only the first input copy and the
// last read-back are exposed.  So with two or more chunks the first and the
// last block are short, about n/(4*chunks) rows, and the rows between them
// form chunks-1 blocks: n = 8192 in 2 chunks runs as 1024, 6144 and 1024
// rows.  An MLP row costs far more than copying it (8192 x 28672 weights:
// about 0.8 us of compute against under 0.1 us of copy), so a short block
// still hides the next, tall block's copy.  Rows are independent in every
// step of the MLP (page "6.2 Tensor-parallel inference", §1: each token's
// output depends on its own row of X only), so splitting by rows changes no
// result.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "tp.h"

namespace {

constexpr int kMaxBlocks = 65;   // chunks <= 64: at most chunks + 1 blocks

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Row-block boundaries: block b covers rows [s[b], s[b + 1]).  Returns the block
// count (0 for n = 0).  Edges are rounded up to a multiple of 128 rows (the
// GEMMs' tile height) where the rows between them stay at least as many, and
// middle blocks where the last of them keeps rows.
int host_blocks(int64_t n, int chunks, int64_t* s) {
    s[0] = 0;
    if (n <= 0) return 0;
    if (chunks == 1 || n < 3) {
        s[1] = n;
        return 1;
    }
    int64_t e = (n + 4 * chunks - 1) / (4 * chunks);
    if (3 * round_up(e, 128) <= n) e = round_up(e, 128);   // the rows between keep at least an edge's height
    const int64_t m = n - 2 * e;                    // >= 1: e <= ceil(n / 8) < n / 2 for n >= 3
    const int mb = chunks - 1;
    int64_t mr = (m + mb - 1) / mb;
    if (round_up(mr, 128) * (mb - 1) < m) mr = round_up(mr, 128);
    int k = 0;
    s[++k] = e;
    for (int64_t r = e; r < n - e;) {
        r = std::min(r + mr, n - e);
        s[++k] = r;
    }
    s[++k] = n;
    return k;
}

}  // namespace

extern "C" int tp_mlp_host_blocks(int64_t n, int chunks, int64_t* starts, int max_blocks) {
    if (n < 0 || chunks < 1 || chunks > 64) return -1;
    int64_t s[kMaxBlocks + 1];
    const int k = host_blocks(n, chunks, s);
    if (starts != nullptr && max_blocks >= k)
        for (int b = 0; b <= k; ++b) starts[b] = s[b];
    return k;
}

extern "C" tp_status tp_mlp_forward_host(int t, int64_t n, int64_t h, int64_t f, const void* x_host,
                                         const void* const* w_gate_up, const void* const* w_down, int64_t ld_down,
                                         const void* bias_down, tp_act act, tp_reduce_mode mode,
                                         tp_dtype partial_dtype, void* x_dev, void* workspace,
                                         size_t workspace_bytes, void* y_dev, void* y_host, tp_dtype y_dtype,
                                         int chunks, tp_stream stream, tp_stream copy_stream) {
    if (chunks < 1 || chunks > 64 || n < 0 || h <= 0) return TP_ERR_INVALID_ARG;
    if (n > 0 && (x_host == nullptr || y_host == nullptr || x_dev == nullptr || y_dev == nullptr))
        return TP_ERR_INVALID_ARG;
    if (y_dtype != TP_BF16 && y_dtype != TP_F32) return TP_ERR_UNSUPPORTED;
    if (n == 0)   // nothing to copy or compute: the MLP entry point checks the other arguments
        return tp_mlp_forward(t, 0, h, f, x_dev, h, w_gate_up, w_down, ld_down, bias_down, act, mode, partial_dtype,
                              workspace, workspace_bytes, y_dev, y_dtype, stream);
    int64_t bounds[kMaxBlocks + 1];
    const int nblk = host_blocks(n, chunks, bounds);
    auto start = [&](int b) -> int64_t { return bounds[b]; };
    int64_t rows = 0;                                          // the tallest block
    for (int b = 0; b < nblk; ++b) rows = std::max(rows, bounds[b + 1] - bounds[b]);
    // The workspace must hold the tallest block's MLP; validate the arguments
    // with it before anything is queued.
    const size_t need = tp_mlp_workspace_size(t, rows, h, f, mode, partial_dtype);
    if (need == 0) return TP_ERR_INVALID_ARG;
    if (workspace_bytes < need) return TP_ERR_WORKSPACE;
    const size_t xrow = static_cast<size_t>(h) * 2;
    const size_t yrow = static_cast<size_t>(h) * (y_dtype == TP_F32 ? 4 : 2);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t cp = reinterpret_cast<cudaStream_t>(copy_stream);

    cudaEvent_t in_ready[kMaxBlocks], out_ready[kMaxBlocks];
    int created = 0;
    tp_status st = TP_OK;
    for (; created < nblk; ++created) {
        if (cudaEventCreateWithFlags(&in_ready[created], cudaEventDisableTiming) != cudaSuccess) {
            st = TP_ERR_CUDA;
            break;
        }
        if (cudaEventCreateWithFlags(&out_ready[created], cudaEventDisableTiming) != cudaSuccess) {
            cudaEventDestroy(in_ready[created]);
            st = TP_ERR_CUDA;
            break;
        }
    }
    // every input copy first, in order, each followed by its event
    for (int b = 0; b < nblk && st == TP_OK; ++b) {
        const int64_t r0 = start(b), nr = start(b + 1) - r0;
        if (cudaMemcpyAsync(static_cast<char*>(x_dev) + r0 * xrow, static_cast<const char*>(x_host) + r0 * xrow,
                            nr * xrow, cudaMemcpyHostToDevice, cp) != cudaSuccess ||
            cudaEventRecord(in_ready[b], cp) != cudaSuccess)
            st = TP_ERR_CUDA;
    }
    // compute block b once its input is on the device; read it back once computed
    for (int b = 0; b < nblk && st == TP_OK; ++b) {
        const int64_t r0 = start(b), nr = start(b + 1) - r0;
        if (cudaStreamWaitEvent(cs, in_ready[b], 0) != cudaSuccess) {
            st = TP_ERR_CUDA;
            break;
        }
        st = tp_mlp_forward(t, nr, h, f, static_cast<char*>(x_dev) + r0 * xrow, h, w_gate_up, w_down, ld_down,
                            bias_down, act, mode, partial_dtype, workspace, workspace_bytes,
                            static_cast<char*>(y_dev) + r0 * yrow, y_dtype, stream);
        if (st != TP_OK) break;
        if (cudaEventRecord(out_ready[b], cs) != cudaSuccess || cudaStreamWaitEvent(cp, out_ready[b], 0) != cudaSuccess ||
            cudaMemcpyAsync(static_cast<char*>(y_host) + r0 * yrow, static_cast<char*>(y_dev) + r0 * yrow, nr * yrow,
                            cudaMemcpyDeviceToHost, cp) != cudaSuccess)
            st = TP_ERR_CUDA;
    }
    // the compute stream ends after the last read-back, so callers can wait on it alone
    if (st == TP_OK && nblk > 0) {
        if (cudaEventRecord(in_ready[0], cp) != cudaSuccess || cudaStreamWaitEvent(cs, in_ready[0], 0) != cudaSuccess)
            st = TP_ERR_CUDA;
    }
    for (int b = 0; b < created; ++b) {   // released once their pending work completes
        cudaEventDestroy(in_ready[b]);
        cudaEventDestroy(out_ready[b]);
    }
    return st;
}
