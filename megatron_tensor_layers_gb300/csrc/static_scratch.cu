// tp_mlp_forward_static: the tensor-parallel MLP forward for callers that
// cannot hand the library a device workspace.
//
// tp_mlp_forward needs a scratch buffer (the intermediate H and, unless the
// reduce is fused, the t partial sums) that the caller allocates.  Some
// callers cannot do that: a host application that loads this library as a
// plugin and owns the whole device memory pool may forbid its plugins from
// calling cudaMalloc so that its accounting stays exact, and a
// latency-critical decode loop cannot afford cudaMalloc/cudaFree on its path,
// because they can synchronise the whole device and stall every stream.
//
// This file gives such callers one entry point that allocates nothing.  Its
// scratch is a file-scope array in the library's device image.  CUDA loads a
// module's device image lazily, so the array comes into being on a GPU when
// the library's module is first loaded there, which at the latest is this
// entry point's first call on that device (its cudaGetSymbolAddress below);
// from then on the GPU holds it until the process exits.  Loading the module
// is a driver-side reservation that can synchronise the device and can fail
// when the device's memory is already taken, so a caller makes the first
// call at start-up, outside its latency-critical loop and before any stream
// capture.  The array is TP_STATIC_SCRATCH_BYTES (16 MiB) long, enough for
// decode-sized batches: e.g. 64 tokens of a Llama-3.1-70B-shaped MLP
// (h=8192, f=28672) at t=4 with fp32 partials needs 12.1 MB.  Larger requests
// are refused with TP_ERR_WORKSPACE before anything is launched.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "kernels.h"
#include "tp.h"

namespace {

static_assert(TP_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// The shared scratch.  Host code must not use this name as an address: on the
// host it is only a stand-in symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_tp_static_scratch[TP_STATIC_SCRATCH_BYTES];

// Device address of the scratch on the current device, looked up once per
// device (the first call on that device does it) and cached.  Two host
// threads making their first call on one device at once both look it up and
// store the same address; the relaxed atomics keep that race well defined.
void* static_scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    static std::atomic<void*> cache[64];
    void* cached = cache[dev].load(std::memory_order_relaxed);
    if (cached == nullptr) {
        if (cudaGetSymbolAddress(&cached, g_tp_static_scratch) != cudaSuccess || cached == nullptr) return nullptr;
        cache[dev].store(cached, std::memory_order_relaxed);
    }
    return cached;
}

}  // namespace

extern "C" tp_status tp_mlp_forward_static(int t, int64_t n, int64_t h, int64_t f, const void* x, int64_t ldx,
                                           const void* const* w_gate_up, const void* const* w_down,
                                           int64_t ld_down, const void* bias_down, tp_act act,
                                           tp_reduce_mode mode, tp_dtype partial_dtype, void* y, tp_dtype y_dtype,
                                           tp_stream stream) {
    // What tp_mlp_forward requires (H and the partials); the optional areas of
    // a fused reduce (the stream-K slots, the one-kernel path's slice
    // partials) are used only if they fit as well.
    const size_t need = tpk::mlp_workspace_required(t, n, h, f, mode, partial_dtype);
    if (need > static_cast<size_t>(TP_STATIC_SCRATCH_BYTES)) return TP_ERR_WORKSPACE;
    if (need == 0) {
        // Invalid arguments, or nothing to compute: let the regular entry
        // point's host-side checks answer, without touching the device.
        return tp_mlp_forward(t, n, h, f, x, ldx, w_gate_up, w_down, ld_down, bias_down, act, mode, partial_dtype,
                              nullptr, 0, y, y_dtype, stream);
    }
    void* scratch = static_scratch_address();
    if (scratch == nullptr) return TP_ERR_CUDA;
    // Every byte of the scratch that this call reads is first written by this
    // call (H by the gate_up GEMM, each partial by the GEMM that produces it),
    // so nothing needs clearing between calls.
    return tp_mlp_forward(t, n, h, f, x, ldx, w_gate_up, w_down, ld_down, bias_down, act, mode, partial_dtype,
                          scratch, TP_STATIC_SCRATCH_BYTES, y, y_dtype, stream);
}
