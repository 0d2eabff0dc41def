// The "all-reduce sum" of t in-memory partial buffers, the all-gather of
// vocab-sharded outputs, and the bounded-wait probe used by failure tests.
//
// Shard reduce (page "vLLM source analysis 13: tensor parallelism in
// detail", §1.1.1 Reduce-Scatter, §1.1.2 All-Gather, and the one-shot
// low-latency sum after §1.2).  On one GPU every "rank" buffer is directly
// addressable, so both orders are a single streaming pass: each thread owns
// 16 bytes of every buffer, loads all t of them (t x 128-bit loads in
// flight), folds them in registers and writes the result.
//   DIRECT: fold ranks 0, 1, ..., t-1 with a float32 carry.
//   RING:   the buffer is cut into t chunks of ceil(K/t) elements; chunk c
//           starts at rank c and folds c, c+1, ..., c+t-1 (mod t), exactly
//           the order in which the ring's reduce-scatter steps add the
//           ranks' copies into it; each addition rounds to the hop dtype
//           (a bf16 wire rounds at every hop).  The all-gather phase moves
//           the finished chunks unchanged, so it is the final write (to
//           `out`, and to every rank buffer when replicating).
// The pass is HBM-bound: t*K*b bytes read, K*b (or t*K*b) written.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace tpk {

struct ReduceArgs {
    const void* p[TP_MAX_SHARDS];
    void* out;
    int64_t count;
    int64_t chunk;
    int t;
    int ring;
    int hop_bf16;
    int out_bf16;
    int replicate;
};

__device__ __forceinline__ float round_bf16(float x) { return bf16_to_f32(f32_to_bf16(x)); }

template <bool IN_BF16>
__device__ __forceinline__ float load_elem(const void* p, int64_t e) {
    if (IN_BF16) return bf16_to_f32(static_cast<const uint16_t*>(p)[e]);
    return static_cast<const float*>(p)[e];
}

template <bool IN_BF16>
__device__ __forceinline__ void store_elem(void* p, int64_t e, float v, bool as_bf16) {
    if (as_bf16)
        static_cast<uint16_t*>(p)[e] = f32_to_bf16(v);
    else
        static_cast<float*>(p)[e] = v;
}

// Index of the ring chunk holding element e: the number of boundaries
// c * chunk (c = 1 .. t-1) at or below e (compares instead of a 64-bit divide).
__device__ __forceinline__ int chunk_of(const ReduceArgs& a, int64_t e) {
    int c = 0;
#pragma unroll
    for (int i = 1; i < TP_MAX_SHARDS; ++i) c += (i < a.t && e >= i * a.chunk) ? 1 : 0;
    return c;
}

template <bool IN_BF16>
__device__ void reduce_scalar(const ReduceArgs& a, int64_t e) {
    const int start = a.ring ? chunk_of(a, e) : 0;
    float acc = load_elem<IN_BF16>(a.p[start], e);
    for (int j = 1; j < a.t; ++j) {
        int r = start + j;
        if (r >= a.t) r -= a.t;
        const float x = load_elem<IN_BF16>(a.p[r], e);
        acc = a.hop_bf16 ? round_bf16(acc + x) : acc + x;
    }
    if (a.out) store_elem<IN_BF16>(a.out, e, acc, a.out_bf16 != 0);
    if (a.replicate)
        for (int r = 0; r < a.t; ++r) store_elem<IN_BF16>(const_cast<void*>(a.p[r]), e, acc, IN_BF16);
}

template <bool IN_BF16>
__device__ __forceinline__ void unpack(const uint4& q, float (&x)[IN_BF16 ? 8 : 4]) {
    if constexpr (IN_BF16) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        x[0] = __uint_as_float(q.x);
        x[1] = __uint_as_float(q.y);
        x[2] = __uint_as_float(q.z);
        x[3] = __uint_as_float(q.w);
    }
}

template <int VEC>
__device__ __forceinline__ void store_vec(void* base, int64_t e0, const float (&acc)[VEC], bool as_bf16) {
    if (as_bf16) {
        uint32_t w[VEC / 2];
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) w[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
        if constexpr (VEC == 8) {
            reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + e0)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + e0)[0] = make_uint2(w[0], w[1]);
        }
    } else {
        float* o = static_cast<float*>(base) + e0;
#pragma unroll
        for (int i = 0; i < VEC; i += 4)
            reinterpret_cast<float4*>(o + i)[0] = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    }
}

// One slice of the reduction per blockIdx.y: the whole buffer in DIRECT
// order, ring chunk y in RING order.  Inside a slice every block folds the
// t buffers in the same rotated order (y, y+1, ... mod t), with G vectors of
// 16 bytes per buffer in flight per thread (G * t 128-bit loads) so that a
// small t still keeps enough bytes moving.  Elements of the slice that do
// not fill a whole aligned vector (its ends, when a chunk boundary or the
// buffer end is not vector aligned) are folded one by one by block 0.
// Launched with t <= MAXT = 8 / G.
template <bool IN_BF16, int G>
__global__ void __launch_bounds__(256) shard_reduce_kernel(const __grid_constant__ ReduceArgs a) {
    constexpr int MAXT = TP_MAX_SHARDS / G;
    constexpr int VEC = IN_BF16 ? 8 : 4;
    constexpr int EB = IN_BF16 ? 2 : 4;
    pdl_wait();                                       // the partials may be the previous grid's output
    if (threadIdx.x == 0) pdl_trigger();              // the next kernel of the stream may take freed SMs
    const int slice = blockIdx.y;
    const int64_t lo = a.ring ? min(static_cast<int64_t>(slice) * a.chunk, a.count) : 0;
    const int64_t hi = a.ring ? min(lo + a.chunk, a.count) : a.count;
    const int64_t v_lo = (lo + VEC - 1) / VEC;        // whole vectors inside [lo, hi)
    const int64_t v_hi = hi / VEC;
    const char* q[MAXT];
#pragma unroll
    for (int j = 0; j < MAXT; ++j) {
        int r = slice + j;
        while (r >= a.t) r -= a.t;
        q[j] = static_cast<const char*>(a.p[j < a.t ? r : 0]);
    }
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t g0 = v_lo + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g0 < v_hi;
         g0 += stride * G) {
        uint4 v[G][MAXT];
#pragma unroll
        for (int u = 0; u < G; ++u) {
            const int64_t gi = g0 + u * stride;
#pragma unroll
            for (int j = 0; j < MAXT; ++j)
                if (gi < v_hi && j < a.t) v[u][j] = __ldcs(reinterpret_cast<const uint4*>(q[j] + gi * VEC * EB));
        }
#pragma unroll
        for (int u = 0; u < G; ++u) {
            const int64_t gi = g0 + u * stride;
            if (gi >= v_hi) continue;
            const int64_t e0 = gi * VEC;
            float acc[VEC];
            unpack<IN_BF16>(v[u][0], acc);
#pragma unroll
            for (int j = 1; j < MAXT; ++j) {
                if (j < a.t) {
                    float x[VEC];
                    unpack<IN_BF16>(v[u][j], x);
                    if (a.hop_bf16) {
#pragma unroll
                        for (int i = 0; i < VEC; ++i) acc[i] = round_bf16(acc[i] + x[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < VEC; ++i) acc[i] = acc[i] + x[i];
                    }
                }
            }
            if (a.out) store_vec<VEC>(a.out, e0, acc, a.out_bf16 != 0);
            if (a.replicate) {
#pragma unroll
                for (int r = 0; r < MAXT; ++r)
                    if (r < a.t) store_vec<VEC>(const_cast<void*>(a.p[r]), e0, acc, IN_BF16);
            }
        }
    }
    if (blockIdx.x == 0) {
        // the slice's elements outside whole vectors: [lo, v_lo*VEC) and [v_hi*VEC, hi),
        // or all of [lo, hi) when no whole vector fits
        const int64_t head_end = v_lo < v_hi ? v_lo * VEC : hi;
        const int64_t tail_beg = v_lo < v_hi ? v_hi * VEC : hi;
        for (int64_t e = lo + threadIdx.x; e < head_end; e += blockDim.x) reduce_scalar<IN_BF16>(a, e);
        for (int64_t e = tail_beg + threadIdx.x; e < hi; e += blockDim.x) reduce_scalar<IN_BF16>(a, e);
    }
}

template <bool IN_BF16, int G>
static int resident_blocks() {
    static std::atomic<int> n{0};               // relaxed: racing first calls store the same value
    int c = n.load(std::memory_order_relaxed);
    if (c <= 0) {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, shard_reduce_kernel<IN_BF16, G>, 256, 0) != cudaSuccess ||
            v <= 0)
            v = 2;
        c = v;
        n.store(c, std::memory_order_relaxed);
    }
    return c;
}

static int sm_count_cached() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::atomic<int> cache[64];        // per device; relaxed: racing first calls store the same value
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <bool IN_BF16, int G>
static void launch_reduce_cfg(const ReduceArgs& a, int64_t count, int t, bool ring, int pdl, cudaStream_t stream) {
    constexpr int VEC = IN_BF16 ? 8 : 4;
    const int slices = ring ? t : 1;
    const int64_t per_slice = (ring ? (count + t - 1) / t : count) / VEC + 1;
    const int sms = std::max(1, sm_count_cached());
    // one persistent wave: all resident blocks of the GPU, shared by the slices
    const int64_t resident = static_cast<int64_t>(sms) * resident_blocks<IN_BF16, G>();
    const int64_t want = (per_slice + 256LL * G - 1) / (256LL * G);
    const int gx = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, std::max<int64_t>(1, resident / slices))));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, slices, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // start early, wait in the kernel
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaLaunchKernelEx(&cfg, shard_reduce_kernel<IN_BF16, G>, a);
}

tp_status launch_shard_reduce(const ReduceDesc& d, cudaStream_t stream) {
    if (d.count == 0) return TP_OK;
    ReduceArgs a;
    for (int r = 0; r < TP_MAX_SHARDS; ++r) a.p[r] = r < d.t ? d.p[r] : nullptr;
    a.out = d.out;
    a.count = d.count;
    a.t = d.t;
    a.chunk = (d.count + d.t - 1) / d.t;
    a.ring = d.ring;
    a.hop_bf16 = d.hop_bf16;
    a.out_bf16 = d.out_bf16;
    a.replicate = d.replicate;
    const bool ring = d.ring != 0;
    // vectors in flight per thread: about 8 loads of 16 bytes whatever t is
    if (d.in_bf16) {
        if (d.t <= 2) launch_reduce_cfg<true, 4>(a, d.count, d.t, ring, d.pdl, stream);
        else if (d.t <= 4) launch_reduce_cfg<true, 2>(a, d.count, d.t, ring, d.pdl, stream);
        else launch_reduce_cfg<true, 1>(a, d.count, d.t, ring, d.pdl, stream);
    } else {
        if (d.t <= 2) launch_reduce_cfg<false, 4>(a, d.count, d.t, ring, d.pdl, stream);
        else if (d.t <= 4) launch_reduce_cfg<false, 2>(a, d.count, d.t, ring, d.pdl, stream);
        else launch_reduce_cfg<false, 1>(a, d.count, d.t, ring, d.pdl, stream);
    }
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// ------------------------------------------------------------------ gather

struct GatherArgs {
    const void* s[TP_MAX_SHARDS];
    int64_t cols[TP_MAX_SHARDS];
    int64_t off[TP_MAX_SHARDS];
    void* out;
    int64_t rows;
    int64_t total_cols;
    int t;
    int elem;
};

// One thread block per (row, shard) segment: copy the shard's row into its
// column slice of the output row, 16 bytes at a time when both ends allow.
__global__ void __launch_bounds__(256) shard_gather_kernel(const __grid_constant__ GatherArgs a) {
    pdl_wait();                                       // the shards may be the previous kernel's output
    if (threadIdx.x == 0) pdl_trigger();
    const int64_t nseg = a.rows * a.t;
    for (int64_t seg = blockIdx.x; seg < nseg; seg += gridDim.x) {
        const int r = static_cast<int>(seg % a.t);
        const int64_t row = seg / a.t;
        const int64_t bytes = a.cols[r] * a.elem;
        if (bytes == 0) continue;
        const char* src = static_cast<const char*>(a.s[r]) + row * bytes;
        char* dst = static_cast<char*>(a.out) + (row * a.total_cols + a.off[r]) * a.elem;
        if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | bytes) & 15) == 0) {
            // four 16-byte loads in flight per thread before their stores
            const int64_t nv = bytes / 16;
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            const int64_t bd = blockDim.x;
            for (int64_t i = threadIdx.x; i < nv; i += 4 * bd) {
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (i + u * bd < nv) v[u] = __ldcs(s4 + i + u * bd);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (i + u * bd < nv) __stcs(d4 + i + u * bd, v[u]);
            }
        } else if (a.elem == 4) {
            for (int64_t i = threadIdx.x; i < a.cols[r]; i += blockDim.x)
                reinterpret_cast<uint32_t*>(dst)[i] = reinterpret_cast<const uint32_t*>(src)[i];
        } else {
            for (int64_t i = threadIdx.x; i < a.cols[r]; i += blockDim.x)
                reinterpret_cast<uint16_t*>(dst)[i] = reinterpret_cast<const uint16_t*>(src)[i];
        }
    }
}

tp_status launch_shard_gather(const GatherDesc& d, cudaStream_t stream) {
    GatherArgs a;
    int64_t off = 0;
    for (int r = 0; r < TP_MAX_SHARDS; ++r) {
        a.s[r] = r < d.t ? d.shards[r] : nullptr;
        a.cols[r] = r < d.t ? d.cols[r] : 0;
        a.off[r] = off;
        off += a.cols[r];
    }
    a.out = d.out;
    a.rows = d.rows;
    a.total_cols = off;
    a.t = d.t;
    a.elem = d.elem_bytes;
    if (d.rows == 0 || off == 0) return TP_OK;
    const int sms = std::max(1, sm_count_cached());
    const int64_t nseg = d.rows * d.t;
    const int grid = static_cast<int>(std::min<int64_t>(nseg, static_cast<int64_t>(sms) * 16));
    const cudaError_t e = launch_pdl(shard_gather_kernel, dim3(grid), dim3(256), 0, stream, a);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// ------------------------------------------------------------------ probe

// Waits on a barrier that nothing signals; the bounded wait must expire,
// record TP_ERR_TIMEOUT and return.
__global__ void expire_wait_kernel(uint64_t limit_ns, int* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    __syncthreads();
}

tp_status launch_expire_wait(uint64_t limit_ns, int* status, cudaStream_t stream) {
    expire_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

}  // namespace tpk
