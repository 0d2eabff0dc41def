// Sequence parallelism: the all-reduce after a row-parallel layer split into
// a reduce-scatter over token rows and an all-gather, with the per-token
// residual add and RMSNorm done between them on each rank's own rows (page
// "Tensor parallelism from scratch", exercise 1 and its reference answer;
// the pre-norm residual of its tp.py TPTransformer, x = x + block(norm(x))).
//
// On one GPU every rank's rows live in the same [n, h] buffers, so the
// kernel processes every row once: row i belongs to rank r = i / ceil(n/t),
// and its t partial rows are folded in that rank's reduce-scatter order
// (DIRECT: 0, 1, ..., t-1; RING: r+1, r+2, ..., r mod t, the order in which
// a ring that leaves chunk r on rank r adds the copies).  The normed row is
// written in place, which is the all-gather.  One thread block per row:
//   1. fold the t partials in fp32, add the residual, write the new residual
//      (bf16), keep the fp32 row in shared memory, accumulate sum of squares;
//   2. block-reduce the sum of squares;
//   3. out = x * rsqrt(mean(x^2) + eps) * weight, rounded to bf16.
// Bytes per row: t*h*b (partials) + 2h (residual) + 2h + 2h (outputs); the
// weight stays in L1/L2.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace tpk {

struct SeqParArgs {
    const void* p[TP_MAX_SHARDS];
    const uint16_t* residual;   // nullable
    const uint16_t* weight;
    uint16_t* residual_out;     // nullable
    uint16_t* out;
    int64_t n, h, rows_per;
    float eps;
    int t;
    int ring;
};

constexpr int kSeqThreads = 256;

__device__ __forceinline__ void bf16x8(const uint16_t* p, float (&x)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

// Unpack one 16-byte vector of a partial buffer (8 bf16 or 4 fp32) to fp32.
template <bool IN_BF16>
__device__ __forceinline__ void unpack16(const uint4& q, float* x) {
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

// G vectors of 16 bytes per thread per pass, with the loads of all t
// partials for all G issued before any is folded (G * t <= 8); t <= 8 / G.
template <bool IN_BF16, int G>
__global__ void __launch_bounds__(kSeqThreads, 4) seqpar_rmsnorm_kernel(const __grid_constant__ SeqParArgs a) {
    constexpr int MAXT = TP_MAX_SHARDS / G;
    constexpr int VEC = IN_BF16 ? 8 : 4;        // elements per 16-byte vector of a partial
    constexpr int EB = IN_BF16 ? 2 : 4;
    extern __shared__ float xrow[];             // the row in fp32, h floats
    __shared__ float warp_sums[kSeqThreads / 32];
    pdl_wait();                                 // the partials may be the previous kernel's output
    if (threadIdx.x == 0) pdl_trigger();
    const int64_t nvec = a.h / VEC;
    for (int64_t row = blockIdx.x; row < a.n; row += gridDim.x) {
        const int owner = static_cast<int>(row / a.rows_per);
        const int start = a.ring ? (owner + 1) % a.t : 0;
        const int64_t base = row * a.h;
        const char* q[MAXT];
#pragma unroll
        for (int j = 0; j < MAXT; ++j) {
            int r = start + j;
            while (r >= a.t) r -= a.t;
            q[j] = static_cast<const char*>(a.p[j < a.t ? r : 0]) + base * EB;
        }
        float ss = 0.0f;
        for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += kSeqThreads * G) {
            uint4 raw[G][MAXT];
            uint4 rres[G];                       // the residual vectors, loaded with the partials
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const int64_t v = v0 + u * kSeqThreads;
#pragma unroll
                for (int j = 0; j < MAXT; ++j)
                    if (v < nvec && j < a.t) raw[u][j] = __ldcs(reinterpret_cast<const uint4*>(q[j]) + v);
                if (v < nvec && a.residual != nullptr) {
                    if constexpr (IN_BF16) {
                        rres[u] = *reinterpret_cast<const uint4*>(a.residual + base + v * VEC);
                    } else {
                        const uint2 r2 = *reinterpret_cast<const uint2*>(a.residual + base + v * VEC);
                        rres[u] = make_uint4(r2.x, r2.y, 0u, 0u);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const int64_t v = v0 + u * kSeqThreads;
                if (v >= nvec) break;
                float acc[VEC];
                unpack16<IN_BF16>(raw[u][0], acc);
#pragma unroll
                for (int j = 1; j < MAXT; ++j) {
                    if (j < a.t) {
                        float x[VEC];
                        unpack16<IN_BF16>(raw[u][j], x);
#pragma unroll
                        for (int i = 0; i < VEC; ++i) acc[i] = acc[i] + x[i];
                    }
                }
                const int64_t e = base + v * VEC;
                if (a.residual != nullptr) {
                    const uint32_t w[4] = {rres[u].x, rres[u].y, rres[u].z, rres[u].w};
                    float rs[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        rs[2 * i] = __uint_as_float(w[i] << 16);
                        rs[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                    }
#pragma unroll
                    for (int i = 0; i < VEC; ++i) acc[i] = rs[i] + acc[i];
                }
                if (a.residual_out != nullptr) {
                    if constexpr (IN_BF16) {
                        *reinterpret_cast<uint4*>(a.residual_out + e) =
                            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                       pack_bf16x2(acc[4 % VEC], acc[5 % VEC]), pack_bf16x2(acc[6 % VEC], acc[7 % VEC]));
                    } else {
                        *reinterpret_cast<uint2*>(a.residual_out + e) =
                            make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
                    }
                }
                float4* xs = reinterpret_cast<float4*>(xrow + v * VEC);
#pragma unroll
                for (int i = 0; i < VEC; i += 4) xs[i / 4] = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
#pragma unroll
                for (int i = 0; i < VEC; ++i) ss += acc[i] * acc[i];
            }
        }
        // block sum of squares
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = ss;
        __syncthreads();
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kSeqThreads / 32; ++w) tot += warp_sums[w];
        const float rstd = rsqrtf(tot / static_cast<float>(a.h) + a.eps);
        for (int64_t v = threadIdx.x; v < a.h / 8; v += kSeqThreads) {
            float wt[8], y[8];
            bf16x8(a.weight + v * 8, wt);
            const float4* xs = reinterpret_cast<const float4*>(xrow + v * 8);
            const float4 x0 = xs[0], x1 = xs[1];
            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = xv[i] * rstd * wt[i];
            *reinterpret_cast<uint4*>(a.out + base + v * 8) = pack8(y);
        }
        __syncthreads();                         // xrow and warp_sums are reused by the next row
    }
}

template <bool IN_BF16, int G>
static tp_status launch_seqpar_cfg(const SeqParArgs& a, int64_t n, size_t smem, cudaStream_t stream) {
    auto kern = seqpar_rmsnorm_kernel<IN_BF16, G>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return TP_ERR_CUDA;
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSeqThreads, smem);
    const int64_t resident = static_cast<int64_t>(std::max(sms, 1)) * std::max(per_sm, 1);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(n, resident)));
    const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kSeqThreads), smem, stream, a);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

tp_status launch_seqpar_rmsnorm(const SeqParDesc& d, cudaStream_t stream) {
    if (d.n == 0) return TP_OK;
    SeqParArgs a;
    for (int r = 0; r < TP_MAX_SHARDS; ++r) a.p[r] = r < d.t ? d.p[r] : nullptr;
    a.residual = static_cast<const uint16_t*>(d.residual);
    a.weight = static_cast<const uint16_t*>(d.weight);
    a.residual_out = static_cast<uint16_t*>(d.residual_out);
    a.out = static_cast<uint16_t*>(d.out);
    a.n = d.n;
    a.h = d.h;
    a.rows_per = (d.n + d.t - 1) / d.t;
    a.eps = d.eps;
    a.t = d.t;
    a.ring = d.ring;
    const size_t smem = static_cast<size_t>(d.h) * sizeof(float);
    if (d.in_bf16) {
        if (d.t <= 2) return launch_seqpar_cfg<true, 4>(a, d.n, smem, stream);
        if (d.t <= 4) return launch_seqpar_cfg<true, 2>(a, d.n, smem, stream);
        return launch_seqpar_cfg<true, 1>(a, d.n, smem, stream);
    }
    if (d.t <= 2) return launch_seqpar_cfg<false, 4>(a, d.n, smem, stream);
    if (d.t <= 4) return launch_seqpar_cfg<false, 2>(a, d.n, smem, stream);
    return launch_seqpar_cfg<false, 1>(a, d.n, smem, stream);
}

}  // namespace tpk
