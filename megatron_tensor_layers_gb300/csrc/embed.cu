// Vocab-parallel input embedding (page "Tensor parallelism from scratch",
// tp.py VocabParallelEmbedding; page "vLLM source analysis 13: tensor
// parallelism in detail", §2.4.1).
//
// Rank r owns ids [r*per, min((r+1)*per, V)), per = ceil(V/t).  Its output
// for an id outside its range is exactly 0 (masked_fill, so a NaN row of
// another rank never leaks), and the t outputs are all-reduced (summed in
// rank order).  Ranges are disjoint, so for every token at most one rank
// holds a real row: the kernel reads that one row (one warp per token,
// 16-byte loads) and forms the rank-order sum of it and t-1 exact zeros in
// float32, which is x + 0.0 in closed form.  That sum is bit-exact to the
// lookup, except that -0.0 becomes +0.0 when t > 1, which is what summing
// the ranks' outputs gives.
// Bytes moved per token: h*b read (owner row) + h*b written (+ t*h*b for the
// optional per-rank outputs) + 4 for the id.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace tpk {

struct EmbedArgs {
    const void* table[TP_MAX_SHARDS];
    void* partials[TP_MAX_SHARDS];
    const int32_t* ids;
    void* out;
    int64_t vocab, h, n, per;
    int t;
    int with_partials;
};

template <bool BF16>
__global__ void __launch_bounds__(256) vocab_embed_kernel(const __grid_constant__ EmbedArgs a) {
    constexpr int VEC = BF16 ? 8 : 4;             // elements per 16-byte vector
    const int lane = threadIdx.x & 31;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nvec = a.h / VEC;
    for (int64_t tok = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; tok < a.n; tok += warps) {
        const int32_t id = a.ids[tok];
        int owner = -1;
        int64_t local = 0;
        if (id >= 0 && id < a.vocab) {     // 32-bit arithmetic: ids and vocab sizes are int32
            const uint32_t u = static_cast<uint32_t>(id), per = static_cast<uint32_t>(a.per);
            owner = static_cast<int>(u / per);
            local = static_cast<int64_t>(u - static_cast<uint32_t>(owner) * per);
        }
        const uint4* src = owner >= 0 ? reinterpret_cast<const uint4*>(a.table[owner]) + local * nvec : nullptr;
        uint4* dst = reinterpret_cast<uint4*>(a.out) + tok * nvec;
        // Up to U row vectors per lane are loaded before any is stored, so a
        // warp has the whole 2 KB row (h = 1024 bf16) in flight at once.
        constexpr int U = 4;
        for (int64_t v0 = lane; v0 < nvec; v0 += 32 * U) {
            uint4 row[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * 32;
                row[u] = (owner >= 0 && v < nvec) ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * 32;
                if (v >= nvec) break;
                const uint32_t w[4] = {row[u].x, row[u].y, row[u].z, row[u].w};
                float x[VEC];
                if constexpr (BF16) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[2 * i] = __uint_as_float(w[i] << 16);
                        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VEC; ++i) x[i] = __uint_as_float(w[i]);
                }
                // The all-reduce: the rank-order sum of the t masked outputs.  At most one of them
                // is non-zero, the rest are exact +0.0, so for t > 1 the sum is x + 0.0 in every
                // order (x itself, except that -0.0 becomes +0.0; NaN and Inf pass), and for t = 1
                // it is x.  __fadd_rn keeps the addition from being contracted or dropped.
                float acc[VEC];
#pragma unroll
                for (int i = 0; i < VEC; ++i) acc[i] = a.t > 1 ? __fadd_rn(x[i], 0.0f) : x[i];
                uint4 o;
                if constexpr (BF16) {
                    o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
                } else {
                    o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                                   __float_as_uint(acc[3]));
                }
                dst[v] = o;
                if (a.with_partials) {
                    for (int r = 0; r < a.t; ++r)
                        reinterpret_cast<uint4*>(a.partials[r])[tok * nvec + v] =
                            owner == r ? row[u] : make_uint4(0, 0, 0, 0);
                }
            }
        }
    }
}

tp_status launch_vocab_embed(const EmbedDesc& d, cudaStream_t stream) {
    if (d.n == 0) return TP_OK;
    EmbedArgs a;
    for (int r = 0; r < TP_MAX_SHARDS; ++r) {
        a.table[r] = r < d.t ? d.table[r] : nullptr;
        a.partials[r] = (d.with_partials && r < d.t) ? d.partials[r] : nullptr;
    }
    a.ids = d.ids;
    a.out = d.out;
    a.vocab = d.vocab;
    a.h = d.h;
    a.n = d.n;
    a.per = d.per;
    a.t = d.t;
    a.with_partials = d.with_partials;
    // one warp per token; at most one resident wave of blocks (grid-stride beyond)
    const int64_t want = (d.n * 32 + 255) / 256;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    static int per_sm[2] = {0, 0};            // a property of the kernel, the same on every GB300
    int& occ = per_sm[d.bf16 ? 1 : 0];
    if (occ <= 0) {
        if (d.bf16)
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, vocab_embed_kernel<true>, 256, 0);
        else
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, vocab_embed_kernel<false>, 256, 0);
    }
    const int64_t resident = static_cast<int64_t>(std::max(sms, 1)) * std::max(occ, 1);
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, resident)));
    // Launched in plain stream order: with programmatic launch, back-to-back lookups of
    // 4096 ids measured 3.33 us per call instead of 2.97.
    if (d.bf16)
        vocab_embed_kernel<true><<<grid, 256, 0, stream>>>(a);
    else
        vocab_embed_kernel<false><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

}  // namespace tpk
