// The tensor-parallel MLP of one to eight tokens in one GEMM kernel plus an
// ordered reduce.
//
// The MLP block computes Y = sum_r act(X G_r) * (X U_r) B_r: the first GEMM is
// column-parallel (rank r holds f/t columns of the gate and up projections),
// the second row-parallel (rank r holds the matching f/t rows of W_down), and
// the all-reduce adds the ranks' partial sums ("6.2 Tensor-parallel
// inference", section 1; the gated form of "Nano-vLLM walkthrough 22",
// MergedColumnParallelLinear and RowParallelLinear).  At a few tokens both
// GEMMs are weight streams of a few MB, and the two-launch path pays a launch
// ramp, a prologue and a serial K loop twice, its second GEMM waiting for the
// first to drain.
//
// Here one CTA pair takes one 64-column slice of a rank's f columns and does
// both GEMMs of that slice:
//   - CTA q loads X, the slice's 32 gate and 32 up rows of half q (all of K)
//     and rows [q h/2, (q+1) h/2) of the slice's 64 columns of W_down, all at
//     launch, so the down weights stream in alongside the gate and up weights;
//   - it computes G and U for its 32 columns (tcgen05.mma, M = 128 over the 8
//     staged token rows, N = 64), applies the activation, rounds H to bf16 as
//     the two-launch path stores it, writes it into its own H tile and sends
//     the tile to the peer with one shared-to-shared bulk copy;
//   - once its own tile is written and the peer's has arrived it multiplies
//     its W_down rows by the slice's H (M = 128 rows of W_down per MMA, N = 16
//     token columns, K = 64: two K steps from each tile; the four W_down tiles
//     are issued by four warps) and stores the fp32 partial of its h/2
//     outputs for every token.
// A second kernel, launched programmatically behind the first, adds the
// slices' partials in slice order in fp32 (rank 0's slices first), adds the
// bias once and stores Y.  That fixed-order sum is the fused all-reduce: the
// ranks' shares never exist as separate [n, h] sums.
//
// Loads: one TMA box for X (all K blocks), one per 4 K blocks of the gate and
// up rows, one for the W_down rows.  Each box lands as consecutive K blocks
// in the MMA's layout (tensor-map views whose K-block stride is below the row
// stride).  A copy has a large fixed cost: at one box per K block a CTA
// streamed about 40 GB/s, with these boxes the whole load takes about a third
// of that time.
//
// Shared memory (1024-byte aligned regions, h <= 1024): X as h/64 K blocks of
// 8 rows x 128 bytes (the M = 128 MMA reads a 16 KB window from each block's
// start; rows 8-127 fall on later blocks and on the gate/up region, land in
// accumulator rows that are never read, and are inside the allocation), gate
// and up rows as h/64 blocks of 64 rows x 128 bytes, W_down as h/256 tiles of
// 128 rows x 128 bytes, two H tiles of 16 rows x 128 bytes (tile q holds
// columns 32q..32q+31, rows n..15 zero), then the barriers: 212 KB at
// h = 1024.  TMEM: G and U in columns 0-63, the down GEMM's tiles in columns
// 64 + 16 t.
//
// Every wait is bounded (TP_ERR_TIMEOUT in the status word, then the CTA
// unwinds and waits for copies in flight); the pair always meets at its
// final cluster barrier, by which point each CTA has received the peer's
// copy, so no CTA exits while a copy into or out of its shared memory may be
// in flight.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace tpk {
namespace {

constexpr int kSliceCols = 64;        // f columns per CTA pair
constexpr int kHalfCols = 32;         // gate (and up) rows per CTA
constexpr int kMaxH = 1024;
constexpr int kMaxKBlocks = kMaxH / 64;
constexpr int kThreads = 128;
constexpr int kTmemCols = 128;
constexpr int kBarBytes = 256;
constexpr int kGroup = 4;             // K blocks per gate/up copy (one barrier each)

struct SmallArgs {
    CUtensorMap mapX;                       // X [n, h]: one box of 8 rows by every K block
    CUtensorMap mapGU[TP_MAX_SHARDS];       // [gate; up] rows of rank r: boxes of 32 + 32 rows by kGroup K blocks
    CUtensorMap mapD[TP_MAX_SHARDS];        // W_down of rank r [h, f/t]: one box of h/256 tiles of 128 rows
    float* part;                            // [slices][n][h] fp32
    int n, h, slices_per_rank, act;
    int* status;
};

struct SmallLayout {
    uint32_t x, gu, dw, hh, bar, total;
    __host__ __device__ explicit SmallLayout(int h) {
        const uint32_t kb = static_cast<uint32_t>(h) / 64;
        x = 0;
        gu = kb * 1024;
        dw = gu + kb * 8192;
        hh = dw + static_cast<uint32_t>(h / 256) * 16384;
        bar = hh + 4096;
        total = bar + kBarBytes;
    }
};

// H = act(G) * U for this CTA's 32 columns, rounded to bf16, into its H tile:
// row = token (lanes 0-15; rows n..15 zero), the 32 columns = 16-byte chunks
// 4q..4q+3 of the 128-byte row, chunk c of row r at chunk c ^ (r mod 8) (the
// 128-byte swizzle).  One 8-column chunk per step: the activation chains of a
// step overlap, and the loop body stays short (this code runs once per CTA).
template <int ACT>
__device__ __forceinline__ void store_h_tile(uint32_t tmem_base, uint32_t tile, uint32_t q, int lane, int n) {
    const uint32_t r = static_cast<uint32_t>(lane);
    const uint32_t row = tile + (r >> 3) * 1024 + (r & 7) * 128;
    const bool live = lane < n;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t g[8], u[8];
        tmem_ld8(tmem_base + 8u * c, g);
        tmem_ld8(tmem_base + 32u + 8u * c, u);
        tmem_ld_wait();
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = act_fn(__uint_as_float(g[e]), ACT) * __uint_as_float(u[e]);
        if (lane < 16) {
            const uint32_t addr = row + (((q * 4 + c) ^ (r & 7)) << 4);
            st_shared_v4(addr, live ? pack_bf16x2(v[0], v[1]) : 0u, live ? pack_bf16x2(v[2], v[3]) : 0u,
                         live ? pack_bf16x2(v[4], v[5]) : 0u, live ? pack_bf16x2(v[6], v[7]) : 0u);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) tp_mlp_small_kernel(const __grid_constant__ SmallArgs args) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_word;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_u32(smem);
    const SmallLayout L(args.h);
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const uint32_t q = cluster_ctarank();
    const int slice = static_cast<int>(blockIdx.x >> 1);
    const int rank = slice / args.slices_per_rank;
    const int j = slice - rank * args.slices_per_rank;
    const int kb_n = args.h / 64;
    const int mt = args.h / 256;
    const uint32_t bar0 = base + L.bar;
    const uint32_t dw_bar = bar0 + 8u * kMaxKBlocks;
    const uint32_t mma1_bar = dw_bar + 8u;
    const uint32_t hx_bar = dw_bar + 16u;
    const uint32_t mma2_bar = dw_bar + 24u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.bar + 8 * (kMaxKBlocks + 4));
    volatile int* abort_flag = &abort_word;

    if (threadIdx.x == 0) {
        abort_word = 0;
        for (int i = 0; i < kb_n / kGroup; ++i) mbar_init(bar0 + 8u * i, 1);   // one per gate/up copy
        mbar_init(dw_bar, 1);
        mbar_init(mma1_bar, 1);
        mbar_init(hx_bar, 1);                       // own H tile written (+ the peer's copy of its tile)
        mbar_init(mma2_bar, static_cast<uint32_t>(mt));   // one commit per W_down tile
        fence_barrier_init();
        prefetch_tmap(&args.mapX);
        prefetch_tmap(&args.mapGU[rank]);
        prefetch_tmap(&args.mapD[rank]);
    }
    if (warp == 1) tmem_alloc<kTmemCols>(smem_u32(tmem_slot));
    __syncwarp();
    tc_fence_before();
    cluster_sync();                                 // the peer arrives on hx_bar: inits first
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_trigger();            // the reduce may take SMs as they free up

    bool aborted = false;
    if (warp == 0) {
        if (lane == 0) {
            // The first kernel of the call: X and the weights may have been written by the
            // previous kernel of the stream, so nothing is loaded before the wait.
            pdl_wait();
            // h/256 + 2 copies (six at h = 1024): X (all K blocks), the gate and up rows in
            // groups of kGroup K blocks, the W_down tiles.  A copy's cost has a large fixed
            // part, so few large boxes stream several times faster per SM than one box per
            // K block.
            const int f0 = j * kSliceCols + static_cast<int>(q) * kHalfCols;
            const int groups = kb_n / kGroup;
            for (int gi = 0; gi < groups; ++gi) {
                const uint32_t bar = bar0 + 8u * gi;
                mbar_arrive_expect_tx(bar, (gi == 0 ? static_cast<uint32_t>(kb_n) * 1024u : 0u) + kGroup * 8192u);
                if (gi == 0) tma_load_3d(base + L.x, &args.mapX, bar, 0, 0, 0);
                tma_load_4d(base + L.gu + gi * kGroup * 8192, &args.mapGU[rank], bar, 0, f0, 0, gi * kGroup);
            }
            mbar_arrive_expect_tx(dw_bar, static_cast<uint32_t>(mt) * 16384u);
            tma_load_3d(base + L.dw, &args.mapD[rank], dw_bar, j * kSliceCols, 0, static_cast<int>(q) * mt);
            // G (accumulator columns 0-31) and U (32-63) of this CTA's 32 columns
            constexpr uint32_t idesc = mma_idesc_bf16(128, 64);
            for (int gi = 0; gi < groups && !aborted; ++gi) {
                if (!mbar_wait(bar0 + 8u * gi, 0, abort_flag, args.status)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                for (int i = gi * kGroup; i < (gi + 1) * kGroup; ++i) {
                    const uint64_t ad = sw128_kmajor_desc(base + L.x + i * 1024);
                    const uint64_t bd = sw128_kmajor_desc(base + L.gu + i * 8192);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma(tmem_base, ad + 2u * k, bd + 2u * k, idesc, (i | k) != 0 ? 1u : 0u);
                }
            }
            if (!aborted) tc_commit(mma1_bar);
        }
        __syncwarp();
        // H of this CTA's 32 columns into its own H tile (tile q), then one bulk copy of the
        // tile to the same place in the peer, completing on the peer's hx_bar.
        if (mbar_wait_warp(mma1_bar, 0, abort_flag, args.status)) {
            tc_fence_after();
            const uint32_t tile = base + L.hh + q * 2048;
            if (args.act == TP_ACT_GELU_TANH_MUL)
                store_h_tile<TP_ACT_GELU_TANH_MUL>(tmem_base, tile, q, lane, args.n);
            else
                store_h_tile<TP_ACT_SILU_MUL>(tmem_base, tile, q, lane, args.n);
            fence_proxy_async_cta();                // the stores before the copy's and the MMAs' reads
            __syncwarp();
            if (lane == 0) {
                mbar_arrive_expect_tx(hx_bar, 2048u);   // own tile written; the peer's copy brings the other
                bulk_copy_s2s(mapa_shared(tile, q ^ 1u), tile, 2048u, mapa_shared(hx_bar, q ^ 1u));
            }
        } else {
            aborted = true;
        }
        __syncwarp();
    }
    // Down GEMM, D[row][token] = sum_k W_down[row][k] H[token][k]: warp t issues the four MMAs
    // of W_down tile t (independent accumulators), K steps 0-1 from H tile 0, 2-3 from tile 1.
    if (!aborted && warp < mt) {
        if (lane == 0) {
            if (!mbar_wait(hx_bar, 0, abort_flag, args.status) || !mbar_wait(dw_bar, 0, abort_flag, args.status)) {
                aborted = true;
            } else {
                tc_fence_after();
                constexpr uint32_t idesc = mma_idesc_bf16(128, 16);
                const uint64_t ad = sw128_kmajor_desc(base + L.dw + warp * 16384);
                const uint64_t b0 = sw128_kmajor_desc(base + L.hh);
                const uint64_t b1 = sw128_kmajor_desc(base + L.hh + 2048);
                const uint32_t d = tmem_base + 64u + 16u * static_cast<uint32_t>(warp);
                tc_mma(d, ad, b0, idesc, 0u);
                tc_mma(d, ad + 2u, b0 + 2u, idesc, 1u);
                tc_mma(d, ad + 4u, b1 + 4u, idesc, 1u);
                tc_mma(d, ad + 6u, b1 + 6u, idesc, 1u);
                tc_commit(mma2_bar);
            }
        }
        aborted = __shfl_sync(0xffffffffu, aborted ? 1 : 0, 0) != 0;
    }
    // fp32 partial [token][column] of this slice; warp w holds W_down rows 32w..32w+31 of each tile
    if (!aborted) {
        if (mbar_wait_warp(mma2_bar, 0, abort_flag, args.status)) {
            tc_fence_after();
            const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + 64u;
            uint32_t v[4][8];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                if (t < mt) tmem_ld8(lane_base + 16u * t, v[t]);
            tmem_ld_wait();
            const int n = args.n;
            float* out = args.part + static_cast<size_t>(slice) * n * args.h + static_cast<int>(q) * (args.h / 2) +
                         warp * 32 + lane;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (t < mt) {
#pragma unroll
                    for (int tok = 0; tok < 8; ++tok)
                        if (tok < n) out[static_cast<size_t>(tok) * args.h + t * 128] = __uint_as_float(v[t][tok]);
                }
            }
        } else {
            aborted = true;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) spin_ns(50000);                // let issued TMA copies and MMAs land
    if (warp == 1) tmem_dealloc<kTmemCols>(tmem_base);
    cluster_sync_relaxed();
}

// Y[idx] = sum over slices s (in order) of part[s][idx], plus the bias, for
// float4 element idx of Y [n, h].  Eight groups of 32 threads each sum a
// contiguous run of slices (its loads all in flight at once); the groups'
// sums are then added in group order.
constexpr int kRedGroups = 8;
constexpr int kRedCols = 32;
constexpr int kRedMaxRun = 16;                      // slices per group: kMaxSlices / kRedGroups

__global__ void __launch_bounds__(kRedGroups * kRedCols) tp_mlp_small_reduce_kernel(const float* part, int slices,
                                                                                     int count4, int h,
                                                                                     const uint16_t* bias, void* y,
                                                                                     int y_f32) {
    __shared__ float4 acc[kRedGroups][kRedCols];
    if (threadIdx.x == 0) pdl_trigger();
    const int g = static_cast<int>(threadIdx.x) / kRedCols;
    const int e = static_cast<int>(threadIdx.x) % kRedCols;
    const int idx = static_cast<int>(blockIdx.x) * kRedCols + e;
    pdl_wait();                                     // the partials are the previous kernel's output
    float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (idx < count4) {
        const int run = (slices + kRedGroups - 1) / kRedGroups;
        const int c0 = min(slices, g * run);
        const int c1 = min(slices, c0 + run);
        const float4* p = reinterpret_cast<const float4*>(part) + idx;
        float4 v[kRedMaxRun];
#pragma unroll
        for (int i = 0; i < kRedMaxRun; ++i)
            if (c0 + i < c1) v[i] = p[static_cast<size_t>(c0 + i) * count4];
#pragma unroll
        for (int i = 0; i < kRedMaxRun; ++i) {
            if (c0 + i < c1) {
                s.x += v[i].x;
                s.y += v[i].y;
                s.z += v[i].z;
                s.w += v[i].w;
            }
        }
    }
    acc[g][e] = s;
    __syncthreads();
    if (g == 0 && idx < count4) {
        float4 t = acc[0][e];
#pragma unroll
        for (int i = 1; i < kRedGroups; ++i) {
            t.x += acc[i][e].x;
            t.y += acc[i][e].y;
            t.z += acc[i][e].z;
            t.w += acc[i][e].w;
        }
        if (bias != nullptr) {
            const int col = (idx * 4) % h;
            t.x += bf16_to_f32(bias[col]);
            t.y += bf16_to_f32(bias[col + 1]);
            t.z += bf16_to_f32(bias[col + 2]);
            t.w += bf16_to_f32(bias[col + 3]);
        }
        if (y_f32) {
            reinterpret_cast<float4*>(y)[idx] = t;
        } else {
            reinterpret_cast<uint2*>(y)[idx] = make_uint2(pack_bf16x2(t.x, t.y), pack_bf16x2(t.z, t.w));
        }
    }
}

}  // namespace

size_t small_mlp_workspace(int t, int64_t n, int64_t h, int64_t f, tp_reduce_mode mode) {
    if (mode != TP_REDUCE_FUSED || t < 1 || t > TP_MAX_SHARDS || n < 1 || n > kSmallMlpMaxRows) return 0;
    if (h < 256 || h > kMaxH || h % 256 != 0 || f <= 0 || f % t != 0 || (f / t) % kSliceCols != 0) return 0;
    const int64_t slices = f / kSliceCols;
    if (slices > kSmallMlpMaxSlices) return 0;
    const size_t bytes = static_cast<size_t>(slices * n * h) * 4;
    return (bytes + 255) & ~static_cast<size_t>(255);
}

tp_status launch_small_mlp(const SmallMlpDesc& d, cudaStream_t stream) {
    if (small_mlp_workspace(d.t, d.n, d.h, d.f, TP_REDUCE_FUSED) == 0) return TP_ERR_UNSUPPORTED;
    SmallArgs a;
    std::memset(&a, 0, sizeof(a));
    const int64_t fs = d.f / d.t;
    const int kb_n = static_cast<int>(d.h / 64);
    if (!make_kblock_map(&a.mapX, d.x, d.n, d.h, d.ldx, 8, kb_n)) return TP_ERR_CUDA;
    for (int r = 0; r < d.t; ++r) {
        if (!make_gated_kblock_map(&a.mapGU[r], d.w_gate_up[r], fs, d.h, d.h, kHalfCols, kGroup)) return TP_ERR_CUDA;
        if (!make_row_tile_map(&a.mapD[r], d.w_down[r], d.h, fs, d.ld_down, 128, static_cast<int>(d.h / 256)))
            return TP_ERR_CUDA;
    }
    a.part = d.part;
    a.n = static_cast<int>(d.n);
    a.h = static_cast<int>(d.h);
    a.slices_per_rank = static_cast<int>(fs / kSliceCols);
    a.act = d.act;
    a.status = d.status;
    const int slices = static_cast<int>(d.f / kSliceCols);
    const int smem = static_cast<int>(SmallLayout(a.h).total) + 1024;
    // The shared memory depends on h, and the opt-in is set once per device: set it for the
    // largest h, so that a first call with a smaller h does not cap later ones.
    static std::atomic<uint64_t> smem_set{0};
    if (!smem_attribute_once(reinterpret_cast<const void*>(tp_mlp_small_kernel),
                             static_cast<int>(SmallLayout(kMaxH).total) + 1024, smem_set))
        return TP_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * slices, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, tp_mlp_small_kernel, a) != cudaSuccess) return TP_ERR_CUDA;

    const int count4 = static_cast<int>(d.n * d.h / 4);
    const int blocks = (count4 + kRedCols - 1) / kRedCols;
    if (launch_pdl(tp_mlp_small_reduce_kernel, dim3(blocks), dim3(kRedGroups * kRedCols), 0, stream,
                   static_cast<const float*>(d.part), slices, count4, a.h, static_cast<const uint16_t*>(d.bias),
                   d.y, d.y_f32) != cudaSuccess)
        return TP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

}  // namespace tpk
