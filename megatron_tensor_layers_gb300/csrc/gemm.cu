// Tensor-parallel GEMMs on the 5th-generation tensor core (sm_103a).
//
// One persistent, warp-specialised kernel family computes, for every shard
// ("group") g of a tensor-parallel layer,
//
//     D_g = sum over K-segments s of  A_{g,s} · B_{g,s}^T        (fp32 accumulate)
//
// with A [M, K] and B [N, K] both K-major bf16 (weights are stored [out, in],
// so x @ w^T is exactly this form).  It serves
//   - ColumnParallelLinear: group = shard, A = the replicated input x,
//     B = the shard's weight block (page "Nano-vLLM walkthrough 22", §3);
//   - the gated MLP up-projection: B's tile is the shard's gate rows stacked
//     on the SAME rows of its up block (the merged "double cut", §5 of the
//     same page) and the epilogue writes act(gate) * up (page "Tensor
//     parallelism from scratch", tp.py TPMLP);
//   - RowParallelLinear: group = shard writing its own partial sum, or one
//     group with t K-segments whose partial products are accumulated in rank
//     order in the same TMEM accumulator ("fused" all-reduce, no partial is
//     ever written) (page "6.2 Tensor-parallel inference", §1: Y = sum_i
//     act(X A_i) B_i);
//   - the vocab-sharded LM head: group = shard, the epilogue writes straight
//     into the shard's column slice of the full logits (zero-copy gather).
//
// Roles (192 threads, one CTA per SM):
//   warp 0  lane 0: TMA producer, fills a STAGES-deep ring of A/B tiles;
//   warp 1  lane 0: MMA issuer (tcgen05.mma, 128 x BN x 16 per instruction)
//           into one of two TMEM accumulators; the whole warp allocates TMEM;
//   warps 2-5: epilogue, 128 threads = the 128 TMEM lanes = the tile's rows;
//           they drain one accumulator while the MMA fills the other.
// Every barrier wait is bounded (1 s); a wait that expires records
// TP_ERR_TIMEOUT and the CTA unwinds and exits normally.
//
// Every GEMM (and the reduce) is launched with programmatic stream
// serialization: it may start while the previous kernel of the stream
// drains.  Its producer executes griddepcontrol.wait before loading anything
// that kernel may have written: for the first kernel of a library call that
// is everything; a split-K or single-CTA GEMM that is a later kernel of the
// same call (whose predecessor writes no weights) loads its first ring of
// weights before the wait.
// The stage ring is split into groups of KSUB stages (K blocks) under one
// full and one empty barrier each, so the producer and MMA threads wait, arm
// and commit once per group; at short K their per-block barrier work, not
// the MMAs, would otherwise set the pace.
// Three kernels share this structure: tp_gemm_kernel (one CTA per tile),
// tp_gemm_pair_kernel (256 x 256 tiles on a CTA pair, cta_group::2) and
// tp_gemm_splitk_kernel (the K loop of a decode-sized tile split over a
// cluster, accumulators added over distributed shared memory).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace tpk {

constexpr int BM = 128;          // tile rows (tokens) = TMEM lanes
constexpr int BK = 64;           // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 192;

enum { EPI_STORE = 0, EPI_GLU = 1 };

struct GemmArgs {
    CUtensorMap mapA[TP_MAX_SHARDS];
    CUtensorMap mapB[TP_MAX_SHARDS];
    void* out[TP_MAX_SHARDS];         // per-group output base (already offset for a gather)
    const void* bias[TP_MAX_SHARDS];  // per-group bf16 bias over output columns, or null
    int64_t ldo;                      // output row stride (elements)
    int out_f32;                      // 1: float32 output, 0: bf16
    int M;                            // rows of A / D
    int N;                            // output columns per group (widest group)
    int n_valid[TP_MAX_SHARDS];       // valid output columns of each group
    int m_tiles, n_tiles, groups, total_tiles;
    int k_blocks;                     // K blocks per segment
    int segs;                         // K segments accumulated into one tile
    int a_per_group;                  // A map index = group (else 0); with segs > 1 it is the segment
    int glu_up_row;                   // row offset of the up block inside B (gated epilogue)
    int group_m;                      // tile raster: bands of group_m row-tiles (about kRasterBandMB of A rows)
    int bands_span_groups;            // 1: a band covers every group's columns (groups share A)
    int a_box_rows;                   // rows of A a TMA box loads (<= 128; fewer when M is small)
    int kgroup_box;                   // tp_gemm_kernel: A and B maps are K-block views, one box per KSUB group
    int rotate_k;                     // start each tile's K loop at block (tile mod k_blocks)
    int act;                          // tp_act for the gated epilogue
    int split;                        // split-K kernel: CTAs per cluster sharing one output tile
    int pdl_prefetch;                 // 1: B may be loaded before waiting for the previous grid
    int* status;                      // library status word
    // stream-K tail (pair kernel, store epilogue): tiles [sk_first, total_tiles)
    // run as sk_parts K-parts each; sk_first == total_tiles: no tail split
    int sk_first;
    int sk_parts;
    int* sk_flags;                    // one per (partial slot, CTA of the pair)
    float* sk_scratch;                // partial slots of 256 x 256 fp32
};

// Tile index -> (group, row-tile, column-tile).  Tiles run in bands of
// group_m row-tiles; inside a band the row-tile varies fastest, so the band's
// A rows stay in L2 while its columns of B stream past.  Bands either repeat
// per group (groups outermost) or, when the groups share A, cover the columns
// of every group, so A is read once for all groups.
__device__ __forceinline__ void tile_coords(const GemmArgs& a, int tile, int& g, int& m, int& n) {
    const int cols = a.bands_span_groups ? a.groups * a.n_tiles : a.n_tiles;
    const int per_span = a.m_tiles * cols;
    const int outer = tile / per_span;                   // the group (0 when bands span the groups)
    const int l = tile - outer * per_span;
    const int width = a.group_m * cols;
    const int band = l / width;
    const int first_m = band * a.group_m;
    const int gm = min(a.m_tiles - first_m, a.group_m);
    const int r = l - band * width;
    m = first_m + r % gm;
    const int col = r / gm;
    if (a.bands_span_groups) {
        g = col / a.n_tiles;
        n = col - g * a.n_tiles;
    } else {
        g = outer;
        n = col;
    }
}

// Store one output element (bf16 or fp32) at (row, col).
__device__ __forceinline__ void store_one(void* base, int64_t ldo, int out_f32, int64_t row, int col, float v) {
    if (out_f32)
        static_cast<float*>(base)[row * ldo + col] = v;
    else
        static_cast<uint16_t*>(base)[row * ldo + col] = f32_to_bf16(v);
}

// Store 32 consecutive fp32 values of one output row, columns [col0, col0 + nvalid).
__device__ __forceinline__ void store_chunk(void* base, int64_t ldo, int out_f32, int64_t row, int col0, int nvalid,
                                            const float (&v)[32]) {
    if (nvalid <= 0) return;
    if (out_f32) {
        float* p = static_cast<float*>(base) + row * ldo + col0;
        if (nvalid == 32 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                reinterpret_cast<float4*>(p)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid) p[j] = v[j];
        }
    } else {
        uint16_t* p = static_cast<uint16_t*>(base) + row * ldo + col0;
        if (nvalid == 32 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 q;
                q.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
                q.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
                q.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
                q.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
                reinterpret_cast<uint4*>(p)[j] = q;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < nvalid) p[j] = f32_to_bf16(v[j]);
        }
    }
}

// AROWS: shared-memory rows of a stage's A tile.  Launches with M <= 64
// (decode) keep 64 rows, and launches with M <= 8 keep 8, and spend the room
// on a deeper B ring, since their time is the weight stream and the bytes
// each SM keeps in flight bound it.  The M = 128 MMA then also reads the
// 16 KB that follow the stage's start as A rows AROWS-127 (the stage's B
// tile and, for short stages, the start of the next stage); those
// accumulator rows are never stored.  PAD_BYTES keeps that read window of
// the last stage inside the allocation.
//
// STG_BYTES: the gated decode configurations also keep, per epilogue warp
// that can hold rows (the first two), a 32-row staging area of one 32-column
// chunk of gate and up accumulators (65 floats a row: 64 values and a pad
// that keeps both the row-wise writes and the column-wise reads free of bank
// conflicts).  A warp with fewer than 32 rows below M stages them there and
// then has every lane compute one output column over those rows, instead of
// each row's lane computing all 32 columns (one token of decode: 1
// activation per lane instead of 32).
template <int BN, int STAGES, int EPI, int AROWS = BM>
struct GemmCfg {
    static constexpr int A_BYTES = AROWS * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;   // two accumulators
    static constexpr int BAR_BYTES = (2 * STAGES + 4) * 8 + 16;
    static constexpr int STG_ROW = 65;
    static constexpr int STG_BYTES = (EPI == EPI_GLU && AROWS < BM) ? 2 * 32 * STG_ROW * 4 : 0;
    static constexpr int MMA_A_BYTES = BM * BK * 2;                    // what the M = 128 MMA reads as A
    static constexpr int TAIL_BYTES = STAGE_BYTES + STG_BYTES + BAR_BYTES;   // from the last stage's start
    static constexpr int PAD_BYTES = (AROWS < BM && TAIL_BYTES < MMA_A_BYTES) ? MMA_A_BYTES - TAIL_BYTES : 0;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STG_BYTES + BAR_BYTES + PAD_BYTES;
    static constexpr int OUT_COLS = (EPI == EPI_GLU) ? BN / 2 : BN;   // output columns per tile
    static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
    static_assert(BN % 32 == 0 && BN <= 256, "M=128 MMA needs N % 16 == 0, N <= 256; epilogue chunks of 32");
    static_assert(STAGE_BYTES % 1024 == 0, "stage tiles must stay 1024-byte aligned");
    static_assert(AROWS == BM || AROWS == 64 || AROWS == 16 || AROWS == 8, "A tiles of 128, 64, 16 or 8 rows");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// KSUB: K blocks per ring slot group.  The STAGES stage buffers form STAGES/KSUB groups with
// one full and one empty barrier each: the producer waits once, arms once and issues KSUB
// blocks' loads; the MMA thread waits once, issues KSUB blocks' MMAs and commits once.  At
// decode sizes with short K the MMA thread's per-block wait, fence and commit (about twice
// the MMAs' own time for a 64-wide tile) otherwise bound the K loop.
template <int BN, int STAGES, int EPI, int AROWS, int KSUB>
__global__ void __launch_bounds__(kThreads, 1) tp_gemm_kernel(const __grid_constant__ GemmArgs args) {
    using Cfg = GemmCfg<BN, STAGES, EPI, AROWS>;
    static_assert(KSUB >= 1 && STAGES % KSUB == 0, "stage groups of KSUB blocks");
    constexpr int GROUPS = STAGES / KSUB;
    // A group holds KSUB stages.  With one box per K block each stage is [A | B]; with K-block
    // boxes (args.kgroup_box) the group is its KSUB A slabs, then its KSUB B tiles, so that one
    // box can bring each (the A window of the M = 128 MMA reads on into the group's later
    // tiles, never past the ring and its tail).
    constexpr uint32_t kGroupBytes = KSUB * Cfg::STAGE_BYTES;
    // Only the 16- and 64-row-A configurations (9 to 64 tokens) use K-block boxes; the others
    // compile without the branch (at short K one more instruction per K block shows in the time).
    constexpr bool kKGroup = KSUB > 1 && (AROWS == 64 || AROWS == 16);
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles.
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    float* stg_base = reinterpret_cast<float*>(base_ptr + STAGES * Cfg::STAGE_BYTES);
    const uint32_t bar_base = base + STAGES * Cfg::STAGE_BYTES + Cfg::STG_BYTES;
    uint8_t* bar_ptr = base_ptr + STAGES * Cfg::STAGE_BYTES + Cfg::STG_BYTES;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * STAGES + 4));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * (2 * STAGES + 4) + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < args.groups && i < TP_MAX_SHARDS; ++i) prefetch_tmap(&args.mapB[i]);
        prefetch_tmap(&args.mapA[0]);
    }
    if (warp == 1) tmem_alloc<Cfg::TMEM_COLS>(smem_u32(tmem_slot));
    __syncwarp();                                      // CTA barriers below are warp-aligned
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_trigger();       // the next grid of the stream may take freed SMs

    const int kb_per_tile = args.k_blocks * args.segs;
    bool aborted = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // With a programmatic launch the previous grid of the stream may still be running
            // (A can be its output).  When that grid is a kernel of the same call, which writes
            // no B (pdl_prefetch), the first ring of the first tile's weights is loaded before
            // the wait and its A blocks after it; the loop below then starts that tile past
            // those groups, so the issue loop itself gains no branch (at decode sizes the
            // producer's issue rate bounds the weight stream: a per-block check of whether a
            // stage was already armed cost 6 %).
            int grp = 0;
            uint32_t phase = 0;
            const uint32_t block_bytes = static_cast<uint32_t>(args.a_box_rows * 128 + Cfg::B_BYTES);
            const bool kgb = kKGroup && args.kgroup_box;
            auto tile_rot = [&](int tile) {
                return !args.rotate_k ? 0
                       : kgb          ? (tile % (args.k_blocks / KSUB)) * KSUB
                                      : tile % args.k_blocks;
            };
            // K block number, segment and A/B map of position kk of a tile's K loop
            auto kpos = [&](int kk, int rot, int g, int& kb, int& ai, int& bi) {
                const int seg = kk / args.k_blocks;
                kb = kk - seg * args.k_blocks + rot;
                if (kb >= args.k_blocks) kb -= args.k_blocks;
                ai = args.segs > 1 ? seg : (args.a_per_group ? g : 0);
                bi = args.segs > 1 ? seg : g;
            };
            int pre_kk = 0;                                // K blocks of the first tile already issued
            if (args.pdl_prefetch && static_cast<int>(blockIdx.x) < args.total_tiles) {
                int g, m, n;
                tile_coords(args, blockIdx.x, g, m, n);
                const int rot = tile_rot(blockIdx.x);
                const int pre_groups = min(GROUPS, (kb_per_tile + KSUB - 1) / KSUB);
                for (int gi = 0; gi < pre_groups; ++gi) {    // B, before the wait
                    const int cnt = min(KSUB, kb_per_tile - gi * KSUB);
                    mbar_arrive_expect_tx(full_bar(gi), static_cast<uint32_t>(cnt) * block_bytes);
                    const uint32_t ga = base + gi * kGroupBytes;
                    if (kgb) {
                        int kb, ai, bi;
                        kpos(gi * KSUB, rot, g, kb, ai, bi);
                        const uint32_t gb = ga + KSUB * Cfg::A_BYTES;
                        if (EPI == EPI_GLU)
                            tma_load_4d(gb, &args.mapB[bi], full_bar(gi), 0, n * (BN / 2), 0, kb);
                        else
                            tma_load_3d(gb, &args.mapB[bi], full_bar(gi), 0, n * BN, kb);
                    } else {
                        for (int i = 0; i < cnt; ++i) {
                            int kb, ai, bi;
                            kpos(gi * KSUB + i, rot, g, kb, ai, bi);
                            const uint32_t sb = ga + i * Cfg::STAGE_BYTES + Cfg::A_BYTES;
                            if (EPI == EPI_GLU)
                                tma_load_3d(sb, &args.mapB[bi], full_bar(gi), kb * BK, n * (BN / 2), 0);
                            else
                                tma_load_2d(sb, &args.mapB[bi], full_bar(gi), kb * BK, n * BN);
                        }
                    }
                }
                pdl_wait();
                for (int gi = 0; gi < pre_groups; ++gi) {    // A, after it
                    const int cnt = min(KSUB, kb_per_tile - gi * KSUB);
                    const uint32_t ga = base + gi * kGroupBytes;
                    if (kgb) {
                        int kb, ai, bi;
                        kpos(gi * KSUB, rot, g, kb, ai, bi);
                        tma_load_3d(ga, &args.mapA[ai], full_bar(gi), 0, m * BM, kb);
                    } else {
                        for (int i = 0; i < cnt; ++i) {
                            int kb, ai, bi;
                            kpos(gi * KSUB + i, rot, g, kb, ai, bi);
                            tma_load_2d(ga + i * Cfg::STAGE_BYTES, &args.mapA[ai], full_bar(gi), kb * BK, m * BM);
                        }
                    }
                }
                pre_kk = min(kb_per_tile, pre_groups * KSUB);
                grp = pre_groups == GROUPS ? 0 : pre_groups;
                phase = pre_groups == GROUPS ? 1u : 0u;
            } else {
                pdl_wait();
            }
            for (int tile = blockIdx.x; tile < args.total_tiles && !aborted; tile += gridDim.x) {
                int g, m, n;
                tile_coords(args, tile, g, m, n);
                // With a few rows of A every CTA would read the same line of A at the same k;
                // starting each tile's K loop (each segment's, with segments) elsewhere spreads
                // those reads over L2 and the weight reads over the DRAM channels.
                // With K-block boxes the rotation moves in whole groups, so that a group's KSUB
                // blocks stay consecutive inside one segment.
                const int rot = tile_rot(tile);
                // (segment, block) advanced incrementally: no division in the issue loop
                const int kk0 = tile == static_cast<int>(blockIdx.x) ? pre_kk : 0;
                int seg = kk0 / args.k_blocks, kin = kk0 - seg * args.k_blocks;
                for (int kk = kk0; kk < kb_per_tile; kk += KSUB) {
                    const int cnt = min(KSUB, kb_per_tile - kk);   // a tile's last group may be short
                    if (!mbar_wait(empty_bar(grp), phase ^ 1u, abort_flag, args.status)) {
                        aborted = true;
                        break;
                    }
                    const uint32_t bar = full_bar(grp);
                    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(cnt) * block_bytes);
                    const uint32_t ga = base + grp * kGroupBytes;
                    if (kgb) {
                        // the whole group in one A box and one B box (cnt == KSUB here)
                        int kb = kin + rot;
                        if (kb >= args.k_blocks) kb -= args.k_blocks;
                        const int ai = args.segs > 1 ? seg : (args.a_per_group ? g : 0);
                        const int bi = args.segs > 1 ? seg : g;
                        kin += KSUB;
                        if (kin == args.k_blocks) {
                            kin = 0;
                            ++seg;
                        }
                        const uint32_t gb = ga + KSUB * Cfg::A_BYTES;    // the group's B tiles
                        tma_load_3d(ga, &args.mapA[ai], bar, 0, m * BM, kb);
                        if (EPI == EPI_GLU)
                            tma_load_4d(gb, &args.mapB[bi], bar, 0, n * (BN / 2), 0, kb);
                        else
                            tma_load_3d(gb, &args.mapB[bi], bar, 0, n * BN, kb);
                    } else {
#pragma unroll
                        for (int i = 0; i < KSUB; ++i) {
                            if (i < cnt) {
                                int kb = kin + rot;
                                if (kb >= args.k_blocks) kb -= args.k_blocks;
                                const int ai = args.segs > 1 ? seg : (args.a_per_group ? g : 0);
                                const int bi = args.segs > 1 ? seg : g;
                                if (++kin == args.k_blocks) {
                                    kin = 0;
                                    ++seg;
                                }
                                const uint32_t sa = ga + i * Cfg::STAGE_BYTES;
                                const uint32_t sb = sa + Cfg::A_BYTES;
                                tma_load_2d(sa, &args.mapA[ai], bar, kb * BK, m * BM);
                                if (EPI == EPI_GLU) {   // gate rows and the same rows of up, one 3-D box
                                    tma_load_3d(sb, &args.mapB[bi], bar, kb * BK, n * (BN / 2), 0);
                                } else {
                                    tma_load_2d(sb, &args.mapB[bi], bar, kb * BK, n * BN);
                                }
                            }
                        }
                    }
                    if (++grp == GROUPS) {
                        grp = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = mma_idesc_bf16(BM, BN);
            // Tile addresses inside a group: per stage [A | B], or (K-block boxes) the A slabs
            // packed box-height apart, then the B tiles
            const bool kg = kKGroup && args.kgroup_box != 0;
            const uint32_t a_stride = kg ? static_cast<uint32_t>(args.a_box_rows) * 128u : Cfg::STAGE_BYTES;
            const uint32_t b_first = kg ? KSUB * Cfg::A_BYTES : Cfg::A_BYTES;
            const uint32_t b_stride = kg ? Cfg::B_BYTES : Cfg::STAGE_BYTES;
            int grp = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = blockIdx.x; tile < args.total_tiles && !aborted; tile += gridDim.x) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.status)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kk = 0; kk < kb_per_tile; kk += KSUB) {
                    const int cnt = min(KSUB, kb_per_tile - kk);
                    if (!mbar_wait(full_bar(grp), phase, abort_flag, args.status)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        if (i < cnt) {
                            const uint32_t ga = base + grp * kGroupBytes;
                            const uint64_t adesc = sw128_kmajor_desc(ga + i * a_stride);
                            const uint64_t bdesc = sw128_kmajor_desc(ga + b_first + i * b_stride);
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k) {
                                // advance 16 bf16 = 32 bytes along K inside the swizzle row
                                tc_mma(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, ((kk + i) | k) != 0 ? 1u : 0u);
                            }
                        }
                    }
                    tc_commit(empty_bar(grp));
                    if (++grp == GROUPS) {
                        grp = 0;
                        phase ^= 1u;
                    }
                }
                if (aborted) break;
                tc_commit(tfull_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int row_in_tile = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < args.total_tiles; tile += gridDim.x) {
            int g, m, n;
            tile_coords(args, tile, g, m, n);
            if (!mbar_wait_warp(tfull_bar(acc), acc_phase, abort_flag, args.status)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const int64_t grow = static_cast<int64_t>(m) * BM + row_in_tile;
            const bool row_ok = grow < args.M;
            // Accumulator rows past M hold whatever the rest of the A tile held; a warp with no
            // row below M skips the tile, and the others feed 0 through the activation there.
            const bool warp_live = static_cast<int64_t>(m) * BM + q * 32 < args.M;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            void* out = args.out[g];
            const uint16_t* bias = static_cast<const uint16_t*>(args.bias[g]);
            const int ncols = args.n_valid[g];
            // rows of this warp below M (1..32 when warp_live)
            const int64_t left = args.M - (static_cast<int64_t>(m) * BM + q * 32);
            const int live = left < 32 ? static_cast<int>(left) : 32;
            if (!warp_live) {
            } else if (EPI == EPI_GLU && Cfg::STG_BYTES > 0 && live < 32) {
                // few rows: stage them, then lane j computes column j of every live row
                float* st = stg_base + (q & 1) * 32 * Cfg::STG_ROW;
                const int64_t row0 = static_cast<int64_t>(m) * BM + q * 32;
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t rg[32], ru[32];
                    tmem_ld32(taddr + c * 32, rg);
                    tmem_ld32(taddr + BN / 2 + c * 32, ru);
                    tmem_ld_wait();
                    if (lane < live) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            st[lane * Cfg::STG_ROW + j] = __uint_as_float(rg[j]);
                            st[lane * Cfg::STG_ROW + 32 + j] = __uint_as_float(ru[j]);
                        }
                    }
                    __syncwarp();
                    const int col = n * (BN / 2) + c * 32 + lane;
                    if (col < ncols) {
                        // rows are independent: unrolled, their activation chains overlap
#pragma unroll 4
                        for (int r = 0; r < live; ++r)
                            store_one(out, args.ldo, args.out_f32, row0 + r, col,
                                      act_fn(st[r * Cfg::STG_ROW + lane], args.act) * st[r * Cfg::STG_ROW + 32 + lane]);
                    }
                    __syncwarp();                         // the next chunk reuses the staging rows
                }
            } else if (EPI == EPI_GLU) {
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t rg[32], ru[32];
                    tmem_ld32(taddr + c * 32, rg);
                    tmem_ld32(taddr + BN / 2 + c * 32, ru);
                    tmem_ld_wait();
                    const int col0 = n * (BN / 2) + c * 32;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = act_fn(row_ok ? __uint_as_float(rg[j]) : 0.0f, args.act) * __uint_as_float(ru[j]);
                    if (row_ok) store_chunk(out, args.ldo, args.out_f32, grow, col0, min(32, ncols - col0), v);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(taddr + c * 32, r);
                    tmem_ld_wait();
                    const int col0 = n * BN + c * 32;
                    const int nvalid = min(32, ncols - col0);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (bias != nullptr) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nvalid) v[j] += bf16_to_f32(bias[col0 + j]);
                    }
                    if (row_ok) store_chunk(out, args.ldo, args.out_f32, grow, col0, nvalid, v);
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(acc));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    if (aborted) spin_ns(50000);    // let issued TMA copies and MMAs land before teardown
    // The producer and MMA roles ran on lane 0 alone; the barrier below is
    // warp-aligned, so each warp first waits for all of its lanes.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) spin_ns(50000);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<Cfg::TMEM_COLS>(tmem_base);
    }
}

// ---------------------------------------------------------- CTA-pair kernel
//
// The same computation on 256 x 256 tiles shared by a cluster of two CTAs on
// neighbouring SMs (tcgen05 cta_group::2).  CTA r of the pair loads rows
// [128r, 128r+128) of the tile's A rows and the r-th 128-row half of its B
// rows (for the gated epilogue: CTA 0 the gate rows, CTA 1 the same rows of
// up); the even CTA issues one M=256, N=256, K=16 MMA that reads both CTAs'
// shared memory and writes each CTA's 128 rows x 256 columns into that CTA's
// TMEM.  Per SM this halves the B bytes that TMA writes into, and the tensor
// core reads out of, shared memory for the same FLOPs, which is what bounds
// the single-CTA kernel.  Both CTAs' loads complete on the even CTA's
// full barrier; MMA completion is multicast to both CTAs' stage and
// accumulator barriers; both epilogues report back to the even CTA.
constexpr int kPairStages = 6;   // 6 x 32 KB ring (7 measured no faster for the gated kernel)
constexpr int kPairKsub = 2;     // K blocks per ring barrier

template <int STAGES, int EPI>
struct PairCfg {
    static constexpr int BN = 256;                           // MMA N (full tile width)
    static constexpr int A_BYTES = 128 * BK * 2;             // this CTA's 128 rows of A
    static constexpr int B_BYTES = 128 * BK * 2;             // this CTA's half of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 16;
    // Store epilogue: per epilogue warp, 32 output rows of 128 bytes (64 bf16 or 32 fp32
    // columns) plus a 16-byte pad, so that a warp writes whole 128-byte lines of 4 rows per
    // store instruction instead of one 16-byte piece of 32 rows.
    static constexpr int STG_PITCH = 144;
    static constexpr int STG_BYTES = (EPI == EPI_STORE) ? 4 * 32 * STG_PITCH : 0;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STG_BYTES + BAR_BYTES;
    static constexpr int OUT_COLS = (EPI == EPI_GLU) ? BN / 2 : BN;
    static constexpr int TILE_M = 256;
    static_assert(STAGE_BYTES % 1024 == 0, "stage tiles must stay 1024-byte aligned");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

// Work item j of a cluster of the pair kernel: first its whole tiles (tile
// cluster + i * nclusters below sk_first), then its stream-K units (unit u =
// cluster + i * nclusters below the tail's tiles x sk_parts: tile sk_first +
// u / sk_parts, part u % sk_parts of the tile's K blocks).  All roles of both
// CTAs of a pair walk the same sequence.
struct PairWork {
    int tile;
    int kb_lo, kb_hi;    // K blocks [kb_lo, kb_hi) of the tile's kb_per_tile
    int part;            // 0: whole tile or the first part (which adds the others); > 0: a partial
};

__device__ __forceinline__ bool pair_work(const GemmArgs& a, int cluster, int nclusters, int j, int kb_per_tile,
                                          PairWork& w) {
    const int whole = a.sk_first > cluster ? (a.sk_first - cluster + nclusters - 1) / nclusters : 0;
    if (j < whole) {
        w.tile = cluster + j * nclusters;
        w.kb_lo = 0;
        w.kb_hi = kb_per_tile;
        w.part = 0;
        return true;
    }
    const int u = cluster + (j - whole) * nclusters;
    if (u >= (a.total_tiles - a.sk_first) * a.sk_parts) return false;
    w.tile = a.sk_first + u / a.sk_parts;
    w.part = u % a.sk_parts;
    w.kb_lo = static_cast<int>(static_cast<int64_t>(w.part) * kb_per_tile / a.sk_parts);
    w.kb_hi = static_cast<int>(static_cast<int64_t>(w.part + 1) * kb_per_tile / a.sk_parts);
    return true;
}

template <int STAGES, int EPI, int KSUB>
__global__ void __launch_bounds__(kThreads, 1) tp_gemm_pair_kernel(const __grid_constant__ GemmArgs args) {
    using Cfg = PairCfg<STAGES, EPI>;
    static_assert(KSUB >= 1 && STAGES % KSUB == 0, "stage groups of KSUB blocks (as in tp_gemm_kernel)");
    constexpr int GROUPS = STAGES / KSUB;
    constexpr int BN = Cfg::BN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    uint8_t* stg_base = base_ptr + STAGES * Cfg::STAGE_BYTES;
    const uint32_t bar_base = base + STAGES * Cfg::STAGE_BYTES + Cfg::STG_BYTES;
    uint8_t* bar_ptr = base_ptr + STAGES * Cfg::STAGE_BYTES + Cfg::STG_BYTES;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
    const uint32_t sk_bar = bar_base + 8u * (2 * STAGES + 4);   // this CTA's epilogue warps stored a partial
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * (2 * STAGES + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * (2 * STAGES + 5) + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();          // 0: issues the MMAs; 1: its peer
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 8);              // 4 epilogue warps x 2 CTAs
        }
        mbar_init(sk_bar, 4);                         // the 4 epilogue warps of this CTA
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < args.groups && i < TP_MAX_SHARDS; ++i) prefetch_tmap(&args.mapB[i]);
        prefetch_tmap(&args.mapA[0]);
    }
    if (warp == 1) tmem_alloc_pair<Cfg::TMEM_COLS>(smem_u32(tmem_slot));
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync();                                    // both CTAs' barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_trigger();

    const int kb_per_tile = args.k_blocks * args.segs;
    bool aborted = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            pdl_wait();                                // A may be the previous grid's output
            int grp = 0;
            uint32_t phase = 0;
            PairWork w;
            for (int wi = 0; !aborted && pair_work(args, cluster, nclusters, wi, kb_per_tile, w); ++wi) {
                int g, m, n;
                tile_coords(args, w.tile, g, m, n);
                const int a_row = m * Cfg::TILE_M + static_cast<int>(rank) * 128;
                const int b_row = (EPI == EPI_GLU) ? (rank == 0 ? n * 128 : args.glu_up_row + n * 128)
                                                   : n * BN + static_cast<int>(rank) * 128;
                int seg = w.kb_lo / args.k_blocks;     // (segment, block), then advanced without division
                int kb = w.kb_lo - seg * args.k_blocks;
                for (int kk = w.kb_lo; kk < w.kb_hi; kk += KSUB) {
                    const int cnt = min(KSUB, w.kb_hi - kk);
                    if (!mbar_wait(empty_bar(grp), phase ^ 1u, abort_flag, args.status)) {
                        aborted = true;
                        break;
                    }
                    if (rank == 0)
                        mbar_arrive_expect_tx(full_bar(grp), static_cast<uint32_t>(cnt) * 2u * Cfg::STAGE_BYTES);
                    const uint32_t leader_full = mapa_shared(full_bar(grp), 0);
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        if (i < cnt) {
                            const int ai = args.segs > 1 ? seg : (args.a_per_group ? g : 0);
                            const int bi = args.segs > 1 ? seg : g;
                            const int kcol = kb * BK;
                            if (++kb == args.k_blocks) {
                                kb = 0;
                                ++seg;
                            }
                            const uint32_t sa = base + (grp * KSUB + i) * Cfg::STAGE_BYTES;
                            tma_load_2d_pair(sa, &args.mapA[ai], leader_full, kcol, a_row);
                            tma_load_2d_pair(sa + Cfg::A_BYTES, &args.mapB[bi], leader_full, kcol, b_row);
                        }
                    }
                    if (++grp == GROUPS) {
                        grp = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer (even CTA)
            constexpr uint32_t idesc = mma_idesc_bf16(256, BN);
            int grp = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            PairWork w;
            for (int wi = 0; !aborted && pair_work(args, cluster, nclusters, wi, kb_per_tile, w); ++wi) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.status)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kk = w.kb_lo; kk < w.kb_hi; kk += KSUB) {
                    const int cnt = min(KSUB, w.kb_hi - kk);
                    if (!mbar_wait(full_bar(grp), phase, abort_flag, args.status)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        if (i < cnt) {
                            const uint32_t sa = base + (grp * KSUB + i) * Cfg::STAGE_BYTES;
                            const uint64_t adesc = sw128_kmajor_desc(sa);
                            const uint64_t bdesc = sw128_kmajor_desc(sa + Cfg::A_BYTES);
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k)
                                tc_mma_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc,
                                            ((kk - w.kb_lo + i) | k) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit_pair(empty_bar(grp), 0x3);
                    if (++grp == GROUPS) {
                        grp = 0;
                        phase ^= 1u;
                    }
                }
                if (aborted) break;
                tc_commit_pair(tfull_bar(acc), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        const int row_in_tile = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t sk_phase = 0;
        PairWork w;
        for (int wi = 0; pair_work(args, cluster, nclusters, wi, kb_per_tile, w); ++wi) {
            int g, m, n;
            tile_coords(args, w.tile, g, m, n);
            if (!mbar_wait_warp(tfull_bar(acc), acc_phase, abort_flag, args.status)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const int64_t grow = static_cast<int64_t>(m) * Cfg::TILE_M + rank * 128 + row_in_tile;
            const bool row_ok = grow < args.M;
            const bool warp_live = static_cast<int64_t>(m) * Cfg::TILE_M + rank * 128 + q * 32 < args.M;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            void* out = args.out[g];
            const uint16_t* bias = static_cast<const uint16_t*>(args.bias[g]);
            const int ncols = args.n_valid[g];
            // Stream-K tail: the partials of tile w.tile occupy slots sk_slot .. sk_slot + sk_parts - 2,
            // each 256 x 256 fp32, this CTA's rows at [rank * 128, rank * 128 + 128).
            const int sk_slot = (w.tile - args.sk_first) * (args.sk_parts - 1);
            const size_t sk_row = (static_cast<size_t>(rank) * 128 + row_in_tile) * 256;
            bool sk_owner = false;
            if (EPI == EPI_STORE && w.part == 0 && w.tile >= args.sk_first && args.sk_parts > 1 && warp_live) {
                // the first part adds the other parts: wait until each has stored its partial
                bool ok = true;
                for (int p = 1; p < args.sk_parts && ok; ++p)
                    ok = flag_wait(args.sk_flags + (sk_slot + p - 1) * 2 + rank, abort_flag, args.status);
                if (!__all_sync(0xffffffffu, ok)) aborted = true;
                sk_owner = true;
            }
            if (EPI == EPI_STORE && w.part > 0) {
                // A later part: store this CTA's rows of the fp32 accumulator to the part's slot; once
                // all four epilogue warps have stored theirs, the first warp raises the slot's flag.
                const int slot = sk_slot + w.part - 1;
                float* dst = args.sk_scratch + static_cast<size_t>(slot) * (256 * 256) + sk_row;
                if (warp_live) {
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        if (n * BN + c * 32 >= ncols) break;
                        uint32_t r[32];
                        tmem_ld32(taddr + c * 32, r);
                        tmem_ld_wait();
                        if (row_ok) {
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj)
                                reinterpret_cast<float4*>(dst + c * 32)[jj] =
                                    make_float4(__uint_as_float(r[4 * jj]), __uint_as_float(r[4 * jj + 1]),
                                                __uint_as_float(r[4 * jj + 2]), __uint_as_float(r[4 * jj + 3]));
                        }
                    }
                }
                __threadfence();                      // this thread's partial is visible GPU-wide
                __syncwarp();
                if (lane == 0) mbar_arrive(sk_bar);
                if (q == 0) {
                    bool ok = true;
                    if (lane == 0) {
                        ok = mbar_wait(sk_bar, sk_phase, abort_flag, args.status);
                        if (ok) st_release_gpu(args.sk_flags + slot * 2 + rank, 1);
                    }
                    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) aborted = true;
                }
                sk_phase ^= 1u;
            } else if (!warp_live || aborted) {   // rows past M (ragged last row-tile): nothing to read or store
            } else if (EPI == EPI_GLU) {
#pragma unroll 1
                for (int c = 0; c < BN / 64; ++c) {
                    uint32_t rg[32], ru[32];
                    tmem_ld32(taddr + c * 32, rg);
                    tmem_ld32(taddr + BN / 2 + c * 32, ru);
                    tmem_ld_wait();
                    const int col0 = n * (BN / 2) + c * 32;
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = act_fn(row_ok ? __uint_as_float(rg[j]) : 0.0f, args.act) * __uint_as_float(ru[j]);
                    if (row_ok) store_chunk(out, args.ldo, args.out_f32, grow, col0, min(32, ncols - col0), v);
                }
            } else {
                // The warp stages whole 128-byte lines of its 32 rows (one 32-column chunk of fp32,
                // two of bf16) in shared memory and writes 4 rows' lines per store instruction
                // instead of one 16-byte piece of 32 rows.  Lines follow the absolute address, so
                // a shard whose columns start 64 bytes into a line (a vocab slice, say) stages
                // from its second chunk.  Chunks outside a whole valid line, and rows whose
                // stride is not a multiple of 128 bytes, take the per-row stores.
                const int es = args.out_f32 ? 4 : 2;
                const bool lines = ((args.ldo * es) & 127) == 0;
                uint8_t* st = stg_base + q * 32 * Cfg::STG_PITCH;
                const int64_t row0 = static_cast<int64_t>(m) * Cfg::TILE_M + rank * 128 + q * 32;
                int line_col = -1;                     // first column of a half-staged bf16 line
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int col0 = n * BN + c * 32;
                    if (col0 >= ncols) break;
                    uint32_t r[32];
                    tmem_ld32(taddr + c * 32, r);
                    tmem_ld_wait();
                    const int nvalid = min(32, ncols - col0);
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (sk_owner && row_ok) {
                        // the later parts' partials, added in part order
                        for (int p = 1; p < args.sk_parts; ++p) {
                            const float4* src = reinterpret_cast<const float4*>(
                                args.sk_scratch + static_cast<size_t>(sk_slot + p - 1) * (256 * 256) + sk_row + c * 32);
#pragma unroll
                            for (int jj = 0; jj < 8; ++jj) {
                                const float4 s = src[jj];
                                v[4 * jj] += s.x;
                                v[4 * jj + 1] += s.y;
                                v[4 * jj + 2] += s.z;
                                v[4 * jj + 3] += s.w;
                            }
                        }
                    }
                    if (bias != nullptr) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nvalid) v[j] += bf16_to_f32(bias[col0 + j]);
                    }
                    const uint32_t off = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(out) + static_cast<uint64_t>(col0) * es) & 127u;
                    int flush_col = -1;
                    if (lines && args.out_f32 && off == 0 && nvalid == 32) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4*>(st + lane * Cfg::STG_PITCH + j * 16) =
                                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        flush_col = col0;
                    } else if (lines && !args.out_f32 && ((off == 0 && col0 + 64 <= ncols && c + 1 < BN / 32) ||
                                                          (off == 64 && line_col >= 0))) {
                        const int half = off == 0 ? 0 : 64;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<uint4*>(st + lane * Cfg::STG_PITCH + half + j * 16) =
                                make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                           pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                        if (off == 0) {
                            line_col = col0;
                        } else {
                            flush_col = line_col;
                            line_col = -1;
                        }
                    } else if (row_ok) {
                        store_chunk(out, args.ldo, args.out_f32, grow, col0, nvalid, v);
                    }
                    if (flush_col >= 0) {
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int rr = i * 4 + (lane >> 3);
                            const int64_t gr = row0 + rr;
                            if (gr < args.M)
                                *reinterpret_cast<uint4*>(static_cast<char*>(out) + (gr * args.ldo + flush_col) * es + (lane & 7) * 16) =
                                    *reinterpret_cast<const uint4*>(st + rr * Cfg::STG_PITCH + (lane & 7) * 16);
                        }
                        __syncwarp();                 // the next line reuses the staging rows
                    }
                }
            }
            // The MMA only needs this warp's TMEM loads finished (wait::ld above) before it
            // overwrites the accumulator; the output stores need no ordering inside the kernel.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(tempty_bar(acc), 0));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            if (aborted) break;
        }
    }

    if (aborted) spin_ns(50000);
    __syncwarp();                                      // reconverge the lane-0 roles (aligned barriers below)
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) spin_ns(50000);
    cluster_sync();                                    // no MMA or remote arrive still targets the peer
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair<Cfg::TMEM_COLS>(tmem_base);
    }
}

// ------------------------------------------------------- split-K cluster kernel
//
// GEMMs with at most 64 token rows (decode, small batches).  Their time is
// the weight stream or, for small weights, the serial K loop of a tile, and
// the plain kernels leave SMs idle or use narrow tiles that stream slowly
// (every MMA instruction costs about the same issue time whatever its N: at
// N = 64 a 64-wide K block took 280 ns per SM, a 3.7 TB/s ceiling on 128
// SMs).  Here a cluster of CS CTAs shares each BN-wide output tile: CTA r
// runs K blocks [r*KB/CS, (r+1)*KB/CS) of the tile's KB = k_blocks * segs
// blocks, in order, into its own TMEM (for the fused reduce these are whole
// shards when CS divides t), stages its fp32 accumulator rows in its shared
// memory, and then every CTA adds, for its share of the tile's 32-column
// output chunks (chunk c belongs to rank c mod CS), the CS staged copies in
// rank order over distributed shared memory and runs the epilogue (bias,
// or act(gate) * up for the gated tile, whose gate and up columns are both
// summed first).  The K blocks are therefore still summed in order in fp32:
// for the fused reduce the shards in rank order (page "6.2 Tensor-parallel
// inference", §1: Y = sum_i act(X A_i) B_i), and no partial leaves the chip.
//
// Per tile and CTA: wait for the accumulator; wait until every epilogue warp
// of the cluster has read this CTA's staging of the previous tile
// (`drained`); stage; free the accumulator; each warp (lane 0, after a warp
// barrier, one cluster fence, then relaxed arrives: together one release)
// arrives on the `staged` barrier of every CTA of the cluster, its own
// included; acquire-wait on its own `staged`; the 128 epilogue threads reduce
// and store this CTA's chunks, one 4-column group of one row per item with
// the CS peer loads in flight together; each warp arrives on every CTA's
// `drained` (not after the CTA's last tile).  One arrival per warp instead
// of per thread: with CS = 8 a tile otherwise cost each CTA 1024 remote
// arrivals on each barrier.  Waits are bounded like every other wait of the
// library, and a relaxed cluster barrier before exit keeps each CTA's shared
// memory alive while its peers may still read it.
template <int BN, int STAGES, int EPI, int ROWS_ = 64>
struct SplitCfg {
    static constexpr int ROWS = ROWS_;                       // staged rows: M <= 64, M <= 16 or M <= 8
    static constexpr int A_BYTES = ROWS * BK * 2;            // 64-, 16- or 8-row A tile (see GemmCfg's AROWS)
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGING_BYTES = ROWS * BN * 4;      // fp32 accumulator rows
    // The 64-row, 256-wide store configuration keeps its staging in the ring (five stages
    // instead of four): valid only when every cluster runs one tile, so that no load is in
    // flight into the ring once the tile's last MMA has completed.  Its launch checks that.
    static constexpr bool STAGING_IN_RING = ROWS == 64 && BN == 256 && STAGES == 5;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int NBARS = 2 * STAGES + 6;
    static constexpr int SMEM_BYTES =
        1024 + STAGES * STAGE_BYTES + (STAGING_IN_RING ? 0 : STAGING_BYTES) + NBARS * 8 + 16;
    static constexpr int OUT_CHUNKS = (EPI == EPI_GLU ? BN / 2 : BN) / 32;   // 32-column output chunks per tile
    static_assert(STAGE_BYTES % 1024 == 0, "stage tiles must stay 1024-byte aligned");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(ROWS == 64 || ROWS == 16 || ROWS == 8, "64, 16 or 8 staged rows");
    static_assert(STAGE_BYTES >= BM * BK * 2, "the M = 128 MMA reads 16 KB of A from the stage's start");
    static_assert(!STAGING_IN_RING || STAGES * STAGE_BYTES >= STAGING_BYTES, "the staging fits the ring");
};

// Four fp32 accumulator values (float4 column `f4col` of `row`) summed over
// the cluster's CS staged copies in rank order; the CS loads are issued
// together before the sum.
template <int ROWS>
__device__ __forceinline__ float4 gather_f4(uint32_t staging, int f4col, int row, int cs) {
    const uint32_t off = staging + static_cast<uint32_t>((f4col * ROWS + row) * 16);
    float4 x[8];
#pragma unroll
    for (int p = 0; p < 8; ++p)
        if (p < cs) x[p] = ld_shared_cluster_f4(mapa_shared(off, static_cast<uint32_t>(p)));
    float4 v = x[0];
#pragma unroll
    for (int p = 1; p < 8; ++p) {
        if (p < cs) {
            v.x += x[p].x;
            v.y += x[p].y;
            v.z += x[p].z;
            v.w += x[p].w;
        }
    }
    return v;
}

// Store four consecutive values of one output row, columns [col0, col0 + nvalid).
__device__ __forceinline__ void store_quad(void* base, int64_t ldo, int out_f32, int64_t row, int col0, int nvalid,
                                           const float (&v)[4]) {
    if (out_f32) {
        float* p = static_cast<float*>(base) + row * ldo + col0;
        if (nvalid == 4 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
            *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nvalid) p[e] = v[e];
        }
    } else {
        uint16_t* p = static_cast<uint16_t*>(base) + row * ldo + col0;
        if (nvalid == 4 && (reinterpret_cast<uintptr_t>(p) & 7) == 0) {
            *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nvalid) p[e] = f32_to_bf16(v[e]);
        }
    }
}

template <int BN, int STAGES, int EPI, int KSUB, int ROWS>
__global__ void __launch_bounds__(kThreads, 1) tp_gemm_splitk_kernel(const __grid_constant__ GemmArgs args) {
    using Cfg = SplitCfg<BN, STAGES, EPI, ROWS>;
    static_assert(KSUB >= 1 && STAGES % KSUB == 0, "stage groups of KSUB blocks (as in tp_gemm_kernel)");
    constexpr int GROUPS = STAGES / KSUB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    constexpr int kStagingOff = Cfg::STAGING_IN_RING ? 0 : STAGES * Cfg::STAGE_BYTES;
    constexpr int kBarOff = STAGES * Cfg::STAGE_BYTES + (Cfg::STAGING_IN_RING ? 0 : Cfg::STAGING_BYTES);
    const uint32_t staging = base + kStagingOff;
    float4* staging_ptr = reinterpret_cast<float4*>(base_ptr + kStagingOff);
    const uint32_t bar_base = base + kBarOff;
    uint8_t* bar_ptr = base_ptr + kBarOff;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar_base + 8u * (2 * STAGES + 2 + a); };
    const uint32_t staged_bar = bar_base + 8u * (2 * STAGES + 4);
    const uint32_t drained_bar = bar_base + 8u * (2 * STAGES + 5);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + 8 * Cfg::NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_ptr + 8 * Cfg::NBARS + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cs = args.split;
    const int crank = static_cast<int>(cluster_ctarank());
    const int cluster = blockIdx.x / cs;
    const int nclusters = gridDim.x / cs;
    // this CTA's K blocks of every tile, in the order (segment, block) of the whole K
    const int kb_all = args.k_blocks * args.segs;
    const int kb_lo = static_cast<int>(static_cast<int64_t>(crank) * kb_all / cs);
    const int kb_hi = static_cast<int>(static_cast<int64_t>(crank + 1) * kb_all / cs);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128);
        }
        // one arrival per epilogue warp of every CTA of the cluster (this CTA's own warps
        // too: a row staged by one warp is reduced by others)
        mbar_init(staged_bar, cs * 4);
        mbar_init(drained_bar, cs * 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        const int nmaps = args.segs > 1 ? args.segs : args.groups;
        for (int i = 0; i < nmaps && i < TP_MAX_SHARDS; ++i) prefetch_tmap(&args.mapB[i]);
        prefetch_tmap(&args.mapA[0]);
    }
    if (warp == 1) tmem_alloc<Cfg::TMEM_COLS>(smem_u32(tmem_slot));
    __syncwarp();
    tc_fence_before();
    cluster_sync();                                      // every CTA's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) pdl_trigger();
    bool aborted = false;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // rotate_k: each CTA holds whole segments; start each segment's loop elsewhere
            auto kblock = [&](int kk, int rot, int g, int& kb, int& ai, int& bi) {
                const int seg = kk / args.k_blocks;
                kb = kk - seg * args.k_blocks + rot;
                if (kb >= args.k_blocks) kb -= args.k_blocks;
                ai = args.segs > 1 ? seg : (args.a_per_group ? g : 0);
                bi = args.segs > 1 ? seg : g;
            };
            auto load_b = [&](uint32_t sb, int bi, uint32_t bar, int kb, int n) {
                if (EPI == EPI_GLU) {   // gate rows and the same rows of up, one 3-D box
                    tma_load_3d(sb, &args.mapB[bi], bar, kb * BK, n * (BN / 2), 0);
                } else {
                    tma_load_2d(sb, &args.mapB[bi], bar, kb * BK, n * BN);
                }
            };
            // B of the first ring fill before waiting for the previous grid of the stream, when
            // that grid is a kernel of the same call (only A can be its output)
            const uint32_t block_bytes = static_cast<uint32_t>(args.a_box_rows * 128 + Cfg::B_BYTES);
            const int nkb = kb_hi - kb_lo;
            int pre = 0;                                   // blocks of the first tile already armed
            if (args.pdl_prefetch && cluster < args.total_tiles) {
                int g, m, n;
                tile_coords(args, cluster, g, m, n);
                const int rot = args.rotate_k ? cluster % args.k_blocks : 0;
                pre = min(STAGES, nkb);
                for (int gi = 0; gi * KSUB < pre; ++gi) {
                    const int cnt = min(KSUB, nkb - gi * KSUB);
                    mbar_arrive_expect_tx(full_bar(gi), static_cast<uint32_t>(cnt) * block_bytes);
                    for (int i = 0; i < cnt; ++i) {
                        int kb, ai, bi;
                        kblock(kb_lo + gi * KSUB + i, rot, g, kb, ai, bi);
                        load_b(base + (gi * KSUB + i) * Cfg::STAGE_BYTES + Cfg::A_BYTES, bi, full_bar(gi), kb, n);
                    }
                }
            }
            pdl_wait();
            int grp = 0;
            uint32_t phase = 0;
            for (int tile = cluster; tile < args.total_tiles && !aborted; tile += nclusters) {
                int g, m, n;
                tile_coords(args, tile, g, m, n);
                const int rot = args.rotate_k ? tile % args.k_blocks : 0;
                int seg = kb_lo / args.k_blocks, kin = kb_lo - (kb_lo / args.k_blocks) * args.k_blocks;
                for (int kk = 0; kk < nkb; kk += KSUB) {
                    const int cnt = min(KSUB, nkb - kk);
                    const bool armed = tile == cluster && kk < pre;   // B in flight since the prefetch
                    const uint32_t bar = full_bar(grp);
                    if (!armed) {
                        if (!mbar_wait(empty_bar(grp), phase ^ 1u, abort_flag, args.status)) {
                            aborted = true;
                            break;
                        }
                        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(cnt) * block_bytes);
                    }
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        if (i < cnt) {
                            int kb = kin + rot;            // (segment, block) advanced without division
                            if (kb >= args.k_blocks) kb -= args.k_blocks;
                            const int ai = args.segs > 1 ? seg : (args.a_per_group ? g : 0);
                            const int bi = args.segs > 1 ? seg : g;
                            if (++kin == args.k_blocks) {
                                kin = 0;
                                ++seg;
                            }
                            const uint32_t sa = base + (grp * KSUB + i) * Cfg::STAGE_BYTES;
                            tma_load_2d(sa, &args.mapA[ai], bar, kb * BK, m * BM);
                            if (!armed) load_b(sa + Cfg::A_BYTES, bi, bar, kb, n);
                        }
                    }
                    if (++grp == GROUPS) {
                        grp = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = mma_idesc_bf16(BM, BN);
            int grp = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            const int nkb = kb_hi - kb_lo;
            for (int tile = cluster; tile < args.total_tiles && !aborted; tile += nclusters) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, args.status)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kk = 0; kk < nkb; kk += KSUB) {
                    const int cnt = min(KSUB, nkb - kk);
                    if (!mbar_wait(full_bar(grp), phase, abort_flag, args.status)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int i = 0; i < KSUB; ++i) {
                        if (i < cnt) {
                            const uint32_t sa = base + (grp * KSUB + i) * Cfg::STAGE_BYTES;
                            const uint64_t adesc = sw128_kmajor_desc(sa);
                            const uint64_t bdesc = sw128_kmajor_desc(sa + Cfg::A_BYTES);
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k)
                                tc_mma(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, ((kk + i) | k) != 0 ? 1u : 0u);
                        }
                    }
                    tc_commit(empty_bar(grp));
                    if (++grp == GROUPS) {
                        grp = 0;
                        phase ^= 1u;
                    }
                }
                if (aborted) break;
                tc_commit(tfull_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;                   // accumulator row = TMEM lane
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t j = 0;                                  // tiles done by this CTA
        for (int tile = cluster; tile < args.total_tiles; tile += nclusters, ++j) {
            int g, m, n;
            tile_coords(args, tile, g, m, n);
            const int64_t grow = static_cast<int64_t>(m) * BM + row;
            const bool row_ok = row < Cfg::ROWS && grow < args.M;
            if (!mbar_wait_warp(tfull_bar(acc), acc_phase, abort_flag, args.status)) {
                aborted = true;
                break;
            }
            // every peer has read this CTA's staging of the previous tile
            if (j > 0 && !mbar_wait_cluster_warp(drained_bar, (j - 1) & 1u, abort_flag, args.status)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            const bool warp_live = q * 32 < Cfg::ROWS && static_cast<int64_t>(m) * BM + q * 32 < args.M;
#pragma unroll 1
            for (int c = 0; c < (warp_live ? BN / 32 : 0); ++c) {
                uint32_t r[32];
                tmem_ld32(taddr + c * 32, r);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        staging_ptr[(c * 8 + i) * Cfg::ROWS + row] =
                            make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                        __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(acc));                // the accumulator is free for the next tile
            // The warp's staged rows are visible to the cluster once lane 0's arrives are: the warp
            // barrier orders every lane's writes before lane 0's fence, and the fence followed by
            // the relaxed arrives is a release (one fence, not one release per peer).
            __syncwarp();
            if (lane == 0) {
                fence_acq_rel_cluster();
                for (int p = 0; p < cs; ++p)
                    mbar_arrive_cluster_relaxed(mapa_shared(staged_bar, static_cast<uint32_t>(p)));
            }
            if (!mbar_wait_cluster_warp(staged_bar, j & 1u, abort_flag, args.status)) {
                aborted = true;
                break;
            }
            void* out = args.out[g];
            const uint16_t* bias = static_cast<const uint16_t*>(args.bias[g]);
            const int ncols = args.n_valid[g];
            // The 128 epilogue threads share the reduction: item = (owned chunk, live row,
            // 4-column group), the 4-column group fastest so that 8 threads store one row's
            // 32 columns together.  Chunk c belongs to rank c mod CS.
            const int64_t left = args.M - static_cast<int64_t>(m) * BM;
            const int rows = left < Cfg::ROWS ? static_cast<int>(left) : Cfg::ROWS;
            const int owned = (Cfg::OUT_CHUNKS - crank + cs - 1) / cs;
            const int items = owned * rows * 8;
#pragma unroll 1
            for (int it = static_cast<int>(threadIdx.x) - 64; it < items; it += 128) {
                const int i = it & 7;
                const int rest = it >> 3;
                const int r = rest % rows;
                const int c = crank + (rest / rows) * cs;
                const int col0 = n * (Cfg::OUT_CHUNKS * 32) + c * 32 + 4 * i;
                if (col0 >= ncols) continue;
                const int nvalid = min(4, ncols - col0);
                const float4 a = gather_f4<Cfg::ROWS>(staging, c * 8 + i, r, cs);
                float v[4] = {a.x, a.y, a.z, a.w};
                if (EPI == EPI_GLU) {
                    const float4 u = gather_f4<Cfg::ROWS>(staging, (BN / 2) / 4 + c * 8 + i, r, cs);
                    v[0] = act_fn(v[0], args.act) * u.x;
                    v[1] = act_fn(v[1], args.act) * u.y;
                    v[2] = act_fn(v[2], args.act) * u.z;
                    v[3] = act_fn(v[3], args.act) * u.w;
                } else if (bias != nullptr) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (e < nvalid) v[e] += bf16_to_f32(bias[col0 + e]);
                }
                store_quad(out, args.ldo, args.out_f32, static_cast<int64_t>(m) * BM + r, col0, nvalid, v);
            }
            // This warp has read (and consumed) its share of every peer's staging; a relaxed
            // arrive suffices, since no peer needs this warp's output stores ordered.  After the
            // CTA's last tile nobody waits on the drained barriers: no arrive is sent, so that no
            // remote arrive can still be in flight at teardown.
            __syncwarp();
            if (lane == 0 && tile + nclusters < args.total_tiles)
                for (int p = 0; p < cs; ++p)
                    mbar_arrive_cluster_relaxed(mapa_shared(drained_bar, static_cast<uint32_t>(p)));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    if (aborted) spin_ns(50000);
    __syncwarp();                                        // reconverge the lane-0 roles (aligned barrier below)
    tc_fence_before();
    // Peers may read this CTA's staging until they reach this barrier.  Every such read was
    // consumed (its value stored) before the reader arrives, every staged arrive was observed
    // by its target's staged wait, and the last tile sends no drained arrives, so nothing
    // remote is in flight: the arrive need not wait for this CTA's output stores.
    cluster_sync_relaxed();
    if (*abort_flag) spin_ns(50000);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<Cfg::TMEM_COLS>(tmem_base);
    }
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static std::atomic<EncodeTiledFn> cached{nullptr};  // racing first calls store the same entry point
    EncodeTiledFn fn = cached.load(std::memory_order_relaxed);
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
        cached.store(fn, std::memory_order_relaxed);
    }
    return fn;
}

// Encoded tensor maps, cached per host thread.  A GEMM call encodes one map
// per operand and shard (up to 16), and an encoding depends only on the
// pointer, the extents, the strides and the box, so a call that repeats an
// earlier call's operands (every decode step, every layer of a replayed
// schedule) copies the earlier encodings instead of encoding again.  The
// cache is direct-mapped; a collision overwrites the older entry.
struct MapKey {
    const void* ptr;
    uint64_t dims[4];
    uint64_t strides[3];
    uint32_t box[4];
    uint32_t rank;
    bool operator==(const MapKey& o) const {
        if (ptr != o.ptr || rank != o.rank) return false;
        for (int i = 0; i < 4; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
        for (int i = 0; i < 3; ++i)
            if (strides[i] != o.strides[i]) return false;
        return true;
    }
};
struct MapEntry {
    CUtensorMap map;
    MapKey key;
    bool valid;
};
constexpr int kMapCacheSlots = 128;

static MapEntry& map_slot(const MapKey& k) {
    thread_local MapEntry cache[kMapCacheSlots];
    uint64_t h = reinterpret_cast<uintptr_t>(k.ptr) * 0x9E3779B97F4A7C15ull;
    for (uint64_t v : {k.dims[0], k.dims[1], k.dims[2], k.dims[3], k.strides[0], k.strides[1], k.strides[2],
                       static_cast<uint64_t>(k.box[0]) | static_cast<uint64_t>(k.box[1]) << 16 |
                           static_cast<uint64_t>(k.box[2]) << 32 | static_cast<uint64_t>(k.box[3]) << 48,
                       static_cast<uint64_t>(k.rank)})
        h = (h ^ v) * 0x100000001B3ull;
    return cache[(h >> 32) % kMapCacheSlots];
}

// Encode (or copy from the cache) one bf16 tensor map of rank 2 to 4 with
// 128-byte swizzle and the given box (innermost first).
static bool encode_map_box(CUtensorMap* m, const void* ptr, uint32_t rank, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box) {
    if (rank < 2 || rank > 4) return false;
    MapKey k = {};
    k.ptr = ptr;
    k.rank = rank;
    for (uint32_t i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
    }
    for (uint32_t i = 0; i + 1 < rank; ++i) k.strides[i] = strides[i];
    MapEntry& e = map_slot(k);
    if (e.valid && e.key == k) {
        *m = e.map;
        return true;
    }
    EncodeTiledFn enc = get_encode_fn();
    if (enc == nullptr) return false;
    cuuint32_t bx[4] = {box[0], box[1], rank > 2 ? box[2] : 1u, rank > 3 ? box[3] : 1u};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, bx, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    e.map = *m;
    e.key = k;
    e.valid = true;
    return true;
}

// Boxes of 64 elements by box_rows rows (by 2 in the third dimension).
static bool encode_map(CUtensorMap* m, const void* ptr, uint32_t rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, int box_rows) {
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 2};
    return encode_map_box(m, ptr, rank, dims, strides, box);
}

// bf16 K-major operand [rows, cols] with row stride ld (elements), tiles of
// box_rows x 64 with 128-byte swizzle; out-of-range elements read as zero.
static bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    return encode_map(m, ptr, 2, dims, strides, box_rows);
}

static int sm_count() {
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

// Row-tiles per raster band: as many as keep about kRasterBandMB of A rows
// (the operand a band re-reads for every column of tiles) resident in L2.
constexpr int kRasterBandMB = 64;
constexpr int kBandsSpanGroups = 1;
static int raster_band(int tile_rows, int64_t k_total) {
    const int64_t tile_bytes = static_cast<int64_t>(tile_rows) * k_total * 2;
    const int64_t band = (static_cast<int64_t>(kRasterBandMB) << 20) / std::max<int64_t>(tile_bytes, 1);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(band, 64)));
}

// Opt a kernel into its dynamic shared memory.  The attribute lasts for the
// process, so it is set once per device (bit `dev` of `done`, one word per
// kernel instantiation) and later launches skip the driver call.
bool smem_attribute_once(const void* kern, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    if (bit != 0) done.fetch_or(bit, std::memory_order_relaxed);
    return true;
}

// Programmatic dependent launch (GemmDesc::pdl): the attribute lets the GEMM
// start before the previous kernel of the stream ends; its producer waits
// (pdl_wait) before loading what that kernel may have written.
static void set_pdl(cudaLaunchAttribute& at) {
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
}

// Tensor map of a gated B block [2 * half_rows, cols] (gate rows, then the same
// rows of up) as a 3-D tensor {cols, half_rows, 2}: one box of box_rows rows of
// each half lands as the gate tile followed by the up tile, in one TMA load.
static bool make_map_glu(CUtensorMap* m, const void* ptr, int64_t half_rows, int64_t cols, int64_t ld, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(half_rows), 2};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(half_rows * ld) * 2};
    return encode_map(m, ptr, 3, dims, strides, box_rows);
}

bool make_operand_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    return make_map(m, ptr, rows, cols, ld, box_rows);
}

bool make_gated_operand_map(CUtensorMap* m, const void* ptr, int64_t half_rows, int64_t cols, int64_t ld,
                            int box_rows) {
    return make_map_glu(m, ptr, half_rows, cols, ld, box_rows);
}

bool make_kblock_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t k, int64_t ld, int box_rows,
                     int box_kblocks) {
    if (k % BK != 0) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(k / BK)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(BK) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows),
                               static_cast<cuuint32_t>(box_kblocks)};
    return encode_map_box(m, ptr, 3, dims, strides, box);
}

bool make_gated_kblock_map(CUtensorMap* m, const void* ptr, int64_t half_rows, int64_t k, int64_t ld, int box_rows,
                           int box_kblocks) {
    if (k % BK != 0) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(half_rows), 2,
                                static_cast<cuuint64_t>(k / BK)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(half_rows * ld) * 2,
                                   static_cast<cuuint64_t>(BK) * 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 2,
                               static_cast<cuuint32_t>(box_kblocks)};
    return encode_map_box(m, ptr, 4, dims, strides, box);
}

bool make_row_tile_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int tile_rows,
                       int box_tiles) {
    if (rows % tile_rows != 0) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(tile_rows),
                                static_cast<cuuint64_t>(rows / tile_rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(ld * tile_rows) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(tile_rows),
                               static_cast<cuuint32_t>(box_tiles)};
    return encode_map_box(m, ptr, 3, dims, strides, box);
}

template <int BN, int STAGES, int EPI, int AROWS = BM, int KSUB = 1>
static tp_status launch_cfg(GemmArgs& a, const GemmDesc& d, cudaStream_t stream) {
    using Cfg = GemmCfg<BN, STAGES, EPI, AROWS>;
    if (AROWS < BM && d.M > AROWS) return TP_ERR_UNSUPPORTED;   // a short A tile holds one m-tile
    a.n_tiles = (d.N + Cfg::OUT_COLS - 1) / Cfg::OUT_COLS;
    a.total_tiles = a.groups * a.m_tiles * a.n_tiles;
    if (a.total_tiles == 0) return TP_OK;
    const int b_box = (EPI == EPI_GLU) ? BN / 2 : BN;
    const int nA = d.segs > 1 ? d.segs : (d.a_per_group ? d.groups : 1);
    const int nB = d.segs > 1 ? d.segs : d.groups;
    // A box only as tall as the rows that exist (decode: a handful of tokens);
    // the rest of the 128-row shared tile is never read into an output row.
    a.a_box_rows = static_cast<int>(std::min<int64_t>(BM, (d.M + 7) / 8 * 8));
    a.group_m = raster_band(BM, d.K * d.segs);
    // decode-sized A; with K segments the rotation stays inside each segment,
    // so the fused reduce still adds the shards in rank order
    a.rotate_k = d.M <= 64 ? 1 : 0;
    // Groups of KSUB K blocks load as one A box and one B box when every group is whole (a
    // copy has a large fixed cost: at one box per K block a CTA streamed about 45 GB/s).
    // Used with the 64-row A tiles (9 to 64 tokens: 70B MLP decode 0.5-0.8 % faster, the QKV
    // GEMM 1.1-1.5 %); with the 8-row tiles it gained nothing and the tiny MLP's two-GEMM path
    // lost 1-2 %, so those keep one box per K block.
    a.kgroup_box = (KSUB > 1 && (AROWS == 64 || AROWS == 16) && d.K % (static_cast<int64_t>(BK) * KSUB) == 0) ? 1 : 0;
    for (int i = 0; i < nA; ++i) {
        const bool ok = a.kgroup_box ? make_kblock_map(&a.mapA[i], d.a[i], d.M, d.K, d.lda, a.a_box_rows, KSUB)
                                     : make_map(&a.mapA[i], d.a[i], d.M, d.K, d.lda, a.a_box_rows);
        if (!ok) return TP_ERR_CUDA;
    }
    for (int i = 0; i < nB; ++i) {
        const int64_t rows = (d.segs == 1 && d.n_valid[i] > 0 && !d.glu) ? d.n_valid[i] : d.b_rows;
        bool ok;
        if (EPI == EPI_GLU)
            ok = a.kgroup_box ? make_gated_kblock_map(&a.mapB[i], d.b[i], d.glu_up_row, d.K, d.ldb, b_box, KSUB)
                              : make_map_glu(&a.mapB[i], d.b[i], d.glu_up_row, d.K, d.ldb, b_box);
        else
            ok = a.kgroup_box ? make_kblock_map(&a.mapB[i], d.b[i], rows, d.K, d.ldb, b_box, KSUB)
                              : make_map(&a.mapB[i], d.b[i], rows, d.K, d.ldb, b_box);
        if (!ok) return TP_ERR_CUDA;
    }
    auto kern = tp_gemm_kernel<BN, STAGES, EPI, AROWS, KSUB>;
    static std::atomic<uint64_t> smem_set{0};
    if (!smem_attribute_once(reinterpret_cast<const void*>(kern), Cfg::SMEM_BYTES, smem_set)) return TP_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return TP_ERR_CUDA;
    const int grid = std::min(a.total_tiles, sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_pdl(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = d.pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return TP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

template <int STAGES, int EPI, int KSUB = 1>
static tp_status launch_pair(GemmArgs& a, const GemmDesc& d, cudaStream_t stream) {
    using Cfg = PairCfg<STAGES, EPI>;
    a.m_tiles = static_cast<int>((d.M + Cfg::TILE_M - 1) / Cfg::TILE_M);
    a.group_m = raster_band(Cfg::TILE_M, d.K * d.segs);
    a.bands_span_groups = (kBandsSpanGroups && d.groups > 1 && !d.a_per_group && d.segs == 1) ? 1 : 0;
    a.a_box_rows = 128;
    a.n_tiles = static_cast<int>((d.N + Cfg::OUT_COLS - 1) / Cfg::OUT_COLS);
    a.total_tiles = a.groups * a.m_tiles * a.n_tiles;
    if (a.total_tiles == 0) return TP_OK;
    const int nA = d.segs > 1 ? d.segs : (d.a_per_group ? d.groups : 1);
    const int nB = d.segs > 1 ? d.segs : d.groups;
    for (int i = 0; i < nA; ++i)
        if (!make_map(&a.mapA[i], d.a[i], d.M, d.K, d.lda, 128)) return TP_ERR_CUDA;
    for (int i = 0; i < nB; ++i) {
        const int64_t rows = (d.segs == 1 && d.n_valid[i] > 0 && !d.glu) ? d.n_valid[i] : d.b_rows;
        if (!make_map(&a.mapB[i], d.b[i], rows, d.K, d.ldb, 128)) return TP_ERR_CUDA;
    }
    auto kern = tp_gemm_pair_kernel<STAGES, EPI, KSUB>;
    static std::atomic<uint64_t> smem_set{0};
    if (!smem_attribute_once(reinterpret_cast<const void*>(kern), Cfg::SMEM_BYTES, smem_set)) return TP_ERR_CUDA;
    const int sms = sm_count();
    if (sms < 2) return TP_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // A persistent grid of pairs that can all be resident at once (per device).
    static std::atomic<int> max_clusters[64];  // relaxed: racing first calls store the same value
    int dev = 0;
    cudaGetDevice(&dev);
    const bool cached_dev = dev >= 0 && dev < 64;
    int mc = cached_dev ? max_clusters[dev].load(std::memory_order_relaxed) : 0;
    if (mc <= 0) {
        int v = 0;
        if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess || v <= 0) v = sms / 2;
        mc = std::min(v, sms / 2);
        if (cached_dev) max_clusters[dev].store(mc, std::memory_order_relaxed);
    }
    int clusters = std::min(a.total_tiles, mc);
    // Stream-K (store epilogue, given a workspace).  When the last wave of whole tiles would leave
    // pairs idle, its L tiles are cut into S = pairs / L parts along K, one unit per pair, so
    // that wave takes about 1/S of a tile's time.  When there are fewer tiles than resident
    // pairs (L = all of them, no whole wave), every tile is cut the same way and the grid grows
    // to L x S pairs, each running one unit.  Each part keeps at least two groups of K blocks.
    a.sk_first = a.total_tiles;
    a.sk_parts = 1;
    if (EPI == EPI_STORE && d.sk_ws != nullptr) {
        const int waves = a.total_tiles / mc;
        const int tail = a.total_tiles - waves * mc;
        const int kbt = a.k_blocks * d.segs;
        const int parts = tail > 0 ? std::min(std::min(mc / tail, kSkMaxParts), kbt / (2 * KSUB)) : 1;
        const int64_t slots = static_cast<int64_t>(tail) * (parts - 1);
        if (parts >= 2 && slots <= kSkMaxSlots && slots * 2 * 4 <= static_cast<int64_t>(kSkFlagBytes) &&
            kSkFlagBytes + static_cast<size_t>(slots) * kSkSlotBytes <= d.sk_ws_bytes) {
            a.sk_first = waves * mc;
            a.sk_parts = parts;
            a.sk_flags = static_cast<int*>(d.sk_ws);
            a.sk_scratch = reinterpret_cast<float*>(static_cast<char*>(d.sk_ws) + kSkFlagBytes);
            if (waves == 0) clusters = tail * parts;   // <= mc: every unit's pair is resident
        }
    }
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.numAttrs = d.pdl ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return TP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

template <int BN, int STAGES, int EPI, int KSUB = 1, int ROWS = 64>
static tp_status launch_split(GemmArgs& a, const GemmDesc& d, int cs, cudaStream_t stream) {
    using Cfg = SplitCfg<BN, STAGES, EPI, ROWS>;
    const int kb_all = a.k_blocks * d.segs;
    if (d.M > Cfg::ROWS || cs < 2 || cs > 8 || cs > kb_all) return TP_ERR_UNSUPPORTED;
    a.split = cs;
    a.m_tiles = 1;
    a.n_tiles = static_cast<int>((d.N + Cfg::OUT_CHUNKS * 32 - 1) / (Cfg::OUT_CHUNKS * 32));
    a.total_tiles = d.groups * a.n_tiles;
    a.group_m = 1;
    a.a_box_rows = static_cast<int>((d.M + 7) / 8 * 8);
    // whole segments per CTA: spread the weight reads by starting each segment's K loop elsewhere
    a.rotate_k = (d.segs > 1 && d.segs % cs == 0) ? 1 : 0;
    auto kern = tp_gemm_splitk_kernel<BN, STAGES, EPI, KSUB, ROWS>;
    static std::atomic<uint64_t> smem_set{0};
    if (!smem_attribute_once(reinterpret_cast<const void*>(kern), Cfg::SMEM_BYTES, smem_set)) return TP_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs * a.total_tiles, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent: no more clusters than can be resident at once (cached per device and size)
    static std::atomic<int> max_clusters[64][9];  // relaxed: racing first calls store the same value
    int dev = 0;
    cudaGetDevice(&dev);
    const bool cached_dev = dev >= 0 && dev < 64;
    int mc = cached_dev ? max_clusters[dev][cs].load(std::memory_order_relaxed) : 0;
    if (mc <= 0) {
        int v = 0;
        if (cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess || v <= 0) return TP_ERR_CUDA;
        mc = v;
        if (cached_dev) max_clusters[dev][cs].store(mc, std::memory_order_relaxed);
    }
    const int cap = d.split_clusters > 0 ? std::min(mc, d.split_clusters) : mc;
    // staging in the ring needs one tile per cluster: the caller falls back to another configuration
    if (Cfg::STAGING_IN_RING && a.total_tiles > cap) return TP_ERR_UNSUPPORTED;
    const int nA = d.segs > 1 ? d.segs : (d.a_per_group ? d.groups : 1);
    const int nB = d.segs > 1 ? d.segs : d.groups;
    const int b_box = EPI == EPI_GLU ? BN / 2 : BN;
    for (int i = 0; i < nA; ++i)
        if (!make_map(&a.mapA[i], d.a[i], d.M, d.K, d.lda, a.a_box_rows)) return TP_ERR_CUDA;
    for (int i = 0; i < nB; ++i) {
        const int64_t rows = (d.segs == 1 && d.n_valid[i] > 0 && !d.glu) ? d.n_valid[i] : d.b_rows;
        const bool ok = (EPI == EPI_GLU) ? make_map_glu(&a.mapB[i], d.b[i], d.glu_up_row, d.K, d.ldb, b_box)
                                         : make_map(&a.mapB[i], d.b[i], rows, d.K, d.ldb, b_box);
        if (!ok) return TP_ERR_CUDA;
    }
    cfg.gridDim = dim3(cs * std::min(a.total_tiles, cap), 1, 1);
    cfg.numAttrs = d.pdl ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) return TP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

// Split-K plan for GEMMs of at most 64 rows: the tile width (256 or 128) and
// cluster size that put the most CTAs to work, one per SM at most, with at
// least two K blocks per CTA.  Returns the cluster size, 0 for no split
// (not the fused reduce, the plain kernel already has a tile for every SM,
// or K is too short).
static int split_plan(const GemmDesc& d, int sms, int& bn) {
    if (d.M > 64 || d.split < 0) return 0;
    // automatic only for the fused reduce: with one output per shard the plain kernel has
    // t times the tiles and was as fast or faster in every measured shape
    if (d.split == 0 && (d.force_bn != 0 || d.pair > 0 || d.segs < 2)) return 0;
    const bool always = d.split > 0;
    const int64_t kb_all = (d.K + BK - 1) / BK * d.segs;
    const int cs_max = static_cast<int>(std::min<int64_t>(8, kb_all / 2));
    int best_cs = 0, best_ctas = 0;
    bn = 0;
    for (int w : {256, 128}) {
        const int out_cols = d.glu ? w / 2 : w;
        const int64_t tiles = d.groups * ((d.N + out_cols - 1) / out_cols);
        if (tiles >= sms && !always) continue;           // the plain kernel already fills the GPU
        const int cs = always ? cs_max : static_cast<int>(std::min<int64_t>(cs_max, sms / tiles));
        if (cs < 2) continue;
        const int ctas = static_cast<int>(std::min<int64_t>(tiles * cs, sms));
        if (ctas > best_ctas) {
            best_ctas = ctas;
            best_cs = cs;
            bn = w;
        }
    }
    return best_cs;
}

// Estimated time units of a launch with output tile width w: whole waves of
// tiles times the per-tile cost (proportional to the MMA N plus a fixed
// share for the A tile).
static long long plan_cost(int tiles, int bn, int sms) {
    const long long waves = (tiles + sms - 1) / sms;
    return waves * (bn + 32);
}

// Kernel, tile width and split-K cluster size for a GEMM on `sms` SMs (pure host
// logic: the launch below follows it, and tp_debug_gemm_plan exposes it to tests).
GemmPlan plan_gemm(const GemmDesc& d, int sms) {
    const int m_tiles = static_cast<int>((d.M + BM - 1) / BM);
    const bool glu = d.glu != 0;
    // Candidate MMA widths, largest first; pick the one with the lowest cost.  96 (store
    // epilogue only: a gated tile splits into gate and up halves of whole 32-column chunks)
    // spreads a narrow weight over more SMs, e.g. 112 tiles instead of 80 for the 1280-row
    // QKV blocks of 8 ranks.
    const int cands[4] = {256, 128, 96, 64};
    int best = 256;
    long long best_cost = -1;
    for (int bn : cands) {
        if (glu && bn == 96) continue;
        const int out_cols = glu ? bn / 2 : bn;
        const int tiles = d.groups * m_tiles * static_cast<int>((d.N + out_cols - 1) / out_cols);
        const long long c = plan_cost(tiles, bn, sms);
        if (best_cost < 0 || c < best_cost) {
            best_cost = c;
            best = bn;
        }
    }
    if (d.force_bn) best = (glu && d.force_bn == 96) ? 128 : d.force_bn;
    // CTA pairs whenever they need no more waves than single CTAs with the same tile width
    // (a pair tile holds 256 rows on two SMs, a single-CTA tile 128 rows on one; per wave the
    // pair kernel does the same work per SM at a higher tensor-pipe rate).  Measured on the 70B
    // MLP: pairs win at n = 256 (3 waves either way) and 512, lose at n = 128 and for the down
    // GEMM at n = 384, where they would add a wave.
    bool pair = false;
    if (d.pair >= 0 && sms >= 2) {
        const int out_cols = glu ? 128 : 256;
        const long long col_tiles = static_cast<long long>(d.groups) * ((d.N + out_cols - 1) / out_cols);
        const long long pair_waves = (col_tiles * ((d.M + 255) / 256) + sms / 2 - 1) / (sms / 2);
        const long long single_waves = (col_tiles * ((d.M + 127) / 128) + sms - 1) / sms;
        pair = d.pair > 0 || (d.M > 128 && d.force_bn == 0 && pair_waves <= single_waves);
    }
    GemmPlan p;
    p.bn = best;
    if (pair) {
        p.kind = 1;
        p.bn = 256;
        return p;
    }
    int split_bn = 0;
    const int cs = split_plan(d, sms, split_bn);
    if (cs >= 2) {
        p.kind = 2;
        p.bn = split_bn;
        p.cs = cs;
    }
    return p;
}

tp_status launch_gemm(const GemmDesc& d, cudaStream_t stream) {
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int g = 0; g < d.groups; ++g) {
        a.out[g] = d.out[g];
        a.bias[g] = d.bias[g];
        a.n_valid[g] = static_cast<int>(d.n_valid[g] > 0 ? d.n_valid[g] : d.N);
    }
    a.ldo = d.ldo;
    a.out_f32 = d.out_f32;
    a.M = static_cast<int>(d.M);
    a.N = static_cast<int>(d.N);
    a.m_tiles = static_cast<int>((d.M + BM - 1) / BM);
    a.groups = d.groups;
    a.k_blocks = static_cast<int>((d.K + BK - 1) / BK);
    a.segs = d.segs;
    a.a_per_group = d.a_per_group;
    a.glu_up_row = static_cast<int>(d.glu_up_row);
    a.act = d.act;
    a.status = d.status;
    a.pdl_prefetch = d.pdl == 1 ? 1 : 0;
    if (d.M == 0 || d.N == 0) return TP_OK;
    // tile indices are 32-bit in the kernels
    if (static_cast<int64_t>(d.groups) * ((d.M + 127) / 128) * ((d.N + 63) / 64) > INT32_MAX) return TP_ERR_UNSUPPORTED;

    const GemmPlan plan = plan_gemm(d, std::max(1, sm_count()));
    const bool glu = d.glu != 0;
    const int best = plan.bn;
    if (plan.kind == 1) {
        if (glu) return launch_pair<kPairStages, EPI_GLU, kPairKsub>(a, d, stream);
        return launch_pair<kPairStages, EPI_STORE, kPairKsub>(a, d, stream);
    }
    if (plan.kind == 2) {
        const int cs = plan.cs;
        if (d.M <= 8) {   // 8 staged rows: 6 / 12 stages instead of 4 / 8
            if (glu) {
                if (plan.bn == 256) return launch_split<256, 6, EPI_GLU, 1, 8>(a, d, cs, stream);
                return launch_split<128, 12, EPI_GLU, 2, 8>(a, d, cs, stream);
            }
            if (plan.bn == 256) return launch_split<256, 6, EPI_STORE, 1, 8>(a, d, cs, stream);
            return launch_split<128, 12, EPI_STORE, 2, 8>(a, d, cs, stream);
        }
        if (d.M <= 16) {  // 16 staged rows: 6 / 12 stages as well
            if (glu) {
                if (plan.bn == 256) return launch_split<256, 6, EPI_GLU, 1, 16>(a, d, cs, stream);
                return launch_split<128, 12, EPI_GLU, 2, 16>(a, d, cs, stream);
            }
            if (plan.bn == 256) return launch_split<256, 6, EPI_STORE, 1, 16>(a, d, cs, stream);
            return launch_split<128, 12, EPI_STORE, 2, 16>(a, d, cs, stream);
        }
        if (glu) {
            if (plan.bn == 256) return launch_split<256, 4, EPI_GLU>(a, d, cs, stream);
            return launch_split<128, 8, EPI_GLU, 2>(a, d, cs, stream);
        }
        if (plan.bn == 256) {
            // five stages with the staging in the ring when every cluster runs one tile (the fused
            // down GEMM of 17-64 tokens, 32 tiles at h = 8192: about 1 % faster), else four
            const tp_status st = launch_split<256, 5, EPI_STORE>(a, d, cs, stream);
            if (st != TP_ERR_UNSUPPORTED) return st;
            return launch_split<256, 4, EPI_STORE>(a, d, cs, stream);
        }
        return launch_split<128, 8, EPI_STORE, 2>(a, d, cs, stream);
    }
    if (d.M <= 8) {    // one to eight tokens: 8-row A tiles, deeper B rings still
        if (glu) {
            if (best == 256) return launch_cfg<256, 6, EPI_GLU, 8>(a, d, stream);
            if (best == 128) return launch_cfg<128, 12, EPI_GLU, 8, 2>(a, d, stream);
            return launch_cfg<64, 20, EPI_GLU, 8, 4>(a, d, stream);
        }
        if (best == 256) return launch_cfg<256, 6, EPI_STORE, 8>(a, d, stream);
        if (best == 128) return launch_cfg<128, 12, EPI_STORE, 8, 2>(a, d, stream);
        if (best == 96) return launch_cfg<96, 16, EPI_STORE, 8, 2>(a, d, stream);
        return launch_cfg<64, 24, EPI_STORE, 8, 4>(a, d, stream);
    }
    if (d.M <= 16) {   // nine to sixteen tokens: 16-row A tiles, rings deeper than with 64 rows
        if (glu) {
            if (best == 256) return launch_cfg<256, 6, EPI_GLU, 16>(a, d, stream);
            if (best == 128) return launch_cfg<128, 10, EPI_GLU, 16, 2>(a, d, stream);
            return launch_cfg<64, 20, EPI_GLU, 16, 4>(a, d, stream);
        }
        if (best == 256) return launch_cfg<256, 6, EPI_STORE, 16>(a, d, stream);
        if (best == 128) return launch_cfg<128, 12, EPI_STORE, 16, 2>(a, d, stream);
        if (best == 96) return launch_cfg<96, 14, EPI_STORE, 16, 2>(a, d, stream);
        return launch_cfg<64, 20, EPI_STORE, 16, 4>(a, d, stream);
    }
    if (d.M <= 64) {   // decode: 64-row A tiles, deeper B rings
        if (glu) {
            if (best == 256) return launch_cfg<256, 5, EPI_GLU, 64>(a, d, stream);
            if (best == 128) return launch_cfg<128, 8, EPI_GLU, 64, 2>(a, d, stream);
            return launch_cfg<64, 12, EPI_GLU, 64, 4>(a, d, stream);
        }
        if (best == 256) return launch_cfg<256, 5, EPI_STORE, 64>(a, d, stream);
        if (best == 128) return launch_cfg<128, 8, EPI_STORE, 64, 2>(a, d, stream);
        if (best == 96) return launch_cfg<96, 10, EPI_STORE, 64, 2>(a, d, stream);
        return launch_cfg<64, 12, EPI_STORE, 64, 4>(a, d, stream);
    }
    if (glu) {
        if (best == 256) return launch_cfg<256, 4, EPI_GLU>(a, d, stream);
        if (best == 128) return launch_cfg<128, 6, EPI_GLU>(a, d, stream);
        return launch_cfg<64, 8, EPI_GLU>(a, d, stream);
    }
    if (best == 256) return launch_cfg<256, 4, EPI_STORE>(a, d, stream);
    if (best == 128) return launch_cfg<128, 6, EPI_STORE>(a, d, stream);
    if (best == 96) return launch_cfg<96, 8, EPI_STORE>(a, d, stream);
    return launch_cfg<64, 8, EPI_STORE>(a, d, stream);
}

}  // namespace tpk
