// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "tp.h"

namespace tpk {

// Stream-K tail of the CTA-pair GEMM with the store epilogue: when a
// workspace is given (GemmDesc::sk_ws), the tiles of a partial last wave are
// split along K into parts; every part after the first writes its fp32
// accumulator (256 x 256) to a slot of the workspace and raises a flag, and
// the first part adds them in order before its epilogue.  Workspace: flags
// (zeroed by the caller before the launch), then the slots.
constexpr size_t kSkFlagBytes = 4096;
constexpr size_t kSkSlotBytes = 256u * 256u * 4u;
constexpr int kSkMaxSlots = 128;
constexpr int kSkMaxParts = 4;
constexpr size_t kSkWorkspaceBytes = kSkFlagBytes + kSkMaxSlots * kSkSlotBytes;

// One tensor-parallel GEMM launch: for each group g,
//   D_g = sum_s A_{g,s} B_{g,s}^T, A [M, K] (lda), B [b_rows, K] (ldb), bf16.
struct GemmDesc {
    int64_t M = 0, N = 0, K = 0;        // K = per-segment depth
    int groups = 1;                      // independent outputs (shards)
    int segs = 1;                        // K segments summed into one output (fused reduce)
    int a_per_group = 0;                 // A operand differs per group
    const void* a[TP_MAX_SHARDS] = {};   // per group (a_per_group), per segment (segs > 1), or a[0]
    int64_t lda = 0;
    const void* b[TP_MAX_SHARDS] = {};   // per group, or per segment
    int64_t ldb = 0;
    int64_t b_rows = 0;                  // rows of each B matrix
    int64_t n_valid[TP_MAX_SHARDS] = {}; // per-group output width when groups differ (0: use N)
    int glu = 0;                         // gated epilogue: B = [gate rows; up rows]
    int64_t glu_up_row = 0;              // first up row inside B
    int act = TP_ACT_NONE;
    void* out[TP_MAX_SHARDS] = {};       // per-group output base
    const void* bias[TP_MAX_SHARDS] = {};
    int64_t ldo = 0;
    int out_f32 = 0;
    int* status = nullptr;
    int force_bn = 0;                    // 0: chosen by cost; else 64/128/256
    int pair = 0;                        // CTA-pair kernel: -1 never, 0 automatic, 1 always
    int split = 0;                       // split-K kernel (fused reduce, M <= 64): -1 never, 0 automatic, 1 always
    int split_clusters = 0;              // > 0: at most this many split-K clusters resident
    // Programmatic dependent launch: the launch may start before the previous kernel of
    // the stream ends, and its producer waits for that kernel (griddepcontrol.wait) before
    // loading.  1: the previous kernel belongs to the same library call and writes no B,
    // so the split-K and single-CTA kernels may load their first ring of B before the
    // wait; 2: the first
    // kernel of a call, whose predecessor may have written anything: nothing is loaded
    // before the wait.
    int pdl = 0;
    // Stream-K tail workspace (see kSkWorkspaceBytes), or null: the pair kernel
    // then runs whole tiles only.  Its flags must be zero when the launch starts.
    void* sk_ws = nullptr;
    size_t sk_ws_bytes = 0;
};

tp_status launch_gemm(const GemmDesc& d, cudaStream_t stream);

// Tensor maps of bf16 K-major operands as the GEMMs load them: 128-byte
// swizzle, boxes 64 elements wide (along K) by box_rows rows, out-of-range
// elements read as zero.  The gated form views [gate rows; up rows] as a 3-D
// tensor {cols, half_rows, 2}, so that one box brings box_rows gate rows
// followed by the same rows of up.  Encoded maps are cached per thread.
bool make_operand_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows);
bool make_gated_operand_map(CUtensorMap* m, const void* ptr, int64_t half_rows, int64_t cols, int64_t ld,
                            int box_rows);
// K-block views, for loading several K blocks with one copy: [rows, k] (row
// stride ld, k a multiple of 64) seen as {64, rows, k/64} with the K-block
// stride (128 bytes) below the row stride, so that one box {64, box_rows,
// box_kblocks} lands as box_kblocks consecutive [box_rows][64] tiles, each in
// the layout of a single-K-block box.  The gated form adds the gate/up
// dimension: a box holds, per K block, box_rows gate rows then the same up
// rows.
bool make_kblock_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t k, int64_t ld, int box_rows,
                     int box_kblocks);
bool make_gated_kblock_map(CUtensorMap* m, const void* ptr, int64_t half_rows, int64_t k, int64_t ld, int box_rows,
                           int box_kblocks);
// Row tiles: [rows, cols] (rows a multiple of tile_rows) seen as {cols,
// tile_rows, rows/tile_rows}; a box {64, tile_rows, box_tiles} lands as
// box_tiles consecutive [tile_rows][64] tiles.
bool make_row_tile_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int tile_rows,
                       int box_tiles);

// Opt a kernel into `bytes` of dynamic shared memory, once per device (bit
// `dev` of `done`, one word per kernel).
bool smem_attribute_once(const void* kern, int bytes, std::atomic<uint64_t>& done);

// The MLP of one to eight tokens in one GEMM kernel plus an ordered reduce
// (fused all-reduce): CTA pairs over 64-column slices of every rank's f
// columns, for h a multiple of 256 up to 1024 and f/t a multiple of 64, at
// most kSmallMlpMaxSlices slices.  Workspace: the slices' fp32 partials
// [f/64][n][h].
constexpr int kSmallMlpMaxRows = 8;
constexpr int kSmallMlpMaxSlices = 128;
struct SmallMlpDesc {
    int t = 0;
    int64_t n = 0, h = 0, f = 0;
    const void* x = nullptr;
    int64_t ldx = 0;
    const void* w_gate_up[TP_MAX_SHARDS] = {};   // [2 f/t, h]: gate rows, then up rows
    const void* w_down[TP_MAX_SHARDS] = {};      // [h, f/t], row stride ld_down
    int64_t ld_down = 0;
    const void* bias = nullptr;                   // [h] bf16 or null
    int act = TP_ACT_SILU_MUL;
    float* part = nullptr;                        // small_mlp_workspace bytes
    void* y = nullptr;                            // [n, h] contiguous
    int y_f32 = 0;
    int* status = nullptr;
};
// Workspace bytes of the one-kernel path, or 0 when it does not apply.
size_t small_mlp_workspace(int t, int64_t n, int64_t h, int64_t f, tp_reduce_mode mode);
tp_status launch_small_mlp(const SmallMlpDesc& d, cudaStream_t stream);

// Workspace bytes tp_mlp_forward cannot do without (H and the partials);
// tp_mlp_workspace_size adds the optional stream-K tail area.  0 for invalid
// arguments.
size_t mlp_workspace_required(int t, int64_t n, int64_t h, int64_t f, tp_reduce_mode mode, tp_dtype partial_dtype);

// The kernel launch_gemm picks for `d` on `sms` SMs: kind 0 = single-CTA tiles of
// width bn, 1 = CTA pairs (256 x 256 tiles), 2 = split-K clusters of cs CTAs on
// tiles of width bn.
struct GemmPlan {
    int kind = 0;
    int bn = 256;
    int cs = 0;
};
GemmPlan plan_gemm(const GemmDesc& d, int sms);

// Shard reduce.
struct ReduceDesc {
    int t = 0;
    int64_t count = 0;
    int in_bf16 = 1;
    const void* p[TP_MAX_SHARDS] = {};
    void* out = nullptr;
    int out_bf16 = 1;
    int ring = 0;
    int hop_bf16 = 0;
    int replicate = 0;
    int pdl = 0;                         // 1: may start before the previous kernel of the call ends
};
tp_status launch_shard_reduce(const ReduceDesc& d, cudaStream_t stream);

// Vocab-parallel embedding.
struct EmbedDesc {
    int t = 0;
    int64_t vocab = 0, h = 0, n = 0, per = 0;
    const int32_t* ids = nullptr;
    const void* table[TP_MAX_SHARDS] = {};
    int bf16 = 1;
    void* out = nullptr;
    void* partials[TP_MAX_SHARDS] = {};
    int with_partials = 0;
};
tp_status launch_vocab_embed(const EmbedDesc& d, cudaStream_t stream);

// Concatenation of t [rows, cols_r] shards along columns.
struct GatherDesc {
    int t = 0;
    int64_t rows = 0;
    int64_t cols[TP_MAX_SHARDS] = {};
    int elem_bytes = 2;
    const void* shards[TP_MAX_SHARDS] = {};
    void* out = nullptr;
};
tp_status launch_shard_gather(const GatherDesc& d, cudaStream_t stream);

// Reduce-scatter over token rows + residual add + RMSNorm (sequence parallelism).
struct SeqParDesc {
    int t = 0;
    int64_t n = 0, h = 0;
    int in_bf16 = 1;
    const void* p[TP_MAX_SHARDS] = {};
    const void* residual = nullptr;
    const void* weight = nullptr;
    void* residual_out = nullptr;
    void* out = nullptr;
    float eps = 1e-6f;
    int ring = 0;
};
tp_status launch_seqpar_rmsnorm(const SeqParDesc& d, cudaStream_t stream);

tp_status launch_expire_wait(uint64_t limit_ns, int* status, cudaStream_t stream);

}  // namespace tpk
