/*
 * tp.h - C ABI of the GB300 (sm_103a) tensor-parallel layer library.
 *
 * The library runs the Megatron-style tensor-parallel layers of an LLM
 * serving stack on ONE GPU: the t ranks of a tensor-parallel group are
 * simulated as t shards whose weights and partial results all live in this
 * GPU's memory, and the collectives (all-reduce, all-gather) become kernels
 * over those in-memory shards.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named x, w, y, bias, table, partials, out, logits, workspace
 *    are DEVICE pointers owned by the caller.  Arguments typed
 *    `const void* const*` / `void* const*` are HOST arrays of t device
 *    pointers (one per shard).  The library never allocates, frees or keeps
 *    a caller buffer.
 *  - Matrices are row-major; `ld*` arguments are row strides in ELEMENTS.
 *    Weights are stored [out, in], so a linear layer computes x @ w^T
 *    (page "Nano-vLLM walkthrough 22: tensor parallelism (2), code", §2).
 *  - Every call validates its arguments on the host first.  A rejected
 *    call returns an error status and launches nothing.  Valid calls enqueue
 *    kernels on `stream` and return TP_OK without waiting; a failed launch
 *    returns TP_ERR_CUDA.  Errors that happen later on the device (a
 *    bounded wait that expired) are reported by tp_device_status().
 *  - Alignment: every device pointer and the row stride in bytes of every
 *    GEMM input (x, w, table) must be a multiple of 16 bytes (TMA tiles and
 *    128-bit loads), else TP_ERR_ALIGNMENT.  GEMM outputs only need a row
 *    stride at least their width (TP_ERR_INVALID_ARG otherwise); rows whose
 *    16-byte chunks are not aligned are written element by element.
 *    Shard counts must be in 1..TP_MAX_SHARDS, else TP_ERR_INVALID_ARG.  Splits that do not divide evenly return
 *    TP_ERR_NOT_DIVISIBLE (the `divide` assertion of the same page, §1).
 *  - GEMM operands (x, w) are bfloat16; accumulation is float32.
 *  - Stream order is kept as the caller sees it.  The GEMM, shard-reduce,
 *    gather and reduce-scatter kernels are launched with programmatic stream
 *    serialization: one may be scheduled while the previous kernel of the
 *    stream is still draining, but it reads nothing, and so writes nothing,
 *    before that kernel has finished and its writes are visible.  A caller's
 *    kernel that follows a library call starts after the call's last kernel
 *    unless the caller opts into the same mechanism.  Launches of this kind
 *    are captured into CUDA graphs like any other.
 *  - Nothing here is thread-safe against concurrent calls that share output
 *    buffers; calls on different streams with disjoint buffers are fine.
 *  - Zero tokens (n = 0, or count / rows = 0) is a valid call: every other
 *    argument is checked as usual, the pointers to data of zero rows (x, y,
 *    partials, out, logits, shard_logits, ids, residual, the host buffers)
 *    may be NULL, and the call returns TP_OK without any CUDA call.
 */
#ifndef TP_GB300_H
#define TP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TP_ABI_VERSION 1
#define TP_MAX_SHARDS 8

typedef enum {
    TP_OK = 0,
    TP_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum, t out of range */
    TP_ERR_NOT_DIVISIBLE = 2, /* a split that does not divide by t */
    TP_ERR_ALIGNMENT = 3,     /* pointer or row stride not 16-byte aligned */
    TP_ERR_UNSUPPORTED = 4,   /* dtype or option combination not provided */
    TP_ERR_CUDA = 5,          /* a CUDA runtime or driver call failed */
    TP_ERR_TIMEOUT = 6,       /* a bounded device-side wait expired */
    TP_ERR_WORKSPACE = 7      /* workspace missing or too small */
} tp_status;

typedef enum { TP_BF16 = 0, TP_F32 = 1 } tp_dtype;

/* How the t partial sums are reduced ("all-reduce sum").
 * DIRECT: one-shot sum in rank order, float32 carry (page "vLLM source
 *         analysis 13: tensor parallelism in detail", low-latency
 *         all-reduce pseudocode after §1.2).
 * RING:   the reduce-scatter + all-gather ring of the same page, §1.1.1 and
 *         §1.1.2: the buffer is cut into t chunks of ceil(K/t) elements and
 *         chunk c is folded in the order c, c+1, ..., c+t-1 (mod t), each
 *         addition rounded to the hop dtype.
 * FUSED:  (row GEMMs only) the shards are accumulated into one float32
 *         accumulator in rank order inside the down-projection GEMM; no
 *         partial is written. */
typedef enum { TP_REDUCE_DIRECT = 0, TP_REDUCE_RING = 1, TP_REDUCE_FUSED = 2 } tp_reduce_mode;

/* Activation fused into the column GEMM epilogue.  With a gated activation
 * each shard's weight is its merged gate_up block [gate rows; up rows] and
 * the output is act(x gate^T) * (x up^T) (page "Tensor parallelism from
 * scratch", tp.py TPMLP; SiLU is x / (1 + exp(-x)); GeLU-tanh as defined in
 * "vLLM source analysis 13", §2.2.2). */
typedef enum { TP_ACT_NONE = 0, TP_ACT_SILU_MUL = 1, TP_ACT_GELU_TANH_MUL = 2 } tp_act;

/* A cudaStream_t.  NULL is the legacy default stream. */
typedef struct CUstream_st* tp_stream;

/* Human-readable name of a status code (static string, never NULL). */
const char* tp_status_string(tp_status s);

/* TP_ABI_VERSION of the loaded library. */
int tp_abi_version(void);

/*
 * ColumnParallelLinear: the weight is cut on its output dimension and every
 * shard sees the full input (page "Nano-vLLM walkthrough 22", §3
 * ColumnParallelLinear; page "6.2 Tensor-parallel inference", §1; for the
 * merged gate_up block, the same page §5 "double cut").
 *
 *   x      [n, in] bf16, row stride ldx (same input for every shard).
 *   w[r]   act == TP_ACT_NONE: [out_full/t, in] bf16, row stride ldw.
 *          gated act: [2*out_full/t, in] bf16 = rank r's gate rows followed
 *          by rank r's up rows, row stride ldw.
 *   bias   NULL, or a host array of t device pointers to [out_full/t] bf16
 *          (only with TP_ACT_NONE; else TP_ERR_UNSUPPORTED).
 *   gather_output == 0: y[r] is [n, out_full/t] with row stride ldy.
 *   gather_output == 1: y[0] is [n, out_full] with row stride ldy and shard
 *          r writes columns [r*out_full/t, (r+1)*out_full/t) (the all-gather
 *          becomes a zero-copy concatenation).
 *   y_dtype TP_BF16 or TP_F32.
 * Requires out_full % t == 0 and in % 8 == 0 (TMA row pitch).
 */
tp_status tp_linear_col(int t, int64_t n, int64_t in, int64_t out_full,
                        const void* x, int64_t ldx,
                        const void* const* w, int64_t ldw,
                        const void* const* bias, tp_act act,
                        int gather_output, void* const* y, int64_t ldy,
                        tp_dtype y_dtype, tp_stream stream);

/*
 * RowParallelLinear: the weight is cut on its input dimension, the input is
 * cut to match, every shard produces a full [n, out] partial sum, the bias
 * is added by rank 0 only, and the partials are all-reduced (page
 * "Nano-vLLM walkthrough 22", §4 RowParallelLinear; page "Mini-SGLang
 * source reading: TP", §3).
 *
 *   x[r]   [n, in_full/t] bf16, row stride ldx.
 *   w[r]   [out, in_full/t] bf16, row stride ldw (ldw = in_full when the
 *          shards are column views of one [out, in_full] matrix).
 *   bias   NULL or [out] bf16, added once (rank 0's partial).
 *   reduce_results == 0: only the partials are written (mode must not be
 *          FUSED); y is ignored.
 *   reduce_results == 1: y [n, out] (row stride ldy, y_dtype) receives the
 *          sum.  DIRECT/RING write the partials first, then reduce them
 *          (RING hops round to partial_dtype); FUSED writes no partial
 *          (partials may be NULL).  A FUSED call of more than 128 rows that
 *          is given a contiguous partials[0] (ldp == out; n * out elements
 *          of partial_dtype, at least 32 MiB + 4 KiB) uses that buffer as
 *          scratch in which the last, partial wave of output tiles is split
 *          along K (stream-K); its contents are overwritten.
 *   partials[r] [n, out] in partial_dtype, row stride ldp (caller-owned
 *          scratch; contents are overwritten).
 * Requires in_full % t == 0 and (in_full/t) % 8 == 0.
 */
tp_status tp_linear_row(int t, int64_t n, int64_t in_full, int64_t out,
                        const void* const* x, int64_t ldx,
                        const void* const* w, int64_t ldw,
                        const void* bias, int reduce_results, tp_reduce_mode mode,
                        tp_dtype partial_dtype, void* const* partials, int64_t ldp,
                        void* y, int64_t ldy, tp_dtype y_dtype, tp_stream stream);

/*
 * The all-reduce (sum) of t partial buffers of `count` elements each (page
 * "vLLM source analysis 13", §1.1 ring all-reduce and the low-latency
 * one-shot sum after §1.2).
 *
 *   partials[r] `count` elements of `dtype` (bf16 or f32), contiguous.
 *   mode       TP_REDUCE_DIRECT: rank-order sum with a float32 carry.
 *              TP_REDUCE_RING: chunk c = [c*ceil(count/t), ...) folded in
 *              the order c, c+1, ... (mod t); every addition is rounded to
 *              hop_dtype (TP_F32 = float32 carry; TP_BF16 = a bf16 wire,
 *              only with bf16 partials).
 *   out        NULL or `count` elements of out_dtype; receives the sum,
 *              rounded once from the carry.
 *   replicate  1: the sum (in dtype) is also written back into every
 *              partials[r], which is what an all-reduce leaves on each rank.
 * At least one of out / replicate must be given.  Bytes moved:
 * t*count*sizeof(dtype) read, plus the writes requested.
 */
tp_status tp_shard_reduce(int t, int64_t count, tp_dtype dtype, const void* const* partials,
                          void* out, tp_dtype out_dtype, tp_reduce_mode mode,
                          tp_dtype hop_dtype, int replicate, tp_stream stream);

/*
 * Workspace bytes for tp_mlp_forward: the intermediate H [n, f] bf16 (rank
 * r's slice is columns [r*f/t, (r+1)*f/t)) plus, unless mode is FUSED, t
 * partials [n, h] of partial_dtype, each 256-byte aligned.  For a FUSED
 * reduce of more than 128 token rows it adds 32 MiB + 4 KiB in which the
 * down GEMM splits the tiles of its last, partial wave along K (stream-K):
 * tp_mlp_forward also runs with only the H bytes, then without that split.
 * For a FUSED reduce of 1 to 8 token rows with h a multiple of 256 up to
 * 1024, (f/t) % 64 == 0 and f/64 <= 128, it returns instead the larger of
 * that and f/64 * n * h * 4 bytes (256-byte aligned): with that many bytes
 * tp_mlp_forward runs both projections in one GEMM kernel whose CTA pairs
 * each take a 64-column slice of a rank's f columns (H never leaves the
 * chip), and a second kernel adds the slices' fp32 partials in slice order,
 * rank 0's slices first; with only the H bytes it runs the two-GEMM path.
 * Returns 0 for invalid arguments.
 */
size_t tp_mlp_workspace_size(int t, int64_t n, int64_t h, int64_t f,
                             tp_reduce_mode mode, tp_dtype partial_dtype);

/*
 * The tensor-parallel MLP block, Y = sum_r act(X A_r) B_r (page "6.2
 * Tensor-parallel inference", §1; page "Tensor parallelism from scratch",
 * tp.py TPMLP): a gated column-parallel GEMM per shard with the activation
 * fused into its epilogue, then the row-parallel down projection and the
 * reduce selected by `mode`.
 *
 *   x            [n, h] bf16, row stride ldx.
 *   w_gate_up[r] [2f/t, h] bf16 contiguous: rank r's gate rows, then its
 *                up rows (the merged double cut).
 *   w_down[r]    [h, f/t] bf16, row stride ld_down.
 *   bias_down    NULL or [h] bf16, added once.
 *   act          TP_ACT_SILU_MUL or TP_ACT_GELU_TANH_MUL.
 *   workspace    device buffer of tp_mlp_workspace_size() bytes (a FUSED
 *                reduce also accepts just the n*f*2 bytes of H, see above),
 *                256-byte aligned; overwritten.
 *   y            [n, h] of y_dtype, contiguous.
 * Requires f % t == 0, (f/t) % 8 == 0 and h % 8 == 0.
 */
tp_status tp_mlp_forward(int t, int64_t n, int64_t h, int64_t f,
                         const void* x, int64_t ldx,
                         const void* const* w_gate_up,
                         const void* const* w_down, int64_t ld_down,
                         const void* bias_down, tp_act act,
                         tp_reduce_mode mode, tp_dtype partial_dtype,
                         void* workspace, size_t workspace_bytes,
                         void* y, tp_dtype y_dtype, tp_stream stream);

/*
 * tp_mlp_forward for activations in host memory, with the copies overlapped
 * with the compute (page "6.2 Tensor-parallel inference", §1: every token's
 * output depends on its own row of X only, so the tokens can be processed
 * in row blocks).
 *
 *   x_host   [n, h] bf16, contiguous, page-locked host memory (read).
 *   y_host   [n, h] of y_dtype, contiguous, page-locked host memory (written).
 *   x_dev    device staging for X, [n, h] bf16; y_dev device [n, h] y_dtype.
 *   workspace  at least tp_mlp_workspace_size(t, m, h, f, mode, partial_dtype)
 *              bytes, m the tallest row block (tp_mlp_host_blocks), 256-byte
 *              aligned.
 *   chunks   1..64: 1 runs all rows as one block.  With chunks >= 2 the first
 *            and the last block have e = ceil(n / (4 chunks)) rows (rounded up
 *            to a multiple of 128 when at least e rows stay between them), and
 *            the n - 2e rows between them form chunks - 1 blocks of equal
 *            height (rounded up to a multiple of 128 where the last of them
 *            keeps rows; that one takes the rest).  n = 8192 in 2 chunks runs
 *            as 1024, 6144, 1024 rows; in 4 chunks as 512, 2432, 2432, 2304,
 *            512.  The exposed first copy and last read-back are the short
 *            edge blocks'.  Block i's host->device copy runs on copy_stream
 *            under the compute of block i-1, its device->host copy under the
 *            compute of block i+1; the MLPs run on `stream`.
 *   Other arguments as tp_mlp_forward.  When the call returns, all work is
 *   queued and `stream` completes after the last read-back (wait on it).
 * Errors as tp_mlp_forward; TP_ERR_WORKSPACE if the workspace is too small
 * for the tallest block.
 */
tp_status tp_mlp_forward_host(int t, int64_t n, int64_t h, int64_t f,
                              const void* x_host,
                              const void* const* w_gate_up,
                              const void* const* w_down, int64_t ld_down,
                              const void* bias_down, tp_act act,
                              tp_reduce_mode mode, tp_dtype partial_dtype,
                              void* x_dev, void* workspace, size_t workspace_bytes,
                              void* y_dev, void* y_host, tp_dtype y_dtype,
                              int chunks, tp_stream stream, tp_stream copy_stream);

/*
 * The row blocks tp_mlp_forward_host cuts n tokens into with `chunks` (host
 * logic only, no CUDA call).  Returns the block count k (0 for n = 0), or -1
 * if n < 0 or chunks is outside 1..64.  starts is NULL or a host array of
 * max_blocks + 1 entries; when it is not NULL and max_blocks >= k, the call
 * writes the k + 1 boundaries: block b covers rows [starts[b], starts[b + 1]),
 * starts[0] = 0, starts[k] = n.  Otherwise it writes nothing (call with NULL
 * first to learn k; k <= chunks + 1).
 */
int tp_mlp_host_blocks(int64_t n, int chunks, int64_t* starts, int max_blocks);

/*
 * tp_mlp_forward for callers that cannot allocate device memory.  This entry
 * point has no counterpart in the pages this library follows; it exists for
 * deployment reasons.
 *
 * Who needs it: a host application that loads this library as a plugin and
 * owns the whole device memory pool (and so forbids its plugins to call
 * cudaMalloc), or a latency-critical decode loop that must not call
 * cudaMalloc/cudaFree because they can synchronise the device and stall every
 * stream.  Such a caller cannot provide tp_mlp_forward's workspace.
 *
 * What it does: exactly tp_mlp_forward (same arguments minus the workspace,
 * same kernels, same results), with the workspace taken from a scratch array
 * of TP_STATIC_SCRATCH_BYTES that is part of the library's device image.
 * It allocates nothing and calls no allocating routine.  The caller still
 * passes and owns x, the weights, the bias and y.
 *
 * Limit: the workspace tp_mlp_forward requires (tp_mlp_workspace_size(t, n,
 * h, f, mode, partial_dtype), less the optional stream-K area of a FUSED
 * reduce of more than 128 rows) must not exceed TP_STATIC_SCRATCH_BYTES
 * (16 MiB), else TP_ERR_WORKSPACE and nothing is launched.  Example: 64
 * tokens of an h=8192, f=28672 MLP at t=4 need 12.1 MB with fp32 partials;
 * a fused reduce needs only the n*f*2 bytes of H.
 *
 * Costs and rules:
 *  - The 16 MiB belong to the library's device image, which CUDA loads
 *    lazily: a GPU reserves them when the module is first loaded there, at
 *    the latest in this entry point's first call on that device, and holds
 *    them until the process exits.
 *  - That first call on each device loads the module if needed and looks up
 *    the array's device address (cudaGetSymbolAddress), caching it.  Loading
 *    can synchronise the device and fails with TP_ERR_CUDA when the device
 *    has no 16 MiB left, so make the first call at start-up, outside any
 *    latency-critical loop and before any stream capture on that device.
 *  - All calls in the process share the one array per device and it keeps
 *    the previous call's contents.  Nothing in it needs to start at zero:
 *    each call writes every byte it later reads.  Calls that can overlap on
 *    the GPU (unordered streams, concurrent host threads) race on the array:
 *    order them on one stream.
 */
#define TP_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
tp_status tp_mlp_forward_static(int t, int64_t n, int64_t h, int64_t f,
                                const void* x, int64_t ldx,
                                const void* const* w_gate_up,
                                const void* const* w_down, int64_t ld_down,
                                const void* bias_down, tp_act act,
                                tp_reduce_mode mode, tp_dtype partial_dtype,
                                void* y, tp_dtype y_dtype, tp_stream stream);

/*
 * VocabParallelEmbedding (page "Tensor parallelism from scratch", tp.py
 * VocabParallelEmbedding; page "vLLM source analysis 13", §2.4.1): rank r
 * owns token ids [r*per, min((r+1)*per, vocab)) with per = ceil(vocab/t).
 * Its output for an id outside that range (including negative ids and ids
 * >= vocab) is exactly 0; the t outputs are summed in rank order.
 *
 *   ids        [n] int32.
 *   table[r]   [rows_r, h] of dtype (bf16 or f32), contiguous, rows_r the
 *              size of rank r's range (may be NULL when rows_r == 0).
 *   out        [n, h] of dtype.
 *   partials   NULL, or t device pointers to [n, h] buffers that also
 *              receive each rank's masked lookup (its pre-all-reduce view).
 * Out-of-range ids are not an error.  The result is bit-exact: each output
 * element is one table value plus exact zeros.  h * sizeof(dtype) must be a
 * multiple of 16 (TP_ERR_ALIGNMENT); h <= 2^31 - 1 and n <= 4 (2^31 - 1)
 * (TP_ERR_INVALID_ARG).
 */
tp_status vocab_parallel_embed(int t, int64_t vocab, int64_t h, const int32_t* ids, int64_t n,
                               const void* const* table, tp_dtype dtype, void* out,
                               void* const* partials, tp_stream stream);

/*
 * Vocab-sharded LM head (page "vLLM source analysis 13", §2.4.2; page
 * "Tensor parallelism from scratch", tp.py TPTransformer): rank r computes
 * logits_r = x table_r^T over its vocab range (same ranges as
 * vocab_parallel_embed) and the parts are concatenated on the vocab axis.
 *
 *   x          [n, h] bf16, row stride ldx.
 *   table[r]   [rows_r, h] bf16 contiguous.
 *   logits     [n, vocab] of out_dtype with row stride ldl: rank r writes
 *              columns [start_r, end_r) directly (zero-copy all-gather); or
 *              NULL, in which case shard_logits[r] ([n, rows_r], contiguous)
 *              receive the per-rank logits (gather them with
 *              tp_shard_gather).
 * Requires h % 8 == 0.
 */
tp_status lm_head_sharded(int t, int64_t n, int64_t h, int64_t vocab,
                          const void* x, int64_t ldx, const void* const* table,
                          void* logits, int64_t ldl, void* const* shard_logits,
                          tp_dtype out_dtype, tp_stream stream);

/*
 * Sequence parallelism: the all-reduce after a row-parallel layer split into
 * a reduce-scatter over token rows and an all-gather, with the residual add
 * and RMSNorm done between them on each rank's own rows (page "Tensor
 * parallelism from scratch", exercise 1: the total communication is
 * unchanged, the per-token work drops to 1/t per rank; the pre-norm residual
 * x = x + block(norm(x)) of its tp.py).  RMSNorm is
 * x / sqrt(mean(x^2) + eps) * weight (the pages name it without a formula).
 *
 *   partials[r]  [n, h] of dtype (bf16 or f32), contiguous: the row-parallel
 *                partial sums.
 *   residual     NULL or [n, h] bf16: the residual stream.
 *   weight       [h] bf16: the RMSNorm weight (one copy on every rank).
 *   mode         TP_REDUCE_DIRECT: a rank sums its rows of the t partials in
 *                rank order; TP_REDUCE_RING: in the order of a reduce-scatter
 *                ring that leaves chunk r on rank r (r+1, r+2, ..., r mod t).
 *                fp32 carry in both.
 *   residual_out NULL or [n, h] bf16: residual + sum, rounded once; may be
 *                the same buffer as residual.
 *   out          [n, h] bf16: RMSNorm of the fp32 residual + sum.
 * Rank r owns rows [r*ceil(n/t), min((r+1)*ceil(n/t), n)); every rank's rows
 * are written in place, so the all-gather back to all tokens costs nothing.
 * Requires h % 8 == 0 (TP_ERR_ALIGNMENT) and h <= 32768 (TP_ERR_UNSUPPORTED).
 */
tp_status tp_reduce_scatter_rmsnorm(int t, int64_t n, int64_t h, tp_dtype dtype,
                                    const void* const* partials, const void* residual,
                                    const void* weight, float eps, tp_reduce_mode mode,
                                    void* residual_out, void* out, tp_stream stream);

/*
 * All-gather of vocab-sharded outputs: shard r is [rows, cols[r]]
 * (contiguous) and lands in columns [sum(cols[:r]), sum(cols[:r+1])) of
 * out [rows, sum(cols)] (contiguous).  `cols` is a host array of t widths.
 * Shards of width 0 may be NULL.
 */
tp_status tp_shard_gather(int t, int64_t rows, const int64_t* cols, tp_dtype dtype,
                          const void* const* shards, void* out, tp_stream stream);

/*
 * Synchronises `stream`, then returns and clears the library's device
 * status word: TP_ERR_TIMEOUT if a bounded device-side wait of an earlier
 * kernel expired, TP_ERR_CUDA if the stream reported an error, else TP_OK.
 */
tp_status tp_device_status(tp_stream stream);

/*
 * Number of collective launches (shard reduces, fused-reduce GEMMs and
 * gathers) issued since load or the last reset.  A debugging counter in the
 * spirit of the all-reduce counter of page "Tensor parallelism from
 * scratch", tp.py.
 */
uint64_t tp_collective_count(void);
void tp_reset_collective_count(void);

/*
 * Width of the GEMM output tile (the tcgen05 MMA N: 64, 96, 128 or 256) used
 * by every later GEMM launch of this process; 0 restores the automatic choice
 * (a cost model over whole waves of tiles).  96 applies to GEMMs without the
 * gated epilogue (a gated GEMM given 96 uses 128).  For tests and tuning.
 * Returns TP_ERR_INVALID_ARG for any other value.
 */
tp_status tp_set_gemm_tile_n(int n);

/*
 * Use of the CTA-pair GEMM kernel (256 x 256 tiles computed by two CTAs on
 * neighbouring SMs with tcgen05 cta_group::2) for later launches: 1 = always,
 * -1 = never, 0 = automatic (pairs when a GEMM has at least 512 rows and two
 * full waves of pair tiles).  For tests and tuning.  TP_ERR_INVALID_ARG for
 * other values.
 */
tp_status tp_set_gemm_cta_pair(int mode);

/*
 * Use of the split-K kernel for the fused reduce (TP_REDUCE_FUSED) at decode
 * sizes (at most 64 token rows): a cluster of CTAs shares each output tile,
 * each CTA accumulating whole shards, and the CTAs add their fp32
 * accumulators in rank order through distributed shared memory.  mode 0 =
 * automatic (when the output has fewer 256-wide tiles than the GPU has SMs),
 * -1 = never, 1 = whenever the shape allows it (at most 64 rows, at least two
 * shards).  max_clusters > 0 caps the clusters resident at once, so that each
 * cluster walks several tiles; 0 = as many as fit.  For tests and tuning.
 * TP_ERR_INVALID_ARG for other values.
 */
tp_status tp_set_gemm_split(int mode, int max_clusters);

/*
 * Test hook for the failure path: launches one thread block that waits, with
 * the library's bounded wait, on a shared-memory barrier that nothing ever
 * signals.  The wait gives up after `limit_ns` nanoseconds (capped at 1 s)
 * and records TP_ERR_TIMEOUT in the status word, which tp_device_status()
 * then returns.  The kernel always exits normally.
 */
tp_status tp_debug_expire_wait(uint64_t limit_ns, tp_stream stream);

/*
 * Test hook for the host-side kernel choice (no CUDA call): the GEMM kernel
 * the library would launch, with the automatic settings, for M rows, an
 * output of N columns per group (per shard), K per segment, `groups`
 * independent outputs or `segs` K segments summed into one (the fused
 * reduce; not both), a gated epilogue or not, on a GPU with `sms` SMs.
 * Writes kind (0: single-CTA tiles, 1: CTA pairs, 2: split-K clusters), the
 * output tile width (the MMA N) and the cluster size (split-K only, else 0).
 * TP_ERR_INVALID_ARG for sizes or counts out of range or null outputs.
 */
tp_status tp_debug_gemm_plan(int64_t m, int64_t n, int64_t k, int groups, int segs, int gated, int sms,
                             int* kind, int* tile_n, int* cluster);

#ifdef __cplusplus
}
#endif

#endif /* TP_GB300_H */
