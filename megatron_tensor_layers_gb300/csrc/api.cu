// C ABI of the tensor-parallel layer library: argument validation, shard
// layout (which buffer and which slice each simulated rank uses), workspace
// carving, and the kernel launches.  See include/tp.h for the contract.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "tp.h"

// The one piece of global device state: the status word that bounded waits
// write TP_ERR_TIMEOUT into.
__device__ int g_tp_status = 0;

namespace {

std::atomic<uint64_t> g_collectives{0};
std::atomic<int> g_tile_n{0};
std::atomic<int> g_pair{0};
std::atomic<int> g_split{0};
std::atomic<int> g_split_clusters{0};

// The GEMM tuning knobs in effect for a launch.
void apply_knobs(tpk::GemmDesc& d) {
    d.force_bn = g_tile_n.load();
    d.pair = g_pair.load();
    d.split = g_split.load();
    d.split_clusters = g_split_clusters.load();
}

// Device address of the status word on the current device, looked up once per
// device and cached.  Host threads may race on a device's first lookup: both
// store the same address, and the relaxed atomics make that race benign.
int* status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    static std::atomic<int*> cache[64];
    int* cached = cache[dev].load(std::memory_order_relaxed);
    if (cached == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tp_status) != cudaSuccess) return nullptr;
        cached = static_cast<int*>(p);
        cache[dev].store(cached, std::memory_order_relaxed);
    }
    return cached;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int esize(tp_dtype d) { return d == TP_F32 ? 4 : 2; }
inline bool dtype_ok(int d) { return d == TP_BF16 || d == TP_F32; }
inline bool ld_ok(int64_t ld, int64_t minimum, int elem) { return ld >= minimum && (ld * elem) % 16 == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline cudaStream_t cs(tp_stream s) { return reinterpret_cast<cudaStream_t>(s); }

#define TP_CHECK(cond, code) \
    do {                     \
        if (!(cond)) return (code); \
    } while (0)

}  // namespace

// tp_mlp_forward's workspace: H [n, f] bf16, then (unless the reduce is
// fused) t partials [n, h]; that much is required.  A fused reduce of more
// than 128 rows (CTA-pair tiles) may also use the stream-K tail area of its
// down GEMM, which tp_mlp_workspace_size includes.
size_t tpk::mlp_workspace_required(int t, int64_t n, int64_t h, int64_t f, tp_reduce_mode mode, tp_dtype partial_dtype) {
    if (t < 1 || t > TP_MAX_SHARDS || n < 0 || h <= 0 || f <= 0 || !dtype_ok(partial_dtype)) return 0;
    if (mode != TP_REDUCE_DIRECT && mode != TP_REDUCE_RING && mode != TP_REDUCE_FUSED) return 0;
    size_t bytes = align256(static_cast<size_t>(n) * static_cast<size_t>(f) * 2);
    if (mode != TP_REDUCE_FUSED)
        bytes += static_cast<size_t>(t) * align256(static_cast<size_t>(n) * static_cast<size_t>(h) * esize(partial_dtype));
    return bytes;
}

static size_t mlp_tail_bytes(int64_t n, tp_reduce_mode mode) {
    return (mode == TP_REDUCE_FUSED && n > 128) ? tpk::kSkWorkspaceBytes : 0;
}

extern "C" {

const char* tp_status_string(tp_status s) {
    switch (s) {
        case TP_OK: return "TP_OK";
        case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG";
        case TP_ERR_NOT_DIVISIBLE: return "TP_ERR_NOT_DIVISIBLE";
        case TP_ERR_ALIGNMENT: return "TP_ERR_ALIGNMENT";
        case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
        case TP_ERR_CUDA: return "TP_ERR_CUDA";
        case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
        case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE";
    }
    return "TP_ERR_UNKNOWN";
}

int tp_abi_version(void) { return TP_ABI_VERSION; }

uint64_t tp_collective_count(void) { return g_collectives.load(); }
void tp_reset_collective_count(void) { g_collectives.store(0); }

tp_status tp_linear_col(int t, int64_t n, int64_t in, int64_t out_full, const void* x, int64_t ldx,
                        const void* const* w, int64_t ldw, const void* const* bias, tp_act act, int gather_output,
                        void* const* y, int64_t ldy, tp_dtype y_dtype, tp_stream stream) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(n >= 0 && in > 0 && out_full > 0, TP_ERR_INVALID_ARG);
    TP_CHECK(n <= INT32_MAX && out_full <= INT32_MAX && in <= INT32_MAX, TP_ERR_INVALID_ARG);
    TP_CHECK((x != nullptr || n == 0) && w != nullptr && y != nullptr, TP_ERR_INVALID_ARG);
    TP_CHECK(act == TP_ACT_NONE || act == TP_ACT_SILU_MUL || act == TP_ACT_GELU_TANH_MUL, TP_ERR_INVALID_ARG);
    TP_CHECK(gather_output == 0 || gather_output == 1, TP_ERR_INVALID_ARG);
    TP_CHECK(dtype_ok(y_dtype), TP_ERR_UNSUPPORTED);
    TP_CHECK(out_full % t == 0, TP_ERR_NOT_DIVISIBLE);
    const int64_t os = out_full / t;
    const bool glu = act != TP_ACT_NONE;
    TP_CHECK(!(glu && bias != nullptr), TP_ERR_UNSUPPORTED);
    TP_CHECK(in % 8 == 0, TP_ERR_ALIGNMENT);
    TP_CHECK(al16(x) && ld_ok(ldx, in, 2) && ld_ok(ldw, in, 2), TP_ERR_ALIGNMENT);
    const int ey = esize(y_dtype);
    TP_CHECK(ldy >= (gather_output ? out_full : os), TP_ERR_INVALID_ARG);
    for (int r = 0; r < t; ++r) {
        TP_CHECK(w[r] != nullptr, TP_ERR_INVALID_ARG);
        TP_CHECK(al16(w[r]), TP_ERR_ALIGNMENT);
        if (bias != nullptr) TP_CHECK(bias[r] != nullptr, TP_ERR_INVALID_ARG);
        if (!gather_output || r == 0) {
            TP_CHECK(y[r] != nullptr || n == 0, TP_ERR_INVALID_ARG);
            TP_CHECK(al16(y[r]), TP_ERR_ALIGNMENT);
        }
    }
    if (n == 0) return TP_OK;
    tpk::GemmDesc d;
    d.M = n;
    d.N = os;
    d.K = in;
    d.groups = t;
    d.a[0] = x;
    d.lda = ldx;
    d.ldb = ldw;
    d.b_rows = glu ? 2 * os : os;
    d.glu = glu ? 1 : 0;
    d.glu_up_row = os;
    d.act = act;
    d.ldo = ldy;
    d.out_f32 = y_dtype == TP_F32;
    d.status = status_ptr();
    d.pdl = 2;                       // may overlap the previous kernel's tail; loads wait for it
    apply_knobs(d);
    for (int r = 0; r < t; ++r) {
        d.b[r] = w[r];
        d.out[r] = gather_output ? static_cast<void*>(static_cast<char*>(y[0]) + r * os * ey) : y[r];
        d.bias[r] = bias ? bias[r] : nullptr;
    }
    if (gather_output) g_collectives++;
    return tpk::launch_gemm(d, cs(stream));
}

// pdl = 1: the reduce may start before the previous kernel of the stream ends
// (programmatic dependent launch); every thread waits for that kernel before
// its first load.
static tp_status shard_reduce_impl(int t, int64_t count, tp_dtype dtype, const void* const* partials, void* out,
                                   tp_dtype out_dtype, tp_reduce_mode mode, tp_dtype hop_dtype, int replicate,
                                   int pdl, tp_stream stream) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(count >= 0 && partials != nullptr, TP_ERR_INVALID_ARG);
    TP_CHECK(mode == TP_REDUCE_DIRECT || mode == TP_REDUCE_RING, TP_ERR_INVALID_ARG);
    TP_CHECK(replicate == 0 || replicate == 1, TP_ERR_INVALID_ARG);
    TP_CHECK(out != nullptr || replicate || count == 0, TP_ERR_INVALID_ARG);
    TP_CHECK(dtype_ok(dtype) && dtype_ok(hop_dtype), TP_ERR_UNSUPPORTED);
    TP_CHECK(out == nullptr || dtype_ok(out_dtype), TP_ERR_UNSUPPORTED);
    TP_CHECK(!(hop_dtype == TP_BF16 && dtype != TP_BF16), TP_ERR_UNSUPPORTED);
    for (int r = 0; r < t; ++r) {
        TP_CHECK(partials[r] != nullptr || count == 0, TP_ERR_INVALID_ARG);
        TP_CHECK(al16(partials[r]), TP_ERR_ALIGNMENT);
    }
    TP_CHECK(out == nullptr || al16(out), TP_ERR_ALIGNMENT);
    if (count == 0) return TP_OK;
    tpk::ReduceDesc d;
    d.t = t;
    d.count = count;
    d.in_bf16 = dtype == TP_BF16;
    for (int r = 0; r < t; ++r) d.p[r] = partials[r];
    d.out = out;
    d.out_bf16 = out_dtype == TP_BF16;
    d.ring = mode == TP_REDUCE_RING;
    d.hop_bf16 = (mode == TP_REDUCE_RING && hop_dtype == TP_BF16) ? 1 : 0;
    d.replicate = replicate;
    d.pdl = pdl;
    g_collectives++;
    return tpk::launch_shard_reduce(d, cs(stream));
}

tp_status tp_shard_reduce(int t, int64_t count, tp_dtype dtype, const void* const* partials, void* out,
                          tp_dtype out_dtype, tp_reduce_mode mode, tp_dtype hop_dtype, int replicate,
                          tp_stream stream) {
    return shard_reduce_impl(t, count, dtype, partials, out, out_dtype, mode, hop_dtype, replicate, 1, stream);
}

// pdl_first = 1: the previous launch of the stream is a kernel of the same
// call that wrote x (tp_mlp_forward's gate_up GEMM), so the GEMM (split-K or
// single-CTA) may load its first ring of weights before waiting for it; 0: the
// first kernel of the call, which loads nothing before that wait.  Every
// launch may start early.
// sk_ws / sk_bytes: the stream-K tail area of a fused reduce (flags already
// zeroed in stream order), or null.
static tp_status linear_row_impl(int t, int64_t n, int64_t in_full, int64_t out, const void* const* x, int64_t ldx,
                                 const void* const* w, int64_t ldw, const void* bias, int reduce_results,
                                 tp_reduce_mode mode, tp_dtype partial_dtype, void* const* partials, int64_t ldp,
                                 void* y, int64_t ldy, tp_dtype y_dtype, int pdl_first, tp_stream stream,
                                 void* sk_ws = nullptr, size_t sk_bytes = 0) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(n >= 0 && in_full > 0 && out > 0, TP_ERR_INVALID_ARG);
    TP_CHECK(n <= INT32_MAX && out <= INT32_MAX && in_full <= INT32_MAX, TP_ERR_INVALID_ARG);
    TP_CHECK(x != nullptr && w != nullptr, TP_ERR_INVALID_ARG);
    TP_CHECK(reduce_results == 0 || reduce_results == 1, TP_ERR_INVALID_ARG);
    TP_CHECK(mode == TP_REDUCE_DIRECT || mode == TP_REDUCE_RING || mode == TP_REDUCE_FUSED, TP_ERR_INVALID_ARG);
    TP_CHECK(!(mode == TP_REDUCE_FUSED && !reduce_results), TP_ERR_INVALID_ARG);
    TP_CHECK(in_full % t == 0, TP_ERR_NOT_DIVISIBLE);
    const int64_t ks = in_full / t;
    TP_CHECK(ks % 8 == 0, TP_ERR_ALIGNMENT);
    TP_CHECK(ld_ok(ldx, ks, 2) && ld_ok(ldw, ks, 2), TP_ERR_ALIGNMENT);
    const bool fused = mode == TP_REDUCE_FUSED;
    if (!fused) {
        TP_CHECK(partials != nullptr, TP_ERR_INVALID_ARG);
        TP_CHECK(dtype_ok(partial_dtype), TP_ERR_UNSUPPORTED);
        TP_CHECK(ldp >= out, TP_ERR_INVALID_ARG);
        if (reduce_results) TP_CHECK(ldp == out, TP_ERR_UNSUPPORTED);   // the reduce streams contiguous partials
    }
    if (reduce_results) {
        TP_CHECK(y != nullptr || n == 0, TP_ERR_INVALID_ARG);
        TP_CHECK(dtype_ok(y_dtype), TP_ERR_UNSUPPORTED);
        TP_CHECK(al16(y), TP_ERR_ALIGNMENT);
        TP_CHECK(ldy >= out, TP_ERR_INVALID_ARG);
        if (!fused) TP_CHECK(ldy == out, TP_ERR_UNSUPPORTED);
    }
    for (int r = 0; r < t; ++r) {
        TP_CHECK((x[r] != nullptr || n == 0) && w[r] != nullptr, TP_ERR_INVALID_ARG);
        TP_CHECK(al16(x[r]) && al16(w[r]), TP_ERR_ALIGNMENT);
        if (!fused) {
            TP_CHECK(partials[r] != nullptr || n == 0, TP_ERR_INVALID_ARG);
            TP_CHECK(al16(partials[r]), TP_ERR_ALIGNMENT);
        }
    }
    if (n == 0) return TP_OK;
    tpk::GemmDesc d;
    d.M = n;
    d.N = out;
    d.K = ks;
    d.lda = ldx;
    d.ldb = ldw;
    d.b_rows = out;
    d.status = status_ptr();
    d.pdl = pdl_first ? 1 : 2;
    apply_knobs(d);
    if (fused) {
        d.groups = 1;
        d.segs = t;
        for (int r = 0; r < t; ++r) {
            d.a[r] = x[r];
            d.b[r] = w[r];
        }
        d.out[0] = y;
        d.bias[0] = bias;
        d.ldo = ldy;
        d.out_f32 = y_dtype == TP_F32;
        // A caller's partial buffer, unused by a fused reduce, may hold the stream-K tail area when
        // its rows are contiguous (ldp == out): then its n * out elements are all the caller's, with
        // no padding between rows that could belong to other data.
        const size_t p0_bytes = (ldp == out && dtype_ok(partial_dtype))
                                    ? static_cast<size_t>(n) * static_cast<size_t>(out) * esize(partial_dtype)
                                    : 0;
        if (sk_ws == nullptr && partials != nullptr && partials[0] != nullptr && n > 128 && al16(partials[0]) &&
            p0_bytes >= tpk::kSkWorkspaceBytes) {
            sk_ws = partials[0];
            sk_bytes = p0_bytes;
            if (cudaMemsetAsync(sk_ws, 0, tpk::kSkFlagBytes, cs(stream)) != cudaSuccess) return TP_ERR_CUDA;
        }
        d.sk_ws = sk_ws;
        d.sk_ws_bytes = sk_bytes;
        g_collectives++;
        return tpk::launch_gemm(d, cs(stream));
    }
    d.groups = t;
    d.a_per_group = 1;
    for (int r = 0; r < t; ++r) {
        d.a[r] = x[r];
        d.b[r] = w[r];
        d.out[r] = partials[r];
        d.bias[r] = r == 0 ? bias : nullptr;   // rank 0 alone adds the bias
    }
    d.ldo = ldp;
    d.out_f32 = partial_dtype == TP_F32;
    tp_status st = tpk::launch_gemm(d, cs(stream));
    if (st != TP_OK || !reduce_results) return st;
    return shard_reduce_impl(t, n * out, partial_dtype, reinterpret_cast<const void* const*>(partials), y, y_dtype,
                             mode, partial_dtype, 0, 1, stream);
}

tp_status tp_linear_row(int t, int64_t n, int64_t in_full, int64_t out, const void* const* x, int64_t ldx,
                        const void* const* w, int64_t ldw, const void* bias, int reduce_results, tp_reduce_mode mode,
                        tp_dtype partial_dtype, void* const* partials, int64_t ldp, void* y, int64_t ldy,
                        tp_dtype y_dtype, tp_stream stream) {
    return linear_row_impl(t, n, in_full, out, x, ldx, w, ldw, bias, reduce_results, mode, partial_dtype, partials,
                           ldp, y, ldy, y_dtype, 0, stream);
}

size_t tp_mlp_workspace_size(int t, int64_t n, int64_t h, int64_t f, tp_reduce_mode mode, tp_dtype partial_dtype) {
    const size_t base = tpk::mlp_workspace_required(t, n, h, f, mode, partial_dtype);
    if (base == 0) return 0;
    return std::max(base + mlp_tail_bytes(n, mode), tpk::small_mlp_workspace(t, n, h, f, mode));
}

tp_status tp_mlp_forward(int t, int64_t n, int64_t h, int64_t f, const void* x, int64_t ldx,
                         const void* const* w_gate_up, const void* const* w_down, int64_t ld_down,
                         const void* bias_down, tp_act act, tp_reduce_mode mode, tp_dtype partial_dtype,
                         void* workspace, size_t workspace_bytes, void* y, tp_dtype y_dtype, tp_stream stream) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(n >= 0 && h > 0 && f > 0, TP_ERR_INVALID_ARG);
    TP_CHECK(n <= INT32_MAX && h <= INT32_MAX && f <= INT32_MAX, TP_ERR_INVALID_ARG);
    TP_CHECK((x != nullptr || n == 0) && w_gate_up != nullptr && w_down != nullptr && (y != nullptr || n == 0),
             TP_ERR_INVALID_ARG);
    TP_CHECK(act == TP_ACT_SILU_MUL || act == TP_ACT_GELU_TANH_MUL, TP_ERR_INVALID_ARG);
    TP_CHECK(mode == TP_REDUCE_DIRECT || mode == TP_REDUCE_RING || mode == TP_REDUCE_FUSED, TP_ERR_INVALID_ARG);
    TP_CHECK(dtype_ok(partial_dtype) && dtype_ok(y_dtype), TP_ERR_UNSUPPORTED);
    TP_CHECK(f % t == 0, TP_ERR_NOT_DIVISIBLE);
    const int64_t fs = f / t;
    TP_CHECK(fs % 8 == 0 && h % 8 == 0, TP_ERR_ALIGNMENT);
    TP_CHECK(al16(x) && ld_ok(ldx, h, 2) && ld_ok(ld_down, fs, 2) && al16(y), TP_ERR_ALIGNMENT);
    for (int r = 0; r < t; ++r) {
        TP_CHECK(w_gate_up[r] != nullptr && w_down[r] != nullptr, TP_ERR_INVALID_ARG);
        TP_CHECK(al16(w_gate_up[r]) && al16(w_down[r]), TP_ERR_ALIGNMENT);
    }
    const size_t need = tpk::mlp_workspace_required(t, n, h, f, mode, partial_dtype);
    TP_CHECK(workspace != nullptr || need == 0, TP_ERR_WORKSPACE);
    TP_CHECK(workspace_bytes >= need, TP_ERR_WORKSPACE);
    TP_CHECK((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, TP_ERR_ALIGNMENT);
    if (n == 0) return TP_OK;

    // One to eight tokens with a fused reduce: one GEMM kernel for both
    // projections plus the ordered reduce, when the workspace holds the
    // slices' partials (tp_mlp_workspace_size includes them).
    const size_t small = tpk::small_mlp_workspace(t, n, h, f, mode);
    if (small > 0 && workspace_bytes >= small) {
        tpk::SmallMlpDesc d;
        d.t = t;
        d.n = n;
        d.h = h;
        d.f = f;
        d.x = x;
        d.ldx = ldx;
        for (int r = 0; r < t; ++r) {
            d.w_gate_up[r] = w_gate_up[r];
            d.w_down[r] = w_down[r];
        }
        d.ld_down = ld_down;
        d.bias = bias_down;
        d.act = act;
        d.part = static_cast<float*>(workspace);
        d.y = y;
        d.y_f32 = y_dtype == TP_F32;
        d.status = status_ptr();
        g_collectives++;
        return tpk::launch_small_mlp(d, cs(stream));
    }

    // Workspace: H [n, f] bf16 (rank r's slice = columns [r*fs, (r+1)*fs)),
    // then t partials [n, h], or, for a fused reduce when the workspace holds
    // it, the stream-K tail area (its flags zeroed here, ahead of both GEMMs).
    char* ws = static_cast<char*>(workspace);
    uint16_t* hbuf = reinterpret_cast<uint16_t*>(ws);
    void* parts[TP_MAX_SHARDS] = {};
    if (mode != TP_REDUCE_FUSED) {
        char* p = ws + align256(static_cast<size_t>(n) * f * 2);
        const size_t pb = align256(static_cast<size_t>(n) * h * esize(partial_dtype));
        for (int r = 0; r < t; ++r) parts[r] = p + r * pb;
    }
    void* sk_ws = nullptr;
    const size_t tail = mlp_tail_bytes(n, mode);
    if (tail > 0 && workspace_bytes >= need + tail) {
        sk_ws = ws + need;
        if (cudaMemsetAsync(sk_ws, 0, tpk::kSkFlagBytes, cs(stream)) != cudaSuccess) return TP_ERR_CUDA;
    }

    // 1) column-parallel gate_up with the gated activation in the epilogue.
    tpk::GemmDesc c;
    c.M = n;
    c.N = fs;
    c.K = h;
    c.groups = t;
    c.a[0] = x;
    c.lda = ldx;
    c.ldb = h;
    c.b_rows = 2 * fs;
    c.glu = 1;
    c.glu_up_row = fs;
    c.act = act;
    c.ldo = f;
    c.out_f32 = 0;
    c.status = status_ptr();
    c.pdl = 2;
    apply_knobs(c);
    for (int r = 0; r < t; ++r) {
        c.b[r] = w_gate_up[r];
        c.out[r] = hbuf + r * fs;
    }
    tp_status st = tpk::launch_gemm(c, cs(stream));
    if (st != TP_OK) return st;

    // 2) row-parallel down projection + the all-reduce.
    const void* hx[TP_MAX_SHARDS];
    for (int r = 0; r < t; ++r) hx[r] = hbuf + r * fs;
    return linear_row_impl(t, n, f, h, hx, f, w_down, ld_down, bias_down, 1, mode, partial_dtype, parts, h, y, h,
                           y_dtype, 1, stream, sk_ws, sk_ws != nullptr ? tail : 0);
}

tp_status vocab_parallel_embed(int t, int64_t vocab, int64_t h, const int32_t* ids, int64_t n,
                               const void* const* table, tp_dtype dtype, void* out, void* const* partials,
                               tp_stream stream) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(vocab > 0 && vocab <= INT32_MAX && h > 0 && h <= INT32_MAX && n >= 0, TP_ERR_INVALID_ARG);
    TP_CHECK(n <= static_cast<int64_t>(INT32_MAX) * 4, TP_ERR_INVALID_ARG);   // one warp per id, four per block
    TP_CHECK(table != nullptr && ((out != nullptr && ids != nullptr) || n == 0), TP_ERR_INVALID_ARG);
    TP_CHECK(dtype_ok(dtype), TP_ERR_UNSUPPORTED);
    TP_CHECK((h * esize(dtype)) % 16 == 0, TP_ERR_ALIGNMENT);
    TP_CHECK(al16(out), TP_ERR_ALIGNMENT);
    const int64_t per = (vocab + t - 1) / t;
    tpk::EmbedDesc d;
    d.t = t;
    d.vocab = vocab;
    d.h = h;
    d.n = n;
    d.per = per;
    d.ids = ids;
    d.bf16 = dtype == TP_BF16;
    d.out = out;
    d.with_partials = partials != nullptr;
    for (int r = 0; r < t; ++r) {
        const int64_t start = std::min<int64_t>(r * per, vocab);
        const int64_t end = std::min<int64_t>((r + 1) * per, vocab);
        if (end > start) {
            TP_CHECK(table[r] != nullptr, TP_ERR_INVALID_ARG);
            TP_CHECK(al16(table[r]), TP_ERR_ALIGNMENT);
        }
        d.table[r] = table[r];
        if (partials != nullptr) {
            TP_CHECK(partials[r] != nullptr || n == 0, TP_ERR_INVALID_ARG);
            TP_CHECK(al16(partials[r]), TP_ERR_ALIGNMENT);
            d.partials[r] = partials[r];
        }
    }
    if (n == 0) return TP_OK;
    g_collectives++;
    return tpk::launch_vocab_embed(d, cs(stream));
}

tp_status lm_head_sharded(int t, int64_t n, int64_t h, int64_t vocab, const void* x, int64_t ldx,
                          const void* const* table, void* logits, int64_t ldl, void* const* shard_logits,
                          tp_dtype out_dtype, tp_stream stream) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(n >= 0 && h > 0 && vocab > 0, TP_ERR_INVALID_ARG);
    TP_CHECK(n <= INT32_MAX && vocab <= INT32_MAX && h <= INT32_MAX, TP_ERR_INVALID_ARG);
    TP_CHECK((x != nullptr || n == 0) && table != nullptr, TP_ERR_INVALID_ARG);
    TP_CHECK(logits != nullptr || shard_logits != nullptr || n == 0, TP_ERR_INVALID_ARG);
    TP_CHECK(dtype_ok(out_dtype), TP_ERR_UNSUPPORTED);
    TP_CHECK(h % 8 == 0, TP_ERR_ALIGNMENT);
    TP_CHECK(al16(x) && ld_ok(ldx, h, 2), TP_ERR_ALIGNMENT);
    const int eo = esize(out_dtype);
    if (logits != nullptr) {
        TP_CHECK(al16(logits), TP_ERR_ALIGNMENT);
        TP_CHECK(ldl >= vocab, TP_ERR_INVALID_ARG);
    }
    const int64_t per = (vocab + t - 1) / t;
    tpk::GemmDesc d;
    d.M = n;
    d.N = per;
    d.K = h;
    d.a[0] = x;
    d.lda = ldx;
    d.ldb = h;
    d.b_rows = per;
    d.out_f32 = out_dtype == TP_F32;
    d.ldo = logits != nullptr ? ldl : 0;
    d.pdl = 2;
    int g = 0;
    for (int r = 0; r < t; ++r) {
        const int64_t start = std::min<int64_t>(r * per, vocab);
        const int64_t end = std::min<int64_t>((r + 1) * per, vocab);
        const int64_t rows = end - start;
        if (rows == 0) continue;   // an empty vocab range contributes no columns
        TP_CHECK(table[r] != nullptr, TP_ERR_INVALID_ARG);
        TP_CHECK(al16(table[r]), TP_ERR_ALIGNMENT);
        d.b[g] = table[r];
        d.n_valid[g] = rows;
        if (logits != nullptr) {
            d.out[g] = static_cast<char*>(logits) + start * eo;
        } else if (n > 0) {
            TP_CHECK(shard_logits[r] != nullptr, TP_ERR_INVALID_ARG);
            TP_CHECK(al16(shard_logits[r]), TP_ERR_ALIGNMENT);
            d.out[g] = shard_logits[r];
        }
        ++g;
    }
    d.groups = g;
    if (n == 0) return TP_OK;
    d.status = status_ptr();
    apply_knobs(d);
    if (logits == nullptr) {
        // per-shard buffers are contiguous [n, rows_r]: one launch per distinct width
        int first = 0;
        tp_status st = TP_OK;
        while (first < g && st == TP_OK) {
            int last = first;
            while (last + 1 < g && d.n_valid[last + 1] == d.n_valid[first]) ++last;
            tpk::GemmDesc e = d;
            e.groups = last - first + 1;
            for (int i = 0; i < e.groups; ++i) {
                e.b[i] = d.b[first + i];
                e.out[i] = d.out[first + i];
                e.n_valid[i] = d.n_valid[first + i];
            }
            e.N = d.n_valid[first];
            e.ldo = d.n_valid[first];
            st = tpk::launch_gemm(e, cs(stream));
            first = last + 1;
        }
        return st;
    }
    g_collectives++;
    return tpk::launch_gemm(d, cs(stream));
}

tp_status tp_reduce_scatter_rmsnorm(int t, int64_t n, int64_t h, tp_dtype dtype, const void* const* partials,
                                    const void* residual, const void* weight, float eps, tp_reduce_mode mode,
                                    void* residual_out, void* out, tp_stream stream) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(n >= 0 && h > 0 && partials != nullptr && weight != nullptr && (out != nullptr || n == 0),
             TP_ERR_INVALID_ARG);
    TP_CHECK(mode == TP_REDUCE_DIRECT || mode == TP_REDUCE_RING, TP_ERR_INVALID_ARG);
    TP_CHECK(eps >= 0.0f, TP_ERR_INVALID_ARG);
    TP_CHECK(dtype_ok(dtype), TP_ERR_UNSUPPORTED);
    TP_CHECK(h % 8 == 0, TP_ERR_ALIGNMENT);
    TP_CHECK(h <= 32768, TP_ERR_UNSUPPORTED);
    TP_CHECK(al16(weight) && al16(out) && (residual == nullptr || al16(residual)) &&
                 (residual_out == nullptr || al16(residual_out)),
             TP_ERR_ALIGNMENT);
    for (int r = 0; r < t; ++r) {
        TP_CHECK(partials[r] != nullptr || n == 0, TP_ERR_INVALID_ARG);
        TP_CHECK(al16(partials[r]), TP_ERR_ALIGNMENT);
    }
    if (n == 0) return TP_OK;
    tpk::SeqParDesc d;
    d.t = t;
    d.n = n;
    d.h = h;
    d.in_bf16 = dtype == TP_BF16;
    for (int r = 0; r < t; ++r) d.p[r] = partials[r];
    d.residual = residual;
    d.weight = weight;
    d.residual_out = residual_out;
    d.out = out;
    d.eps = eps;
    d.ring = mode == TP_REDUCE_RING;
    g_collectives++;
    return tpk::launch_seqpar_rmsnorm(d, cs(stream));
}

tp_status tp_shard_gather(int t, int64_t rows, const int64_t* cols, tp_dtype dtype, const void* const* shards,
                          void* out, tp_stream stream) {
    TP_CHECK(t >= 1 && t <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(rows >= 0 && cols != nullptr && shards != nullptr && (out != nullptr || rows == 0), TP_ERR_INVALID_ARG);
    TP_CHECK(dtype_ok(dtype), TP_ERR_UNSUPPORTED);
    tpk::GatherDesc d;
    d.t = t;
    d.rows = rows;
    d.elem_bytes = esize(dtype);
    d.out = out;
    for (int r = 0; r < t; ++r) {
        TP_CHECK(cols[r] >= 0, TP_ERR_INVALID_ARG);
        TP_CHECK(cols[r] == 0 || rows == 0 || shards[r] != nullptr, TP_ERR_INVALID_ARG);
        d.cols[r] = cols[r];
        d.shards[r] = shards[r];
    }
    if (rows == 0) return TP_OK;
    g_collectives++;
    return tpk::launch_shard_gather(d, cs(stream));
}

tp_status tp_device_status(tp_stream stream) {
    if (cudaStreamSynchronize(cs(stream)) != cudaSuccess) return TP_ERR_CUDA;
    int* p = status_ptr();
    if (p == nullptr) return TP_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TP_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return TP_ERR_CUDA;
    }
    return static_cast<tp_status>(v);
}

tp_status tp_set_gemm_tile_n(int n) {
    if (n != 0 && n != 64 && n != 96 && n != 128 && n != 256) return TP_ERR_INVALID_ARG;
    g_tile_n.store(n);
    return TP_OK;
}

tp_status tp_set_gemm_cta_pair(int mode) {
    if (mode < -1 || mode > 1) return TP_ERR_INVALID_ARG;
    g_pair.store(mode);
    return TP_OK;
}

tp_status tp_set_gemm_split(int mode, int max_clusters) {
    if (mode < -1 || mode > 1 || max_clusters < 0) return TP_ERR_INVALID_ARG;
    g_split.store(mode);
    g_split_clusters.store(max_clusters);
    return TP_OK;
}

tp_status tp_debug_gemm_plan(int64_t m, int64_t n, int64_t k, int groups, int segs, int gated, int sms, int* kind,
                             int* tile_n, int* cluster) {
    TP_CHECK(m > 0 && n > 0 && k > 0 && sms >= 1, TP_ERR_INVALID_ARG);
    TP_CHECK(groups >= 1 && groups <= TP_MAX_SHARDS && segs >= 1 && segs <= TP_MAX_SHARDS, TP_ERR_INVALID_ARG);
    TP_CHECK(groups == 1 || segs == 1, TP_ERR_INVALID_ARG);
    TP_CHECK(kind != nullptr && tile_n != nullptr && cluster != nullptr, TP_ERR_INVALID_ARG);
    tpk::GemmDesc d;
    d.M = m;
    d.N = n;
    d.K = k;
    d.groups = groups;
    d.segs = segs;
    d.glu = gated ? 1 : 0;
    const tpk::GemmPlan p = tpk::plan_gemm(d, sms);
    *kind = p.kind;
    *tile_n = p.bn;
    *cluster = p.cs;
    return TP_OK;
}

tp_status tp_debug_expire_wait(uint64_t limit_ns, tp_stream stream) {
    if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
    int* p = status_ptr();
    if (p == nullptr) return TP_ERR_CUDA;
    return tpk::launch_expire_wait(limit_ns, p, cs(stream));
}

}  // extern "C"
