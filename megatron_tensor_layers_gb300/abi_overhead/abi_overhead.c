/*
 * Host cost of enqueuing the C-ABI entry points, with no Python in the loop.
 *
 * For each entry point this program makes `warm` untimed calls, then CALLS
 * calls one after another on one stream, each timed on the host clock from
 * entry to return (enqueue only: the calls do not wait for the GPU).  CALLS
 * stays below the depth of the launch queue, so a call never blocks on the
 * device.  It then times CALLS calls as a whole with CUDA events for the
 * device time per call.  Inputs are zero-filled device buffers at the sizes
 * the entry points see in decode and in the small configurations of the
 * benchmark.  Prints one JSON object: per entry point the median and mean
 * host microseconds per call and the device microseconds per call.
 *
 * Build: gcc -O2 -I<repo>/include -I<cuda>/include abi_overhead.c
 *        -L<package> -ltp_gb300 -L<cuda>/lib64 -lcudart -o abi_overhead
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include "tp.h"

#define CALLS 200

static double now_us(void) {
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return ts.tv_sec * 1e6 + ts.tv_nsec * 1e-3;
}

static void* dev_zero(size_t bytes) {
    void* p = NULL;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc(%zu) failed\n", bytes);
        exit(2);
    }
    cudaMemset(p, 0, bytes);
    return p;
}

static int cmp_double(const void* a, const void* b) {
    const double x = *(const double*)a, y = *(const double*)b;
    return (x > y) - (x < y);
}

typedef tp_status (*call_fn)(void* ctx);

static int first = 1;

static void time_entry(const char* name, call_fn fn, void* ctx, cudaStream_t s) {
    static double host[CALLS];
    for (int i = 0; i < 20; ++i)
        if (fn(ctx) != TP_OK) {
            fprintf(stderr, "%s failed\n", name);
            exit(3);
        }
    cudaStreamSynchronize(s);
    for (int i = 0; i < CALLS; ++i) {
        const double t0 = now_us();
        fn(ctx);
        host[i] = now_us() - t0;
        if ((i & 15) == 15) cudaStreamSynchronize(s); /* keep the launch queue short */
    }
    cudaStreamSynchronize(s);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a, s);
    for (int i = 0; i < CALLS; ++i) fn(ctx);
    cudaEventRecord(b, s);
    cudaEventSynchronize(b);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    double mean = 0.0;
    for (int i = 0; i < CALLS; ++i) mean += host[i];
    mean /= CALLS;
    qsort(host, CALLS, sizeof(double), cmp_double);
    printf("%s\"%s\": {\"host_us_median\": %.3f, \"host_us_mean\": %.3f, \"device_us_per_call\": %.3f}",
           first ? "" : ", ", name, host[CALLS / 2], mean, ms * 1e3 / CALLS);
    first = 0;
}

/* ---- the calls ---- */
typedef struct {
    cudaStream_t s;
    /* reduce: t=4, one token of h=8192 (16 KiB per partial) */
    void* parts[4];
    void* red_out;
    /* tiny MLP: t=2, n=8, h=1024, f=3072 */
    void *x, *wgu[2], *wd[2], *hbuf, *hs[2], *tparts[2], *y, *ws;
    size_t ws_bytes;
    /* embedding: t=2, V=151936, h=1024, 4096 ids */
    void *ids, *table[2], *emb;
} Ctx;

static tp_status c_reduce(void* p) {
    Ctx* c = (Ctx*)p;
    return tp_shard_reduce(4, 8192, TP_BF16, (const void* const*)c->parts, c->red_out, TP_BF16, TP_REDUCE_DIRECT,
                           TP_F32, 0, c->s);
}
static tp_status c_col(void* p) {
    Ctx* c = (Ctx*)p;
    return tp_linear_col(2, 8, 1024, 3072, c->x, 1024, (const void* const*)c->wgu, 1024, NULL, TP_ACT_SILU_MUL, 0,
                         (void* const*)c->hs, 3072, TP_BF16, c->s);
}
static tp_status c_row_fused(void* p) {
    Ctx* c = (Ctx*)p;
    return tp_linear_row(2, 8, 3072, 1024, (const void* const*)c->hs, 3072, (const void* const*)c->wd, 1536, NULL, 1,
                         TP_REDUCE_FUSED, TP_BF16, NULL, 1024, c->y, 1024, TP_BF16, c->s);
}
static tp_status c_mlp_direct(void* p) {
    Ctx* c = (Ctx*)p;
    return tp_mlp_forward(2, 8, 1024, 3072, c->x, 1024, (const void* const*)c->wgu, (const void* const*)c->wd, 1536,
                          NULL, TP_ACT_SILU_MUL, TP_REDUCE_DIRECT, TP_BF16, c->ws, c->ws_bytes, c->y, TP_BF16, c->s);
}
static tp_status c_mlp_fused(void* p) {
    Ctx* c = (Ctx*)p;
    return tp_mlp_forward(2, 8, 1024, 3072, c->x, 1024, (const void* const*)c->wgu, (const void* const*)c->wd, 1536,
                          NULL, TP_ACT_SILU_MUL, TP_REDUCE_FUSED, TP_BF16, c->ws, c->ws_bytes, c->y, TP_BF16, c->s);
}
static tp_status c_embed(void* p) {
    Ctx* c = (Ctx*)p;
    return vocab_parallel_embed(2, 151936, 1024, (const int32_t*)c->ids, 4096, (const void* const*)c->table, TP_BF16,
                                c->emb, NULL, c->s);
}

int main(void) {
    Ctx c;
    memset(&c, 0, sizeof(c));
    if (cudaStreamCreateWithFlags(&c.s, cudaStreamNonBlocking) != cudaSuccess) return 2;
    for (int r = 0; r < 4; ++r) c.parts[r] = dev_zero(8192 * 2);
    c.red_out = dev_zero(8192 * 2);
    c.x = dev_zero(8 * 1024 * 2);
    for (int r = 0; r < 2; ++r) {
        c.wgu[r] = dev_zero((size_t)3072 * 1024 * 2);
        c.wd[r] = dev_zero((size_t)1024 * 1536 * 2);
    }
    c.hbuf = dev_zero((size_t)8 * 3072 * 2);
    c.hs[0] = c.hbuf;
    c.hs[1] = (char*)c.hbuf + 1536 * 2;
    c.y = dev_zero(8 * 1024 * 2);
    c.ws_bytes = tp_mlp_workspace_size(2, 8, 1024, 3072, TP_REDUCE_DIRECT, TP_BF16);
    c.ws = dev_zero(c.ws_bytes);
    c.ids = dev_zero(4096 * 4);
    for (int r = 0; r < 2; ++r) c.table[r] = dev_zero((size_t)75968 * 1024 * 2);
    c.emb = dev_zero((size_t)4096 * 1024 * 2);
    cudaDeviceSynchronize();

    printf("{");
    time_entry("tp_shard_reduce_t4_n1", c_reduce, &c, c.s);
    time_entry("tp_linear_col_tiny_gated", c_col, &c, c.s);
    time_entry("tp_linear_row_tiny_fused", c_row_fused, &c, c.s);
    time_entry("tp_mlp_forward_tiny_direct", c_mlp_direct, &c, c.s);
    time_entry("tp_mlp_forward_tiny_fused", c_mlp_fused, &c, c.s);
    time_entry("vocab_parallel_embed_4096", c_embed, &c, c.s);
    printf(", \"calls\": %d}\n", CALLS);
    return tp_device_status(c.s) == TP_OK ? 0 : 4;
}
