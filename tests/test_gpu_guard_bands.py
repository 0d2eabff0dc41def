"""Guard bands: every kernel writes only inside its outputs.

compute-sanitizer is not available on this machine, so out-of-bounds writes are
caught directly: each output is a strided view inside a larger buffer filled
with a canary pattern (padding after every row and a band after the end),
the kernels run on ragged shapes, and every canary must be intact afterwards.
"""

import pytest
import torch

from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

pytestmark = pytest.mark.gpu
DEV = "cuda"
CANARY_BF16 = -12345          # int16 pattern
CANARY_F32 = -987654321       # int32 pattern


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    tp.load()


def guarded(rows, cols, dtype, pad_cols=24, pad_rows=3):
    """A [rows, cols] view (row stride cols + pad_cols) inside a canary-filled buffer."""
    ld = cols + pad_cols
    itype, canary = (torch.int16, CANARY_BF16) if dtype == torch.bfloat16 else (torch.int32, CANARY_F32)
    buf = torch.full(((rows + pad_rows) * ld,), canary, dtype=itype, device=DEV)
    view = buf.view(dtype)[: rows * ld].view(rows, ld)[:, :cols]
    mask = torch.ones(((rows + pad_rows) * ld,), dtype=torch.bool, device=DEV)
    mask.view(-1)[: rows * ld].view(rows, ld)[:, :cols] = False
    return view, buf, mask, canary


def intact(buf, mask, canary):
    return bool(torch.all(buf[mask] == canary).item())


def ints(shape, seed, dtype=torch.bfloat16):
    return synth.int_valued(shape, -3, 3, seed, dtype=dtype, device=DEV)


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
def test_gemm_outputs_stay_inside(pair, ydt):
    tp.tp_set_gemm_cta_pair(pair if pair else -1)
    try:
        t, n, k, os_ = 3, 530, 200, 136
        x = ints((n, k), 1)
        w = [ints((os_, k), 2 + r) for r in range(t)]
        outs = [guarded(n, os_, ydt) for _ in range(t)]
        tp.tp_linear_col(x, w, y=[o[0] for o in outs], y_dtype=ydt)
        g = guarded(n, os_ * t, ydt)
        tp.tp_linear_col(x, w, gather_output=True, y=g[0], y_dtype=ydt)
        wgu = [ints((2 * os_, k), 9 + r) for r in range(t)]
        hg = [guarded(n, os_, ydt) for _ in range(t)]
        tp.tp_linear_col(x, wgu, act="silu", y=[o[0] for o in hg], y_dtype=ydt)
        xs = [ints((n, 72), 20 + r) for r in range(t)]
        ws = [ints((264, 72), 30 + r) for r in range(t)]
        yf = guarded(n, 264, ydt)
        tp.tp_linear_row(xs, ws, mode="fused", y=yf[0], y_dtype=ydt)
        parts = [guarded(n, 264, torch.float32) for _ in range(t)]
        tp.tp_linear_row(xs, ws, reduce_results=False, partials=[p[0] for p in parts], partial_dtype=torch.float32)
        torch.cuda.synchronize()
        for o in outs + [g] + hg + [yf] + parts:
            assert intact(o[1], o[2], o[3])
    finally:
        tp.tp_set_gemm_cta_pair(0)


def test_lm_head_and_gather_stay_inside():
    t, V, n, h = 3, 1001, 300, 64
    x = ints((n, h), 40)
    table = ints((V, h), 41)
    per = (V + t - 1) // t
    shards = [table[r * per:min((r + 1) * per, V)].contiguous() for r in range(t)]
    lg = guarded(n, V, torch.float32)
    tp.lm_head_sharded(x, shards, V, logits=lg[0], out_dtype=torch.float32)
    per_shard = tp.lm_head_sharded(x, shards, V, per_shard=True, out_dtype=torch.bfloat16)
    cat_buf = torch.full((n * V + 4096,), CANARY_BF16, dtype=torch.int16, device=DEV)
    cat = cat_buf.view(torch.bfloat16)[: n * V].view(n, V)
    tp.tp_shard_gather(per_shard, out=cat)
    torch.cuda.synchronize()
    assert intact(lg[1], lg[2], lg[3])
    assert bool(torch.all(cat_buf[n * V:] == CANARY_BF16).item())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["direct", "ring"])
def test_reduce_embed_seqpar_stay_inside(dtype, mode):
    t, count = 3, 10007
    parts = [synth.normal_f32((count,), 1.0, 50 + r, device=DEV).to(dtype) for r in range(t)]
    itype, canary = (torch.int16, CANARY_BF16) if dtype == torch.bfloat16 else (torch.int32, CANARY_F32)
    ob = torch.full((count + 4096,), canary, dtype=itype, device=DEV)
    tp.tp_shard_reduce(parts, out=ob.view(dtype)[:count], mode=mode)
    # embedding: rows of 16 bf16 in a buffer with a guard band after the last row
    V, h, n = 97, 16, 333
    table = synth.normal_bf16((V, h), 1.0, 60, device=DEV)
    per = (V + t - 1) // t
    shards = [table[r * per:min((r + 1) * per, V)].contiguous() for r in range(t)]
    ids = synth.uniform_ids(n, V, 61, device=DEV)
    eb = torch.full((n * h + 4096,), CANARY_BF16, dtype=torch.int16, device=DEV)
    tp.vocab_parallel_embed(ids, shards, V, out=eb.view(torch.bfloat16)[: n * h].view(n, h))
    # reduce-scatter + RMSNorm
    n2, h2 = 37, 520
    p2 = [synth.normal_f32((n2, h2), 1.0, 70 + r, device=DEV).to(dtype) for r in range(t)]
    w2 = synth.normal_bf16((h2,), 1.0, 80, device=DEV)
    rb = torch.full((n2 * h2 + 4096,), CANARY_BF16, dtype=torch.int16, device=DEV)
    nb = torch.full((n2 * h2 + 4096,), CANARY_BF16, dtype=torch.int16, device=DEV)
    tp.tp_reduce_scatter_rmsnorm(p2, w2, mode=mode, residual_out=rb.view(torch.bfloat16)[: n2 * h2].view(n2, h2),
                                 out=nb.view(torch.bfloat16)[: n2 * h2].view(n2, h2))
    torch.cuda.synchronize()
    assert bool(torch.all(ob[count:] == canary).item())
    assert bool(torch.all(eb[n * h:] == CANARY_BF16).item())
    assert bool(torch.all(rb[n2 * h2:] == CANARY_BF16).item())
    assert bool(torch.all(nb[n2 * h2:] == CANARY_BF16).item())


@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
def test_split_k_cluster_outputs_stay_inside(ydt):
    """The split-K cluster kernel (decode-sized rows) writes through its own
    reduction epilogue: the fused row GEMM, and with the split forced the
    gated column GEMM and per-shard partials."""
    t, n, ks, out = 3, 37, 136, 200
    xs = [ints((n, ks), 50 + r) for r in range(t)]
    ws = [ints((out, ks), 60 + r) for r in range(t)]
    yf = guarded(n, out, ydt)
    tp.tp_linear_row(xs, ws, mode="fused", y=yf[0], y_dtype=ydt)
    tp.tp_set_gemm_split(1, 0)
    try:
        x = ints((n, 256), 70)
        wgu = [ints((2 * 72, 256), 71 + r) for r in range(t)]
        hg = [guarded(n, 72, ydt) for _ in range(t)]
        tp.tp_linear_col(x, wgu, act="silu", y=[o[0] for o in hg], y_dtype=ydt)
        xp = [ints((n, 264), 80 + r) for r in range(t)]        # 5 K blocks: two CTAs per cluster
        wp = [ints((out, 264), 90 + r) for r in range(t)]
        parts = [guarded(n, out, torch.float32) for _ in range(t)]
        tp.tp_linear_row(xp, wp, reduce_results=False, partials=[p[0] for p in parts], partial_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        tp.tp_set_gemm_split(0, 0)
    assert tp.tp_device_status() == 0
    for o in [yf] + hg + parts:
        assert intact(o[1], o[2], o[3])


@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
def test_fused_stream_k_tail_stays_inside(ydt):
    """The fused down GEMM + reduce whose last wave is split along K (1100 rows: 5 row
    tiles, the last ragged, by 32 column tiles of 256): the output is a strided view
    with canaries, and the scratch the call borrows (a contiguous fp32 partials[0])
    sits inside a canary-filled buffer.  The kernel writes the output and, inside the
    scratch, only the flags and the partial slots: every canary outside both survives."""
    t, n, h, fs = 4, 1100, 8192, 1024
    hs = [ints((n, fs), 40 + r) for r in range(t)]
    wds = [ints((h, fs), 50 + r) for r in range(t)]
    y, ybuf, ymask, ycan = guarded(n, h, ydt)
    s, sbuf, smask, scan = guarded(n, h, torch.float32, pad_cols=0, pad_rows=3)
    tp.tp_linear_row(hs, wds, mode="fused", y=y, y_dtype=ydt, partials=[s] * t)
    plain = tp.tp_linear_row(hs, wds, mode="fused", y_dtype=ydt)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    assert intact(ybuf, ymask, ycan)
    assert torch.equal(y, plain)                 # integer inputs: exact with or without the split
    # the scratch's writes stay in its first 32 MiB + 4 KiB, inside the caller's n * h elements
    assert (4096 + 128 * 256 * 256 * 4) // 4 <= n * h
    assert intact(sbuf, smask, scan)


def test_fused_stream_k_on_two_streams():
    """Two fused MLP calls with the stream-K tail on two streams at once, each with its
    own workspace (flags and slots): each result equals the same call made alone."""
    t, n, h, f = 4, 768, 8192, 28672
    fs = f // t
    wgu = [synth.normal_bf16((2 * fs, h), 0.02, 60 + r, device=DEV) for r in range(t)]
    wds = [synth.normal_bf16((h, fs), 0.02, 70 + r, device=DEV) for r in range(t)]
    xs = [synth.normal_bf16((n, h), 1.0, 80 + i, device=DEV) for i in range(2)]
    alone = [tp.tp_mlp_forward(x, wgu, wds, mode="fused") for x in xs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    wss = [torch.empty(tp.tp_mlp_workspace_size(t, n, h, f, "fused", torch.bfloat16), dtype=torch.uint8, device=DEV)
           for _ in range(2)]
    ys = [torch.empty((n, h), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    for _ in range(3):
        for i in range(2):
            streams[i].wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(streams[i]):
                tp.tp_mlp_forward(xs[i], wgu, wds, mode="fused", workspace=wss[i], y=ys[i],
                                  stream=streams[i])
        torch.cuda.synchronize()
        assert tp.tp_device_status() == 0
        for i in range(2):
            assert torch.equal(ys[i], alone[i])


@pytest.mark.parametrize("n", [5, 13])
@pytest.mark.parametrize("tile_n", [64, 96, 128, 256])
@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
def test_few_row_gemm_outputs_stay_inside(tile_n, ydt, n):
    """Five and thirteen rows (the 8- and 16-row A tiles with the deepest B rings) at every
    tile width: the plain, gated and row GEMMs write only inside their outputs."""
    tp.tp_set_gemm_tile_n(tile_n)
    try:
        t, k, os_ = 3, 1000, 200
        x = ints((n, k), 160)
        w = [ints((os_, k), 161 + r) for r in range(t)]
        outs = [guarded(n, os_, ydt) for _ in range(t)]
        tp.tp_linear_col(x, w, y=[o[0] for o in outs], y_dtype=ydt)
        wgu = [ints((2 * os_, k), 165 + r) for r in range(t)]
        hg = [guarded(n, os_, ydt) for _ in range(t)]
        tp.tp_linear_col(x, wgu, act="silu", y=[o[0] for o in hg], y_dtype=ydt)
        xs = [ints((n, k), 170 + r) for r in range(t)]
        pg = [guarded(n, os_, torch.float32, pad_cols=0) for _ in range(t)]
        tp.tp_linear_row(xs, w, reduce_results=False, partials=[o[0] for o in pg], partial_dtype=torch.float32)
        torch.cuda.synchronize()
        assert tp.tp_device_status() == 0
        for o in outs + hg + pg:
            assert intact(o[1], o[2], o[3])
    finally:
        tp.tp_set_gemm_tile_n(0)
