"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Integer-valued inputs make GEMM results exact in fp32, so those cases are
compared bit for bit; float cases use the gates of tests/gpu_helpers.py.
Shapes span several tiles with ragged tails in M, N and K, and the edge
cases of each layer (t = 1, empty ranges, out-of-range ids, specials).
"""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

from gpu_helpers import exact, f64, gemm_gate, h_flip_check, half_ulp_bf16, mlp_check

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    tp.load()
    torch.cuda.init()
    yield
    assert tp.tp_device_status() == 0


def ints(shape, seed, lo=-3, hi=3, dtype=torch.bfloat16):
    return synth.int_valued(shape, lo, hi, seed, dtype=dtype, device=DEV)


def normal(shape, std, seed):
    return synth.normal_bf16(shape, std, seed, device=DEV)


# ------------------------------------------------------------ column parallel

@pytest.mark.parametrize("t,n,k,os_", [(1, 200, 320, 136), (2, 130, 192, 264), (4, 5, 64, 72), (3, 257, 128, 40)])
@pytest.mark.parametrize("gather", [False, True])
def test_linear_col_integer_exact(t, n, k, os_, gather):
    x = ints((n, k), 1)
    w = [ints((os_, k), 10 + r) for r in range(t)]
    b = [ints((os_,), 20 + r, -8, 8) for r in range(t)]
    y = tp.tp_linear_col(x, w, bias=b, gather_output=gather, y_dtype=torch.float32)
    torch.cuda.synchronize()
    xf = f64(x)
    refs = [O.linear(xf, f64(w[r]), f64(b[r])) for r in range(t)]
    if gather:
        exact(f64(y), O.shard_gather(refs))
    else:
        for r in range(t):
            exact(f64(y[r]), refs[r])


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("n", [8, 200])
def test_linear_col_gated_tiny_config(act, n):
    # tiny TP-MLP config: t=2, h=1024, f=3072 -> per-shard gate_up [3072, 1024]
    t, h, f = 2, 1024, 3072
    fs = f // t
    x = normal((n, h), 1.0, 0)
    wg, wu = normal((f, h), 0.02, 1), normal((f, h), 0.02, 2)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    for ydt in (torch.float32, torch.bfloat16):
        ys = tp.tp_linear_col(x, wgu, act=act, y_dtype=ydt)
        torch.cuda.synchronize()
        xf, wgf, wuf = f64(x), f64(wg), f64(wu)
        for r in range(t):
            blk = O.merged_column_shard([wgf, wuf], t, r)
            ref = O.glu(O.linear(xf, blk[:fs]), O.linear(xf, blk[fs:]), act)
            gemm_gate(f64(ys[r]), ref, bf16_out=ydt == torch.bfloat16)


def test_linear_col_gated_ragged_tiles():
    # f/t not a multiple of the 128-wide output tile, n and h ragged
    t, n, h, fs = 3, 131, 200, 88
    x = normal((n, h), 1.0, 5)
    wgu = [normal((2 * fs, h), 0.05, 6 + r) for r in range(t)]
    ys = tp.tp_linear_col(x, wgu, act="silu", y_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        w = f64(wgu[r])
        ref = O.glu(O.linear(f64(x), w[:fs]), O.linear(f64(x), w[fs:]), "silu")
        gemm_gate(f64(ys[r]), ref, bf16_out=False)


# --------------------------------------------------------------- row parallel

@pytest.mark.parametrize("mode", ["fused", "direct", "ring"])
@pytest.mark.parametrize("t,n,ks,out", [(2, 200, 192, 264), (4, 7, 64, 72), (1, 129, 128, 256), (3, 64, 96, 40)])
def test_linear_row_integer_exact(mode, t, n, ks, out):
    x = [ints((n, ks), 30 + r) for r in range(t)]
    w = [ints((out, ks), 40 + r) for r in range(t)]
    bias = ints((out,), 50, -8, 8)
    y = tp.tp_linear_row(x, w, bias=bias, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    parts = [O.linear(f64(x[r]), f64(w[r]), f64(bias) if r == 0 else None) for r in range(t)]
    exact(f64(y), O.reduce_direct(parts))


def test_linear_row_partials_bias_on_rank0_only():
    t, n, ks, out = 4, 16, 64, 48
    x = [ints((n, ks), 60 + r) for r in range(t)]
    w = [ints((out, ks), 70 + r) for r in range(t)]
    bias = ints((out,), 80, 1, 9)
    parts = tp.tp_linear_row(x, w, bias=bias, reduce_results=False, partial_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        exact(f64(parts[r]), O.linear(f64(x[r]), f64(w[r]), f64(bias) if r == 0 else None))


def test_row_worked_example_from_page():
    # Nano-vLLM walkthrough 22, section 4: W=[[1,2,3,4],[5,6,7,8]], b=[10,20], x=[[1,1,1,1]], t=2.
    # Padded to the 8-element row pitch the ABI needs: the extra columns are zero.
    W = torch.zeros((2, 16), dtype=torch.bfloat16, device=DEV)
    W[:, 0:2] = torch.tensor([[1, 2], [5, 6]], dtype=torch.bfloat16)
    W[:, 8:10] = torch.tensor([[3, 4], [7, 8]], dtype=torch.bfloat16)
    x = torch.zeros((1, 16), dtype=torch.bfloat16, device=DEV)
    x[0, 0:2] = 1
    x[0, 8:10] = 1
    b = torch.tensor([10, 20], dtype=torch.bfloat16, device=DEV)
    parts = tp.tp_linear_row([x[:, :8], x[:, 8:]], [W[:, :8], W[:, 8:]], bias=b, reduce_results=False,
                             partial_dtype=torch.float32,
                             partials=[torch.empty((1, 4), device=DEV)[:, :2] for _ in range(2)])   # row stride 4
    torch.cuda.synchronize()
    assert parts[0][:, :2].tolist() == [[13.0, 31.0]] and parts[1][:, :2].tolist() == [[7.0, 15.0]]


# --------------------------------------------------------------- shard reduce

def _partials(t, count, dtype, seed):
    if dtype == torch.bfloat16:
        return [synth.normal_bf16((count,), 1.0, seed + r, device=DEV) for r in range(t)]
    return [synth.normal_f32((count,), 1.0, seed + r, device=DEV) for r in range(t)]


@pytest.mark.parametrize("t", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("count", [1, 7, 8 * 1024 + 5, 3 * 65536])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_shard_reduce_bit_exact_vs_emulation(t, count, dtype):
    parts = _partials(t, count, dtype, 100)
    pf = [f64(p) for p in parts]
    # direct, float32 carry, output in the partial dtype and in fp32
    y = tp.tp_shard_reduce(parts, mode="direct")
    y32 = tp.tp_shard_reduce(parts, mode="direct", out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref32 = O.reduce_direct_f32(pf)
    exact(f64(y32), ref32)
    exact(f64(y), O.round_to_bf16(ref32) if dtype == torch.bfloat16 else ref32)
    # ring, float32 carry
    yr = tp.tp_shard_reduce(parts, mode="ring", out_dtype=torch.float32, hop_dtype=torch.float32)
    torch.cuda.synchronize()
    bufs, _ = O.ring_allreduce(pf, hop="f32")
    exact(f64(yr), bufs[0])
    if dtype == torch.bfloat16:
        # ring with a bf16 wire: every hop rounds
        yb = tp.tp_shard_reduce(parts, mode="ring", hop_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        bufs, _ = O.ring_allreduce(pf, hop="bf16")
        exact(f64(yb), bufs[0])


@pytest.mark.parametrize("mode", ["direct", "ring"])
def test_shard_reduce_replicate_is_allreduce(mode):
    t, count = 4, 10000 + 3
    parts = _partials(t, count, torch.bfloat16, 200)
    pf = [f64(p) for p in parts]
    tp.tp_shard_reduce(parts, mode=mode, replicate=True, hop_dtype=torch.float32)
    torch.cuda.synchronize()
    if mode == "direct":
        ref = O.round_to_bf16(O.reduce_direct_f32(pf))
    else:
        ref = O.round_to_bf16(O.ring_allreduce(pf, hop="f32")[0][0])
    for p in parts:
        exact(f64(p), ref)


def test_shard_reduce_fp32_within_1e6_of_fp64():
    for t in (2, 4, 8):
        parts = _partials(t, 1 << 20, torch.float32, 300 + t)
        y = tp.tp_shard_reduce(parts, mode="direct")
        torch.cuda.synchronize()
        ref = O.reduce_direct([f64(p) for p in parts])
        assert np.max(np.abs(f64(y) - ref)) <= 1e-6 * np.max(np.abs(ref))


def test_shard_reduce_ring_order_observable():
    # bf16 wire: element c of chunk c holds 1.0 at the rank that adds it last;
    # the two small values meet first and survive (see the oracle pin).
    a, e = 1.0, 2.0 ** -8
    n = 3
    vals = [[e, a, e], [e, e, a], [a, e, e]]
    parts = [torch.tensor(v, dtype=torch.bfloat16, device=DEV) for v in vals]
    out = tp.tp_shard_reduce(parts, mode="ring", hop_dtype=torch.bfloat16)
    direct = tp.tp_shard_reduce(parts, mode="direct")
    torch.cuda.synchronize()
    assert out.float().tolist() == [1.0 + 2 ** -7] * n
    assert direct.float().tolist() == [1.0 + 2 ** -7] * n   # fp32 carry keeps every bit here


# -------------------------------------------------------------------- MLP

@pytest.mark.parametrize("mode", ["direct", "ring", "fused"])
@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
def test_mlp_forward_tiny_config(mode, act):
    # t=2, h=1024, f=3072, n=8 tokens, W ~ N(0, 0.02), X ~ N(0, 1), seed 0
    t, n, h, f = 2, 8, 1024, 3072
    fs = f // t
    x = normal((n, h), 1.0, 0)
    wg, wu, wd = normal((f, h), 0.02, 1), normal((f, h), 0.02, 2), normal((h, f), 0.02, 3)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs] for r in range(t)]          # column views, ld = f
    xf, wgf, wuf, wdf = f64(x), f64(wg), f64(wu), f64(wd)
    for pdt in (torch.float32, torch.bfloat16):
        for ydt in (torch.float32, torch.bfloat16):
            y = tp.tp_mlp_forward(x, wgu, wds, act=act, mode=mode, partial_dtype=pdt, y_dtype=ydt)
            torch.cuda.synchronize()
            mlp_check(f64(y), xf, wgf, wuf, wdf, t, act=act, mode=mode,
                      partial="bf16" if pdt == torch.bfloat16 else "f32", y_bf16=ydt == torch.bfloat16)


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("t,n,h,fs", [(2, 8, 1024, 1536), (2, 600, 320, 200), (4, 130, 256, 72)])
def test_gated_column_h_is_the_exact_rounding(act, t, n, h, fs):
    """H = act(G) * U stored in bf16 is the exact value's rounding, up to flips
    at rounding midpoints, on the tiny config and on ragged multi-tile shapes
    (single-CTA and CTA-pair kernels)."""
    x = normal((n, h), 1.0, 260)
    wgu = [normal((2 * fs, h), 0.02 if h >= 1024 else 0.05, 261 + r) for r in range(t)]
    hs = tp.tp_linear_col(x, wgu, act=act)
    torch.cuda.synchronize()
    xf = f64(x)
    for r in range(t):
        w = f64(wgu[r])
        h_flip_check(f64(hs[r]), O.glu(O.linear(xf, w[:fs]), O.linear(xf, w[fs:]), act))


def test_mlp_forward_integer_variant_and_bias():
    # integer-valued (-3..3) variant of the tiny config; bias added once
    t, n, h, f = 2, 8, 1024, 3072
    fs = f // t
    x = ints((n, h), 0)
    wg, wu, wd = ints((f, h), 1), ints((f, h), 2), ints((h, f), 3)
    bias = ints((h,), 4, -8, 8)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    xf, wgf, wuf, wdf, bf = f64(x), f64(wg), f64(wu), f64(wd), f64(bias)
    for mode in ("direct", "ring", "fused"):
        for pdt in (torch.float32, torch.bfloat16):
            y = tp.tp_mlp_forward(x, wgu, wds, bias_down=bias, mode=mode, partial_dtype=pdt, y_dtype=torch.float32)
            torch.cuda.synchronize()
            mlp_check(f64(y), xf, wgf, wuf, wdf, t, bias=bf, mode=mode,
                      partial="bf16" if pdt == torch.bfloat16 else "f32")


def test_mlp_decode_shapes_small():
    # decode-like: a handful of tokens against wide shards
    t, h, f = 4, 512, 2048
    fs = f // t
    wg, wu, wd = normal((f, h), 0.02, 11), normal((f, h), 0.02, 12), normal((h, f), 0.02, 13)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs] for r in range(t)]
    for n in (1, 16, 64):
        x = normal((n, h), 1.0, 20 + n)
        for mode in ("direct", "fused"):
            y = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
            torch.cuda.synchronize()
            mlp_check(f64(y), f64(x), f64(wg), f64(wu), f64(wd), t, mode=mode)


# ---------------------------------------------------------------- embedding

def _table_shards(table, t):
    v = table.shape[0]
    out = []
    for r in range(t):
        s, e = O.vocab_range(v, t, r)
        out.append(table[s:e].contiguous() if e > s else None)
    return out


@pytest.mark.parametrize("t", [2, 4])
def test_vocab_embed_bit_exact_config(t):
    V, h, n = 151936, 1024, 4096
    table = normal((V, h), 0.02, 6)
    ids = synth.uniform_ids(n, V, 5, device=DEV)
    shards = _table_shards(table, t)
    partials = [torch.empty((n, h), dtype=torch.bfloat16, device=DEV) for _ in range(t)]
    out = tp.vocab_parallel_embed(ids, shards, V, partials=partials)
    torch.cuda.synchronize()
    ref, refp = O.vocab_parallel_embedding(ids.cpu().numpy(), f64(table), t)
    exact(f64(out), ref)
    for r in range(t):
        exact(f64(partials[r]), refp[r])


@pytest.mark.parametrize("t,V", [(1, 50), (3, 50), (4, 3), (8, 101)])
def test_vocab_embed_edges(t, V):
    h = 16
    table = normal((V, h), 1.0, 7)
    tb = table.clone()
    tb[0, 0] = float("nan")
    tb[0, 1] = float("inf")
    tb[0, 2] = -0.0
    ids = torch.tensor([-1, V, 10 ** 6, 0, V - 1, -(2 ** 31), 2 ** 31 - 1] + list(range(min(V, 20))),
                       dtype=torch.int32, device=DEV)
    out = tp.vocab_parallel_embed(ids, _table_shards(tb, t), V)
    torch.cuda.synchronize()
    ref, _ = O.vocab_parallel_embedding(ids.cpu().numpy(), f64(tb), t)
    exact(f64(out), ref)


@pytest.mark.parametrize("t", [1, 2, 3])
def test_vocab_embed_every_bf16_pattern(t):
    """The all-reduce of one row and t-1 exact zeros, formed on packed bf16
    pairs: every one of the 65536 bf16 bit patterns (zeros of both signs,
    subnormals, infinities, NaNs) as a table value, against the oracle's sum."""
    V, h = 64, 1024
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(V, h)
    table = bits.view(torch.bfloat16).to(DEV)
    ids = torch.tensor(list(range(V - 1, -1, -1)) + [-5, V, 7], dtype=torch.int32, device=DEV)
    parts = [torch.empty((ids.numel(), h), dtype=torch.bfloat16, device=DEV) for _ in range(t)]
    out = tp.vocab_parallel_embed(ids, _table_shards(table, t), V, partials=parts)
    torch.cuda.synchronize()
    ref, refp = O.vocab_parallel_embedding(ids.cpu().numpy(), f64(table), t)
    exact(f64(out), ref)
    for r in range(t):
        exact(f64(parts[r]), refp[r])
    if t == 1:       # a single rank's lookup is the row itself, NaN payloads included
        assert torch.equal(out[:V].view(torch.int16), table[ids[:V].long()].view(torch.int16))


@pytest.mark.parametrize("t", [1, 3])
def test_vocab_embed_f32_table(t):
    V, h, n = 37, 20, 300
    table = synth.normal_f32((V, h), 1.0, 8, device=DEV)
    table[0, :4] = torch.tensor([float("nan"), float("-inf"), -0.0, 1e-41])
    ids = synth.uniform_ids(n, V + 3, 9, device=DEV) - 1      # includes -1 and ids >= V
    out = tp.vocab_parallel_embed(ids, _table_shards(table, t), V)
    torch.cuda.synchronize()
    ref, _ = O.vocab_parallel_embedding(ids.cpu().numpy(), f64(table), t)
    exact(f64(out), ref)


def test_vocab_embed_many_ids_ragged():
    """More ids than one wave of warps (one warp per id, n/4 blocks) with a ragged last block."""
    V, h, n, t = 151936, 1024, 70001, 4
    table = normal((V, h), 0.02, 6)
    ids = synth.uniform_ids(n, V, 15, device=DEV)
    out = tp.vocab_parallel_embed(ids, _table_shards(table, t), V)
    torch.cuda.synchronize()
    ref, _ = O.vocab_parallel_embedding(ids.cpu().numpy(), f64(table), t)
    exact(f64(out), ref)


def test_vocab_embed_worked_example_structure():
    # vLLM source analysis 13, section 2.4.1: V=10, ids [[1,6],[3,8]], two ranges of 5 rows
    V, h, t = 10, 8, 2
    table = normal((V, h), 1.0, 42)
    ids = torch.tensor([1, 6, 3, 8], dtype=torch.int32, device=DEV)
    parts = [torch.empty((4, h), dtype=torch.bfloat16, device=DEV) for _ in range(t)]
    out = tp.vocab_parallel_embed(ids, _table_shards(table, t), V, partials=parts)
    torch.cuda.synchronize()
    owners = [0, 1, 0, 1]
    for i, o in enumerate(owners):
        assert torch.count_nonzero(parts[1 - o][i]) == 0
        assert torch.equal(parts[o][i], table[ids[i].item()])
    assert torch.equal(out, table[ids.long()])


# ------------------------------------------------------------------ LM head

@pytest.mark.parametrize("t,V,n,h", [(2, 1000, 130, 64), (3, 1000, 64, 128), (4, 151936, 96, 1024), (8, 77, 5, 32)])
def test_lm_head_concat_and_per_shard(t, V, n, h):
    x = normal((n, h), 1.0, 8)
    table = normal((V, h), 0.02, 6)
    shards = _table_shards(table, t)
    logits = tp.lm_head_sharded(x, shards, V, out_dtype=torch.float32)
    per = tp.lm_head_sharded(x, shards, V, per_shard=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref, refp = O.lm_head_sharded(f64(x), f64(table), t)
    gemm_gate(f64(logits), ref, bf16_out=False)
    for r in range(t):
        if refp[r].shape[1]:
            gemm_gate(f64(per[r]), refp[r], bf16_out=False)
    # the explicit all-gather of the per-shard logits gives the same bits
    nonempty = [p for p in per if p.shape[1] > 0]
    cat = tp.tp_shard_gather(nonempty)
    torch.cuda.synchronize()
    exact(f64(cat), f64(logits))


def test_lm_head_integer_exact_bf16():
    t, V, n, h = 4, 1024, 136, 256
    x = ints((n, h), 9)
    table = ints((V, h), 10)
    logits = tp.lm_head_sharded(x, _table_shards(table, t), V, out_dtype=torch.float32)
    torch.cuda.synchronize()
    exact(f64(logits), O.lm_head_unsharded(f64(x), f64(table)))


# -------------------------------------------------------------- gather / misc

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_shard_gather_bit_exact(dtype):
    cols = [8, 3, 0, 16, 5]
    shards = [synth.normal_f32((37, c), 1.0, 400 + i, device=DEV).to(dtype) for i, c in enumerate(cols)]
    out = tp.tp_shard_gather(shards)
    torch.cuda.synchronize()
    exact(f64(out), O.shard_gather([f64(s) for s in shards]))


def test_collective_counter_counts_reduces():
    t, n, h, f = 2, 8, 256, 512
    x = normal((n, h), 1.0, 1)
    wgu = [normal((f, h), 0.02, 2 + r) for r in range(t)]
    wds = [normal((h, f // t), 0.02, 5 + r) for r in range(t)]
    tp.tp_reset_collective_count()
    tp.tp_mlp_forward(x, wgu, wds, mode="direct")
    tp.tp_mlp_forward(x, wgu, wds, mode="fused")
    torch.cuda.synchronize()
    assert tp.tp_collective_count() == 2     # one all-reduce per MLP, as the pages count them


def test_bounded_wait_expires_and_reports():
    tp.tp_debug_expire_wait(2_000_000)       # 2 ms on a barrier nothing signals
    assert tp.tp_device_status() == 6        # TP_ERR_TIMEOUT, and the context still works
    assert tp.tp_device_status() == 0        # cleared
    a = torch.ones(16, device=DEV, dtype=torch.bfloat16)
    out = tp.tp_shard_reduce([a, a])
    torch.cuda.synchronize()
    assert out.float().sum().item() == 32.0


# ------------------------------------------------- every tile width, exactly

@pytest.fixture
def tile_n(request):
    tp.tp_set_gemm_tile_n(request.param)
    yield request.param
    tp.tp_set_gemm_tile_n(0)


@pytest.mark.parametrize("tile_n", [64, 96, 128, 256], indirect=True)
def test_every_tile_width_integer_exact(tile_n):
    # plain column GEMM: ragged M (300), N (200 per shard), K (8 blocks + 24)
    t, n, k, os_ = 2, 300, 536, 200
    x = ints((n, k), 90)
    w = [ints((os_, k), 91 + r) for r in range(t)]
    y = tp.tp_linear_col(x, w, y_dtype=torch.float32)
    # row GEMM, fused over 3 K-segments and unfused
    xs = [ints((n, 136), 95 + r) for r in range(3)]
    ws = [ints((264, 136), 98 + r) for r in range(3)]
    yf = tp.tp_linear_row(xs, ws, mode="fused", y_dtype=torch.float32)
    yd = tp.tp_linear_row(xs, ws, mode="direct", partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        exact(f64(y[r]), O.linear(f64(x), f64(w[r])))
    ref = O.reduce_direct([O.linear(f64(xs[r]), f64(ws[r])) for r in range(3)])
    exact(f64(yf), ref)
    exact(f64(yd), ref)


@pytest.mark.parametrize("tile_n", [64, 96, 128, 256], indirect=True)
@pytest.mark.parametrize("k", [2200, 2560])
@pytest.mark.parametrize("n", [1, 5, 8, 9, 12, 16, 17, 64])
def test_every_tile_width_few_rows(tile_n, n, k):
    """Decode-sized GEMMs at every tile width: up to 8 rows take the 8-row A tiles
    with the deepest B rings (24 stages at width 64), 9 to 16 rows the 16-row A
    tiles, 17 to 64 rows the 64-row A tiles.  K = 2200 (35 blocks, a ragged last
    one) wraps every ring with one box per K block; K = 2560 (40 blocks) loads the
    16- and 64-row tiles' groups of K blocks as single boxes.  The plain and the
    row GEMMs are integer-exact, the gated GEMM's H is the exact rounding up to
    flips at midpoints."""
    t, os_ = 3, 328
    x = ints((n, k), 130 + n)
    w = [ints((os_, k), 131 + r) for r in range(t)]
    y = tp.tp_linear_col(x, w, y_dtype=torch.float32)
    xs = [ints((n, k), 140 + r) for r in range(t)]
    ws = [ints((os_, k), 145 + r) for r in range(t)]
    yd = tp.tp_linear_row(xs, ws, mode="direct", partial_dtype=torch.float32, y_dtype=torch.float32)
    xg = normal((n, k), 1.0, 150)
    wgu = [normal((2 * os_, k), 0.02, 151 + r) for r in range(t)]
    hs = tp.tp_linear_col(xg, wgu, act="silu", y_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    for r in range(t):
        exact(f64(y[r]), O.linear(f64(x), f64(w[r])))
    exact(f64(yd), O.reduce_direct([O.linear(f64(xs[r]), f64(ws[r])) for r in range(t)]))
    for r in range(t):
        wr = f64(wgu[r])
        h_flip_check(f64(hs[r]), O.glu(O.linear(f64(xg), wr[:os_]), O.linear(f64(xg), wr[os_:]), "silu"))


@pytest.mark.parametrize("tile_n", [64, 96, 128, 256], indirect=True)
def test_every_tile_width_gated(tile_n):
    t, n, h, fs = 2, 260, 320, 200
    x = normal((n, h), 1.0, 120)
    wgu = [normal((2 * fs, h), 0.05, 121 + r) for r in range(t)]
    ys = tp.tp_linear_col(x, wgu, act="silu", y_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        w = f64(wgu[r])
        ref = O.glu(O.linear(f64(x), w[:fs]), O.linear(f64(x), w[fs:]), "silu")
        gemm_gate(f64(ys[r]), ref, bf16_out=False)


@pytest.mark.parametrize("t", [3, 5, 8])
@pytest.mark.parametrize("count", [20, 37, 100, 1003])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_shard_reduce_ring_chunks_shorter_than_vectors(t, count, dtype):
    # chunk = ceil(count/t) can be shorter than a 16-byte vector, so several
    # chunk boundaries cut the same vector; with replicate every element must
    # still be folded exactly once from the original partials.
    parts = _partials(t, count, dtype, 900 + t)
    pf = [f64(p) for p in parts]
    out = torch.empty((count,), dtype=torch.float32, device=DEV)
    tp.tp_shard_reduce(parts, out=out, mode="ring", replicate=True)
    torch.cuda.synchronize()
    bufs, _ = O.ring_allreduce(pf, hop="f32")
    exact(f64(out), bufs[0])
    rounded = O.round_to_bf16(bufs[0]) if dtype == torch.bfloat16 else bufs[0]
    for p in parts:
        exact(f64(p), rounded)


# ------------------------------------------------------ CTA-pair GEMM kernel

@pytest.fixture
def pair_on():
    tp.tp_set_gemm_cta_pair(1)
    yield
    tp.tp_set_gemm_cta_pair(0)


def test_pair_kernel_integer_exact(pair_on):
    # ragged M (300: the second CTA of the second tile has no rows), N, K
    t, n, k, os_ = 2, 300, 536, 200
    x = ints((n, k), 190)
    w = [ints((os_, k), 191 + r) for r in range(t)]
    b = [ints((os_,), 193 + r, -8, 8) for r in range(t)]
    y = tp.tp_linear_col(x, w, bias=b, y_dtype=torch.float32)
    yg = tp.tp_linear_col(x, w, bias=b, gather_output=True, y_dtype=torch.float32)
    xs = [ints((n, 136), 195 + r) for r in range(3)]
    ws = [ints((264, 136), 198 + r) for r in range(3)]
    yf = tp.tp_linear_row(xs, ws, mode="fused", y_dtype=torch.float32)
    yd = tp.tp_linear_row(xs, ws, mode="direct", partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    refs = [O.linear(f64(x), f64(w[r]), f64(b[r])) for r in range(t)]
    for r in range(t):
        exact(f64(y[r]), refs[r])
    exact(f64(yg), O.shard_gather(refs))
    ref = O.reduce_direct([O.linear(f64(xs[r]), f64(ws[r])) for r in range(3)])
    exact(f64(yf), ref)
    exact(f64(yd), ref)
    assert tp.tp_device_status() == 0


@pytest.mark.parametrize("t,V,n,h", [(3, 1000, 520, 128), (4, 151936, 256, 1024)])
def test_pair_kernel_lm_head(pair_on, t, V, n, h):
    x = ints((n, h), 210)
    table = ints((V, h), 211)
    logits = tp.lm_head_sharded(x, _table_shards(table, t), V, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = sorted({r for r in (0, 1, 127, 128, 255, 256, n - 1) if r < n})
    exact(f64(logits[rows]), O.lm_head_unsharded(f64(x[rows]), f64(table)))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_pair_kernel_line_staged_stores(pair_on, dtype):
    """The CTA-pair store epilogue writes whole 128-byte output lines through
    shared memory when the row pitch allows it.  Logits in a buffer with a
    320-column pitch: with bf16 the second shard starts 64 bytes into a line
    (its first chunk falls back to per-row stores), every shard ends in a
    partial line, the last row-tile is ragged; the pad columns must stay
    untouched and every logit exact."""
    t, V, n, h, pitch = 3, 288, 520, 128, 320
    x = ints((n, h), 260)
    table = ints((V, h), 261)
    canary = -12345.0
    buf = torch.full((n, pitch), canary, dtype=dtype, device=DEV)
    logits = buf[:, :V]
    tp.lm_head_sharded(x, _table_shards(table, t), V, logits=logits, out_dtype=dtype)
    torch.cuda.synchronize()
    exact(f64(logits.contiguous()), O.lm_head_unsharded(f64(x), f64(table)))
    assert bool(torch.all(buf[:, V:] == canary).item())
    assert tp.tp_device_status() == 0


def test_pair_kernel_gated(pair_on):
    t, n, h, fs = 2, 600, 320, 200
    x = normal((n, h), 1.0, 220)
    wgu = [normal((2 * fs, h), 0.05, 221 + r) for r in range(t)]
    ys = tp.tp_linear_col(x, wgu, act="silu", y_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        w = f64(wgu[r])
        ref = O.glu(O.linear(f64(x), w[:fs]), O.linear(f64(x), w[fs:]), "silu")
        gemm_gate(f64(ys[r]), ref, bf16_out=False)


@pytest.mark.parametrize("mode", ["direct", "fused"])
def test_pair_kernel_mlp(pair_on, mode):
    t, n, h, f = 2, 520, 1024, 3072
    fs = f // t
    x = normal((n, h), 1.0, 230)
    wg, wu, wd = normal((f, h), 0.02, 231), normal((f, h), 0.02, 232), normal((h, f), 0.02, 233)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs] for r in range(t)]
    y = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    mlp_check(f64(y), f64(x), f64(wg), f64(wu), f64(wd), t, mode=mode)


@pytest.mark.parametrize("chunks", [1, 3, 4])
def test_mlp_forward_host_matches_device_entry_point(chunks):
    t, n, h, f = 2, 1000, 1024, 3072
    fs = f // t
    x = normal((n, h), 1.0, 240)
    wg, wu, wd = normal((f, h), 0.02, 241), normal((f, h), 0.02, 242), normal((h, f), 0.02, 243)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs] for r in range(t)]
    y_dev = tp.tp_mlp_forward(x, wgu, wds, mode="direct", partial_dtype=torch.float32, y_dtype=torch.float32)
    xh = torch.empty((n, h), dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(x)
    yh = torch.full((n, h), float("nan"), dtype=torch.float32, pin_memory=True)
    ws = torch.empty(tp.tp_mlp_host_workspace_size(t, n, h, f, chunks, "direct", torch.float32), dtype=torch.uint8,
                     device=DEV)
    xd = torch.empty_like(x)
    yd = torch.empty((n, h), dtype=torch.float32, device=DEV)
    tp.tp_mlp_forward_host(xh, wgu, wds, y_host=yh, x_dev=xd, y_dev=yd, workspace=ws, mode="direct",
                           partial_dtype=torch.float32, chunks=chunks)
    torch.cuda.current_stream().synchronize()
    got = O.f32_bits_to_f64(yh.view(torch.int32).numpy().view(np.uint32))
    # rows are independent and every kernel choice depends only on the block's shape, so
    # the host-buffer path gives the device entry point's bits where the blocks match:
    # one block, or with two or more chunks short first and last blocks around chunks - 1
    # taller ones
    if chunks == 1:
        assert torch.equal(yh.to(DEV), y_dev)
    else:
        bounds = tp.tp_mlp_host_blocks(n, chunks)
        assert len(bounds) == chunks + 2 and bounds[1] == n - bounds[-2] == 128
        for a, b in zip(bounds, bounds[1:]):
            yb = tp.tp_mlp_forward(x[a:b], wgu, wds, mode="direct", partial_dtype=torch.float32,
                                   y_dtype=torch.float32)
            assert torch.equal(yh[a:b].to(DEV), yb), (a, b)
    mlp_check(got, f64(x), f64(wg), f64(wu), f64(wd), t)


@pytest.mark.parametrize("mode", ["direct", "fused"])
@pytest.mark.parametrize("n,chunks", [(1, 1), (3, 8), (7, 2), (13, 64), (40, 5), (129, 3)])
def test_mlp_forward_host_small_blocks(n, chunks, mode):
    """Few tokens cut into many row blocks (down to one row): each block's MLP is the device
    entry point's on that block, bit for bit; in fused mode blocks of up to 8 rows take the
    one-kernel path (h = 1024, 64-column slices) when the workspace holds their partials."""
    t, h, f = 2, 1024, 3072
    fs = f // t
    x = normal((n, h), 1.0, 250 + n)
    wg, wu, wd = normal((f, h), 0.02, 251), normal((f, h), 0.02, 252), normal((h, f), 0.02, 253)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs] for r in range(t)]
    ws = torch.empty(tp.tp_mlp_host_workspace_size(t, n, h, f, chunks, mode, torch.float32), dtype=torch.uint8,
                     device=DEV)
    xh = torch.empty((n, h), dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(x)
    yh = torch.full((n, h), float("nan"), dtype=torch.float32, pin_memory=True)
    xd = torch.empty_like(x)
    yd = torch.empty((n, h), dtype=torch.float32, device=DEV)
    tp.tp_mlp_forward_host(xh, wgu, wds, y_host=yh, x_dev=xd, y_dev=yd, workspace=ws, mode=mode,
                           partial_dtype=torch.float32, chunks=chunks)
    torch.cuda.current_stream().synchronize()
    assert tp.tp_device_status() == 0
    bounds = tp.tp_mlp_host_blocks(n, chunks)
    assert bounds[0] == 0 and bounds[-1] == n and len(bounds) <= chunks + 2
    for a, b in zip(bounds, bounds[1:]):
        yb = tp.tp_mlp_forward(x[a:b], wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32,
                               workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(yh[a:b].to(DEV), yb), (a, b)
    got = O.f32_bits_to_f64(yh.view(torch.int32).numpy().view(np.uint32))
    mlp_check(got, f64(x), f64(wg), f64(wu), f64(wd), t, mode=mode)


# ------------------------------------------- sequence parallelism (RS + norm)

def _rs_fold_f32(pf, t, n, order):
    """fp32 fold of each row's partials in its owner's reduce-scatter order."""
    out = np.empty_like(pf[0])
    for r, (lo, hi) in enumerate(O.token_chunks(n, t)):
        seq = list(range(t)) if order == "direct" else O.reduce_scatter_fold_order(t, r)
        acc = pf[seq[0]][lo:hi].astype(np.float32)
        for j in seq[1:]:
            acc = (acc + pf[j][lo:hi].astype(np.float32)).astype(np.float32)
        out[lo:hi] = acc
    return out


@pytest.mark.parametrize("t,n,h", [(1, 5, 64), (2, 9, 1000), (3, 10, 256), (4, 37, 8192), (8, 20, 512)])
@pytest.mark.parametrize("order", ["direct", "ring"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_reduce_scatter_rmsnorm(t, n, h, order, dtype):
    parts = [(synth.normal_f32((n, h), 1.0, 500 + r, device=DEV)).to(dtype) for r in range(t)]
    resid = normal((n, h), 1.0, 520)
    w = normal((h,), 1.0, 521)
    res_out = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    _, out = tp.tp_reduce_scatter_rmsnorm(parts, w, residual=resid, eps=1e-6, mode=order, residual_out=res_out)
    torch.cuda.synchronize()
    pf = [f64(p) for p in parts]
    # the new residual: bit-exact against the fp32 fold in the owner's order, + residual, rounded once
    x32 = (_rs_fold_f32(pf, t, n, order).astype(np.float32) + f64(resid).astype(np.float32)).astype(np.float32)
    exact(f64(res_out), O.round_to_bf16(x32.astype(np.float64)))
    # the normed rows against the fp64 oracle
    _, normed, _ = O.sequence_parallel_residual_norm(pf, f64(resid), f64(w), 1e-6, order)
    got = f64(out)
    bound = half_ulp_bf16(normed) + 1e-4 * np.abs(normed) + 1e-6
    assert np.all(np.abs(got - normed) <= bound), float(np.max(np.abs(got - normed) - bound))


def _random_seqpar_shapes(count, seed):
    """Seeded shapes: t 1..8, n 1..300 (rows not divisible by t included), h a multiple of 8
    up to 32768, orders and partial dtypes mixed."""
    rnd = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        t = int(rnd.integers(1, 9))
        n = int(rnd.integers(1, 301))
        h = 8 * int(rnd.choice([rnd.integers(1, 129), rnd.integers(129, 4097)]))
        out.append((t, n, h, str(rnd.choice(["direct", "ring"])), bool(rnd.integers(0, 2))))
    return out


@pytest.mark.parametrize("t,n,h,order,f32", _random_seqpar_shapes(12, 404))
def test_reduce_scatter_rmsnorm_random(t, n, h, order, f32):
    dtype = torch.float32 if f32 else torch.bfloat16
    parts = [(synth.normal_f32((n, h), 1.0, 600 + r, device=DEV)).to(dtype) for r in range(t)]
    resid = normal((n, h), 1.0, 620)
    w = normal((h,), 1.0, 621)
    res_out = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    _, out = tp.tp_reduce_scatter_rmsnorm(parts, w, residual=resid, eps=1e-6, mode=order, residual_out=res_out)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    pf = [f64(p) for p in parts]
    x32 = (_rs_fold_f32(pf, t, n, order).astype(np.float32) + f64(resid).astype(np.float32)).astype(np.float32)
    exact(f64(res_out), O.round_to_bf16(x32.astype(np.float64)))
    _, normed, _ = O.sequence_parallel_residual_norm(pf, f64(resid), f64(w), 1e-6, order)
    got = f64(out)
    bound = half_ulp_bf16(normed) + 1e-4 * np.abs(normed) + 1e-6
    assert np.all(np.abs(got - normed) <= bound), float(np.max(np.abs(got - normed) - bound))


def test_reduce_scatter_rmsnorm_in_place_and_no_residual():
    t, n, h = 4, 16, 256
    parts = [normal((n, h), 1.0, 530 + r) for r in range(t)]
    resid = normal((n, h), 1.0, 540)
    w = normal((h,), 1.0, 541)
    r0 = resid.clone()
    tp.tp_reduce_scatter_rmsnorm(parts, w, residual=resid, residual_out=resid)       # in place
    _, out0 = tp.tp_reduce_scatter_rmsnorm(parts, w)                                # no residual stream
    torch.cuda.synchronize()
    pf = [f64(p) for p in parts]
    x32 = (_rs_fold_f32(pf, t, n, "direct").astype(np.float32) + f64(r0).astype(np.float32)).astype(np.float32)
    exact(f64(resid), O.round_to_bf16(x32.astype(np.float64)))
    _, normed, _ = O.sequence_parallel_residual_norm(pf, None, f64(w), 1e-6)
    assert np.all(np.abs(f64(out0) - normed) <= half_ulp_bf16(normed) + 1e-4 * np.abs(normed) + 1e-6)


# ---------------------------------------------------- QKV column-parallel linear

def test_qkv_worked_example_through_linear_col():
    # Nano-vLLM walkthrough 22, section 5: q 4 heads, k/v 2 heads, head_size 2, t=2; every row of head
    # h holds the head's constant.  Hidden is padded from 3 to 8 columns (the ABI's row pitch); x picks
    # column 0, so output column j of rank r is the constant of the j-th row of rank r's merged block.
    hs, hid, t = 2, 8, 2

    def by_head(nheads, base):
        return torch.tensor([[float(base + h)] * hid for h in range(nheads) for _ in range(hs)], dtype=torch.bfloat16)

    q, k, v = by_head(4, 0), by_head(2, 10), by_head(2, 20)
    blocks = [torch.from_numpy(O.qkv_shard(q.float().numpy(), k.float().numpy(), v.float().numpy(), 4, 2, hs, t, r))
              .to(torch.bfloat16).to(DEV) for r in range(t)]
    x = torch.zeros((1, hid), dtype=torch.bfloat16, device=DEV)
    x[0, 0] = 1
    y = tp.tp_linear_col(x, blocks, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert y[0][0].tolist() == [0.0, 0.0, 1.0, 1.0, 10.0, 10.0, 20.0, 20.0]
    assert y[1][0].tolist() == [2.0, 2.0, 3.0, 3.0, 11.0, 11.0, 21.0, 21.0]


@pytest.mark.parametrize("t,nh,nkv,hd", [(2, 16, 8, 64), (4, 32, 8, 128), (8, 64, 8, 128)])
def test_qkv_merged_layout_integer_exact(t, nh, nkv, hd):
    hid, n = 256, 70
    wq, wk, wv = ints((nh * hd, hid), 300), ints((nkv * hd, hid), 301), ints((nkv * hd, hid), 302)
    x = ints((n, hid), 303)
    wqf, wkf, wvf = f64(wq), f64(wk), f64(wv)
    blocks = [synth.from_bits_u16(O.bf16_from_f64_bits(O.qkv_shard(wqf, wkf, wvf, nh, nkv, hd, t, r)), device=DEV)
              for r in range(t)]
    y = tp.tp_linear_col(x, blocks, y_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        exact(f64(y[r]), O.linear(f64(x), O.qkv_shard(wqf, wkf, wvf, nh, nkv, hd, t, r)))


@pytest.mark.parametrize("t,nh,nkv,hd", [(8, 64, 4, 64), (4, 32, 2, 64)])
def test_qkv_gqa_replicated_layout_integer_exact(t, nh, nkv, hd):
    # t > KV heads: each rank's block carries one replicated KV head (6.2 Tensor-parallel inference, §2.2)
    hid, n = 128, 40
    wq, wk, wv = ints((nh * hd, hid), 310), ints((nkv * hd, hid), 311), ints((nkv * hd, hid), 312)
    x = ints((n, hid), 313)
    wqf, wkf, wvf = f64(wq), f64(wk), f64(wv)
    blocks = [synth.from_bits_u16(O.bf16_from_f64_bits(O.qkv_shard_gqa(wqf, wkf, wvf, nh, nkv, hd, t, r)), device=DEV)
              for r in range(t)]
    y = tp.tp_linear_col(x, blocks, y_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        exact(f64(y[r]), O.linear(f64(x), O.qkv_shard_gqa(wqf, wkf, wvf, nh, nkv, hd, t, r)))


# --------------------------------------------- split-K kernel of the fused reduce

@pytest.fixture
def split_knob(request):
    mode, cap = request.param
    tp.tp_set_gemm_split(mode, cap)
    yield mode, cap
    tp.tp_set_gemm_split(0, 0)


# (mode, max clusters): automatic; always with every cluster resident; always with one
# cluster walking every tile and with three (the staging hand-off between tiles)
@pytest.mark.parametrize("split_knob", [(0, 0), (1, 0), (1, 1), (1, 3)], indirect=True)
@pytest.mark.parametrize("t,n,ks,out", [(2, 1, 64, 1000), (3, 9, 200, 520), (4, 64, 128, 8192), (5, 17, 64, 300),
                                        (8, 33, 96, 2056)])
def test_fused_row_split_k_integer_exact(split_knob, t, n, ks, out):
    x = [ints((n, ks), 60 + r) for r in range(t)]
    w = [ints((out, ks), 70 + r) for r in range(t)]
    bias = ints((out,), 80, -8, 8)
    y = tp.tp_linear_row(x, w, bias=bias, mode="fused", y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    parts = [O.linear(f64(x[r]), f64(w[r]), f64(bias) if r == 0 else None) for r in range(t)]
    exact(f64(y), O.reduce_direct(parts))


@pytest.mark.parametrize("split_knob", [(0, 0), (1, 0), (1, 2)], indirect=True)
@pytest.mark.parametrize("t,n,ks,out", [(3, 5, 512, 100), (2, 64, 1024, 600), (1, 8, 320, 256)])
def test_split_k_within_shards_integer_exact(split_knob, t, n, ks, out):
    """K ranges that cut through shards (cluster size not dividing t), the
    row GEMM writing per-shard partials, and the column GEMM, all through the
    split-K kernel when it applies."""
    x = [ints((n, ks), 110 + r) for r in range(t)]
    w = [ints((out, ks), 120 + r) for r in range(t)]
    bias = ints((out,), 130, -8, 8)
    parts = [O.linear(f64(x[r]), f64(w[r]), f64(bias) if r == 0 else None) for r in range(t)]
    if t > 1:
        y = tp.tp_linear_row(x, w, bias=bias, mode="fused", y_dtype=torch.float32)
        p32 = tp.tp_linear_row(x, w, bias=bias, reduce_results=False, partial_dtype=torch.float32)
        torch.cuda.synchronize()
        exact(f64(y), O.reduce_direct(parts))
        for r in range(t):
            exact(f64(p32[r]), parts[r])
    # column parallel: shard r of the output is x[0] @ w[r]^T (+ its bias slice)
    bcol = [ints((out,), 140 + r, -8, 8) for r in range(t)]
    yc = tp.tp_linear_col(x[0], w, bias=bcol, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    for r in range(t):
        exact(f64(yc[r]), O.linear(f64(x[0]), f64(w[r]), f64(bcol[r])))


@pytest.mark.parametrize("split_knob", [(0, 0), (1, 1)], indirect=True)
@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("t,n,h,f", [(2, 8, 1024, 3072), (4, 33, 512, 2048), (3, 1, 256, 600)])
def test_split_k_gated_column(split_knob, act, t, n, h, f):
    x = normal((n, h), 1.0, 150)
    wg = normal((f, h), 0.02, 151)
    wu = normal((f, h), 0.02, 152)
    fs = f // t
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    hs = tp.tp_linear_col(x, wgu, act=act)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    xf, wgf, wuf = f64(x), f64(wg), f64(wu)
    for r in range(t):
        ref = O.glu(O.linear(xf, wgf[r * fs:(r + 1) * fs]), O.linear(xf, wuf[r * fs:(r + 1) * fs]), act)
        gemm_gate(f64(hs[r]), ref, bf16_out=True)


@pytest.mark.parametrize("t", [2, 4, 8])
@pytest.mark.parametrize("n", [1, 16, 64])
def test_fused_row_split_k_float_and_deterministic(t, n):
    ks, out = 256, 4096
    x = [normal((n, ks), 1.0, 90 + r) for r in range(t)]
    w = [normal((out, ks), 0.02, 100 + r) for r in range(t)]
    y1 = tp.tp_linear_row(x, w, mode="fused")
    y2 = tp.tp_linear_row(x, w, mode="fused")
    y32 = tp.tp_linear_row(x, w, mode="fused", y_dtype=torch.float32)
    tp.tp_set_gemm_split(-1, 0)
    try:
        y_plain = tp.tp_linear_row(x, w, mode="fused", y_dtype=torch.float32)
    finally:
        tp.tp_set_gemm_split(0, 0)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    ref = O.reduce_direct([O.linear(f64(x[r]), f64(w[r])) for r in range(t)])
    gemm_gate(f64(y1), ref, bf16_out=True)
    gemm_gate(f64(y32), ref, bf16_out=False)
    gemm_gate(f64(y_plain), ref, bf16_out=False)


def test_allreduce_count_of_a_28_layer_forward(golden_dir):
    """The call sequence of one prefill forward at TP=2 (embedding, then per
    layer the attention output projection and the MLP, then the LM head) on
    tiny shapes: the library counts one collective per all-reduce the page
    counts, and the LM head adds its gather."""
    import json, os
    with open(os.path.join(golden_dir, "tpscratch_allreduce_count.json")) as fh:
        g = json.load(fh)
    t, layers, n, h, f, V = g["tp"], g["layers"], 8, 64, 128, 100
    per = (V + t - 1) // t
    table = normal((V, h), 0.02, 11)
    shards = [table[r * per:min((r + 1) * per, V)].contiguous() for r in range(t)]
    ids = synth.uniform_ids(n, V, 12, device=DEV)
    wo = [normal((h, h // t), 0.02, 13 + r) for r in range(t)]
    wgu = [normal((2 * f // t, h), 0.02, 20 + r) for r in range(t)]
    wds = [normal((h, f // t), 0.02, 30 + r) for r in range(t)]
    tp.tp_reset_collective_count()
    x = tp.vocab_parallel_embed(ids, shards, V)
    for _ in range(layers):
        heads = [x[:, r * (h // t):(r + 1) * (h // t)].contiguous() for r in range(t)]   # stands in for attention
        x = x + tp.tp_linear_row(heads, wo)
        x = x + tp.tp_mlp_forward(x, wgu, wds)
    torch.cuda.synchronize()
    assert tp.tp_collective_count() == g["prefill_forward_allreduces"]
    tp.lm_head_sharded(x, shards, V)
    torch.cuda.synchronize()
    assert tp.tp_collective_count() == g["prefill_forward_allreduces"] + 1


# ------------------------------------------------------------ zero tokens

def test_zero_tokens_every_entry_point():
    """An empty batch (n = 0, empty CUDA tensors, whose data pointers may be null) is a valid
    call of every entry point: each returns its empty outputs, launches nothing (the
    collective counter does not move) and leaves no device error."""
    t, h, f = 2, 256, 1024
    fs = f // t
    x = torch.empty((0, h), dtype=torch.bfloat16, device=DEV)
    wgu = [normal((2 * fs, h), 0.02, 900 + r) for r in range(t)]
    wd = [normal((h, fs), 0.02, 910 + r) for r in range(t)]
    torch.cuda.synchronize()
    tp.tp_reset_collective_count()
    for mode in ("direct", "ring", "fused"):
        assert tp.tp_mlp_forward(x, wgu, wd, mode=mode).shape == (0, h)
        assert tp.tp_mlp_forward_static(x, wgu, wd, mode=mode).shape == (0, h)
        assert tp.tp_linear_row([torch.empty((0, fs), dtype=torch.bfloat16, device=DEV)] * t, wd,
                                mode=mode).shape == (0, h)
    ys = tp.tp_linear_col(x, wgu, act="silu")
    assert [y.shape for y in ys] == [(0, fs)] * t
    assert tp.tp_linear_col(x, [w[:fs] for w in wgu], gather_output=True).shape == (0, f)
    parts = [torch.empty((0,), dtype=torch.float32, device=DEV) for _ in range(t)]
    for mode in ("direct", "ring"):
        assert tp.tp_shard_reduce(parts, mode=mode).shape == (0,)
    xh = torch.empty((0, h), dtype=torch.bfloat16)          # zero bytes need no page-locking
    yh = torch.empty((0, h), dtype=torch.bfloat16)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    assert tp.tp_mlp_forward_host(xh, wgu, wd, y_host=yh, x_dev=x, y_dev=torch.empty_like(x), workspace=ws) is yh
    vocab = 1000
    table = [normal(((vocab + 1) // 2, h), 1.0, 920 + r)[: min((r + 1) * 500, vocab) - r * 500] for r in range(t)]
    table = [tb.contiguous() for tb in table]
    ids = torch.empty((0,), dtype=torch.int32, device=DEV)
    assert tp.vocab_parallel_embed(ids, table, vocab).shape == (0, h)
    assert tp.lm_head_sharded(x, table, vocab).shape == (0, vocab)
    assert [s.shape for s in tp.lm_head_sharded(x, table, vocab, per_shard=True)] == [(0, 500)] * t
    assert tp.tp_shard_gather([torch.empty((0, c), dtype=torch.bfloat16, device=DEV) for c in (8, 16)]).shape == (0, 24)
    sp = [torch.empty((0, h), dtype=torch.float32, device=DEV) for _ in range(t)]
    _, out = tp.tp_reduce_scatter_rmsnorm(sp, normal((h,), 1.0, 930))
    assert out.shape == (0, h)
    torch.cuda.synchronize()
    assert tp.tp_collective_count() == 0
    assert tp.tp_device_status() == 0
