"""Randomized parity sweep over the GEMM, embedding, LM-head and gather entry points.

Seeded random shapes (shard count, tokens, K, output width, all ragged
against the tiles), output dtypes, gather/bias options, reduce orders and the
kernel-selection knobs (CTA pairs, split-K clusters, tile width) drive the
column and row linears through every GEMM kernel and epilogue.  Inputs are
small integers, so every fp32 result is exact and a bf16 result is the exact
value rounded once: both are compared bit for bit with the CPU oracle.  The
gated column GEMM (SiLU is transcendental) uses the float gate.  The
embedding (bf16 and fp32 tables, ids out of range, t > V) and the LM head
with its gather (ragged vocab, so shards start mid-line in the logits) are
swept the same way, bit-exact, and so is the shard reduce (odd counts, any t,
both orders, bf16 or fp32 wire, replication) against the oracle's emulation of
the same fold order.
"""

import random

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

from gpu_helpers import f64, gemm_gate

pytestmark = pytest.mark.gpu

DEV = "cuda"
CASES = 48


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    tp.load()
    torch.cuda.init()
    yield
    assert tp.tp_device_status() == 0


def ints(shape, seed, lo=-3, hi=3):
    return synth.int_valued(shape, lo, hi, seed, dtype=torch.bfloat16, device=DEV)


def _case(i):
    rnd = random.Random(1000 + i)
    t = rnd.choice([1, 2, 3, 4, 5, 8])
    n = rnd.choice([1, 2, 7, 8, 16, 31, 33, 64, 65, 130, 257, 300, 530, 700])
    k = 8 * rnd.randint(1, 64)                    # per-shard K for the row GEMM, in for the column GEMM
    os_ = 8 * rnd.randint(1, 65)                  # per-shard output width
    pair = rnd.choice([-1, 0, 0, 1]) if n >= 64 else rnd.choice([-1, 0])
    split = rnd.choice([-1, 0, 0, 1])
    tile_n = rnd.choice([0, 0, 64, 128, 256]) if pair != 1 else 0
    y_f32 = rnd.random() < 0.5
    return dict(t=t, n=n, k=k, os_=os_, pair=pair, split=split, tile_n=tile_n, y_f32=y_f32,
                gather=rnd.random() < 0.3, bias=rnd.random() < 0.5,
                mode=rnd.choice(["direct", "ring", "fused"]), seed=2000 + 50 * i)


def _knobs(c):
    tp.tp_set_gemm_cta_pair(c["pair"])
    tp.tp_set_gemm_split(c["split"], 0)
    tp.tp_set_gemm_tile_n(c["tile_n"])


def _reset():
    tp.tp_set_gemm_cta_pair(0)
    tp.tp_set_gemm_split(0, 0)
    tp.tp_set_gemm_tile_n(0)


def _expect(ref, y_f32):
    return ref if y_f32 else O.round_to_bf16(ref)


@pytest.mark.parametrize("i", range(CASES))
def test_column_linear_random(i):
    c = _case(i)
    t, n, k, os_, s = c["t"], c["n"], c["k"], c["os_"], c["seed"]
    ydt = torch.float32 if c["y_f32"] else torch.bfloat16
    x = ints((n, k), s)
    w = [ints((os_, k), s + 1 + r) for r in range(t)]
    b = [ints((os_,), s + 20 + r, -8, 8) for r in range(t)] if c["bias"] else None
    _knobs(c)
    try:
        y = tp.tp_linear_col(x, w, bias=b, gather_output=c["gather"], y_dtype=ydt)
        torch.cuda.synchronize()
    finally:
        _reset()
    assert tp.tp_device_status() == 0
    refs = [O.linear(f64(x), f64(w[r]), f64(b[r]) if b else None) for r in range(t)]
    if c["gather"]:
        assert np.array_equal(f64(y), _expect(O.shard_gather(refs), c["y_f32"])), c
    else:
        for r in range(t):
            assert np.array_equal(f64(y[r]), _expect(refs[r], c["y_f32"])), (c, r)


@pytest.mark.parametrize("i", range(CASES))
def test_row_linear_random(i):
    c = _case(i)
    t, n, k, os_, s = c["t"], c["n"], c["k"], c["os_"], c["seed"]
    ydt = torch.float32 if c["y_f32"] else torch.bfloat16
    x = [ints((n, k), s + 30 + r) for r in range(t)]
    w = [ints((os_, k), s + 40 + r) for r in range(t)]
    bias = ints((os_,), s + 49, -8, 8) if c["bias"] else None
    _knobs(c)
    try:
        y = tp.tp_linear_row(x, w, bias=bias, mode=c["mode"], partial_dtype=torch.float32, y_dtype=ydt)
        parts = tp.tp_linear_row(x, w, bias=bias, reduce_results=False, partial_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        _reset()
    assert tp.tp_device_status() == 0
    pref = [O.linear(f64(x[r]), f64(w[r]), f64(bias) if (bias is not None and r == 0) else None) for r in range(t)]
    for r in range(t):
        assert np.array_equal(f64(parts[r]), pref[r]), (c, r)
    # integer partial sums stay below 2^24: every fold order gives the exact sum
    assert np.array_equal(f64(y), _expect(O.reduce_direct(pref), c["y_f32"])), c


@pytest.mark.parametrize("i", range(0, CASES, 3))
def test_gated_column_random(i):
    c = _case(i)
    t, n, k, os_, s = c["t"], c["n"], c["k"], c["os_"], c["seed"]
    x = synth.normal_bf16((n, k), 1.0, s, device=DEV)
    wgu = [synth.normal_bf16((2 * os_, k), 0.05, s + 1 + r, device=DEV) for r in range(t)]
    act = "silu" if i % 2 == 0 else "gelu_tanh"
    _knobs(c)
    try:
        hs = tp.tp_linear_col(x, wgu, act=act, y_dtype=torch.bfloat16)
        torch.cuda.synchronize()
    finally:
        _reset()
    assert tp.tp_device_status() == 0
    xf = f64(x)
    for r in range(t):
        wf = f64(wgu[r])
        ref = O.glu(O.linear(xf, wf[:os_]), O.linear(xf, wf[os_:]), act)
        gemm_gate(f64(hs[r]), ref, bf16_out=True)


def _vocab_case(i):
    rnd = random.Random(5000 + i)
    t = rnd.choice([1, 2, 3, 4, 5, 8])
    vocab = rnd.choice([1, 2, 3, 7, 50, 101, 1000, 4097])
    h = 8 * rnd.randint(1, 40)
    n = rnd.choice([1, 5, 64, 300, 1025])
    return t, vocab, h, n, 6000 + 20 * i


def _vocab_shards(table, vocab, t):
    out = []
    for r in range(t):
        s, e = O.vocab_range(vocab, t, r)
        out.append(table[s:e].contiguous() if e > s else None)
    return out


@pytest.mark.parametrize("i", range(16))
def test_vocab_embed_random(i):
    t, vocab, h, n, s = _vocab_case(i)
    dtype = torch.bfloat16 if i % 2 == 0 else torch.float32
    table = synth.normal_f32((vocab, h), 1.0, s, device=DEV).to(dtype)
    ids = (synth.uniform_ids(n, vocab + 6, s + 1, device=DEV) - 3).to(torch.int32)   # some ids out of range
    parts = [torch.empty((n, h), dtype=dtype, device=DEV) for _ in range(t)]
    out = tp.vocab_parallel_embed(ids, _vocab_shards(table, vocab, t), vocab, partials=parts)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    ref, refp = O.vocab_parallel_embedding(ids.cpu().numpy(), f64(table), t)
    assert np.array_equal(f64(out), ref), (t, vocab, h, n)
    for r in range(t):
        assert np.array_equal(f64(parts[r]), refp[r]), (t, vocab, h, n, r)


@pytest.mark.parametrize("i", range(12))
def test_lm_head_and_gather_random(i):
    t, vocab, h, n, s = _vocab_case(100 + i)   # ragged vocab: shards start mid-line in the logits
    x = ints((n, h), s)
    table = ints((vocab, h), s + 1)
    shards = _vocab_shards(table, vocab, t)
    logits = tp.lm_head_sharded(x, shards, vocab, out_dtype=torch.float32)
    per_shard = tp.lm_head_sharded(x, shards, vocab, per_shard=True, out_dtype=torch.float32)
    gathered = tp.tp_shard_gather([p for p in per_shard if p.shape[1] > 0])
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    ref = O.linear(f64(x), f64(table))
    assert np.array_equal(f64(logits), ref), (t, vocab, h, n)
    assert np.array_equal(f64(gathered), ref), (t, vocab, h, n)


@pytest.mark.parametrize("i", range(16))
def test_shard_reduce_random(i):
    """Random counts (odd, below one vector, across ring-chunk boundaries), shard counts,
    dtypes, orders, wire dtypes and replication, against the oracle's emulation of the
    same fold order (message-passing ring for RING)."""
    rnd = random.Random(7000 + i)
    t = rnd.choice([1, 2, 3, 4, 5, 7, 8])
    count = rnd.choice([1, 3, 7, 8, 9, 63, 1000, 4099, 65537, 200003])
    dtype = rnd.choice([torch.bfloat16, torch.float32])
    mode = rnd.choice(["direct", "ring"])
    hop = torch.bfloat16 if (mode == "ring" and dtype == torch.bfloat16 and rnd.random() < 0.5) else torch.float32
    replicate = rnd.random() < 0.3
    out_dtype = torch.float32 if rnd.random() < 0.5 else dtype
    parts = [synth.normal_f32((count,), 1.0, 7100 + 10 * i + r, device=DEV).to(dtype) for r in range(t)]
    pf = [f64(p) for p in parts]
    out = tp.tp_shard_reduce(parts, mode=mode, hop_dtype=hop, replicate=replicate, out_dtype=out_dtype,
                             alloc_out=not replicate)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    if mode == "direct":
        ref = O.reduce_direct_f32(pf)
    else:
        ref = O.ring_allreduce(pf, hop="bf16" if hop == torch.bfloat16 else "f32")[0][0]
    case = (t, count, dtype, mode, hop, replicate, out_dtype)
    if out is not None:
        want = O.round_to_bf16(ref) if out_dtype == torch.bfloat16 else ref
        assert np.array_equal(f64(out), want), case
    if replicate:
        want = O.round_to_bf16(ref) if dtype == torch.bfloat16 else ref
        for r in range(t):
            assert np.array_equal(f64(parts[r]), want), (case, r)
