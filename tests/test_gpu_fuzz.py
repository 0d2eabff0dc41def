"""Randomized parity sweep over the GEMM entry points.

Seeded random shapes (shard count, tokens, K, output width, all ragged
against the tiles), output dtypes, gather/bias options, reduce orders and the
kernel-selection knobs (CTA pairs, split-K clusters, tile width) drive the
column and row linears through every GEMM kernel and epilogue.  Inputs are
small integers, so every fp32 result is exact and a bf16 result is the exact
value rounded once: both are compared bit for bit with the CPU oracle.  The
gated column GEMM (SiLU is transcendental) uses the float gate.
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
