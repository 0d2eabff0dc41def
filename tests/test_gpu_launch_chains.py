"""The kernels of one call run as a chain (gate_up GEMM -> down GEMM -> shard
reduce) in which each later kernel may start before the previous one ends
(programmatic dependent launch) and waits inside the kernel before reading
what that kernel wrote.  These tests check the chain where an ordering bug
would show: replayed from a CUDA graph, back to back without a host sync and
with the workspace reused, and against the CPU oracle.  Every kernel here is
deterministic (fixed fold order, no atomics), so repeated results must be
bit-identical.
"""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

from gpu_helpers import f64, mlp_check

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    tp.load()
    torch.cuda.init()
    yield
    assert tp.tp_device_status() == 0


def _mlp(t, n, h, f, seed):
    fs = f // t
    x = synth.normal_bf16((n, h), 1.0, seed, device=DEV)
    wg = synth.normal_bf16((f, h), 0.02, seed + 1, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, seed + 2, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, seed + 3, device=DEV)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    return x, wg, wu, wd, wgu, wds


def _same_bits(a, b):
    assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("mode", ["direct", "ring", "fused"])
@pytest.mark.parametrize("t,n,h,f", [(2, 8, 1024, 3072), (4, 1, 512, 2048), (4, 200, 512, 2048)])
def test_mlp_graph_replay_bit_identical_to_eager(mode, t, n, h, f):
    x, wg, wu, wd, wgu, wds = _mlp(t, n, h, f, 300)
    ws = torch.empty(max(256, tp.tp_mlp_workspace_size(t, n, h, f, mode, torch.bfloat16)), dtype=torch.uint8,
                     device=DEV)
    y_graph = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tp.tp_mlp_forward(x, wgu, wds, mode=mode, workspace=ws, y=y_graph)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tp.tp_mlp_forward(x, wgu, wds, mode=mode, workspace=ws, y=y_graph)
    for seed in (310, 311, 312):
        x.copy_(synth.normal_bf16((n, h), 1.0, seed, device=DEV))
        y_graph.zero_()
        g.replay()
        y_eager = tp.tp_mlp_forward(x, wgu, wds, mode=mode)
        torch.cuda.synchronize()
        _same_bits(y_graph, y_eager)
    assert tp.tp_device_status() == 0


@pytest.mark.parametrize("mode", ["direct", "fused"])
def test_mlp_back_to_back_calls_share_workspace(mode):
    """Several calls queued without a host sync, one workspace: each call's
    first kernel may start while the previous call's last kernel drains, but
    it loads nothing before that kernel has finished, and it writes H only
    after those loads, so it cannot overwrite H or the partials while the
    previous call's kernels still read them."""
    t, n, h, f = 4, 16, 1024, 4096
    x, wg, wu, wd, wgu, wds = _mlp(t, n, h, f, 320)
    xs = [synth.normal_bf16((n, h), 1.0, 330 + i, device=DEV) for i in range(6)]
    ws = torch.empty(max(256, tp.tp_mlp_workspace_size(t, n, h, f, mode, torch.float32)), dtype=torch.uint8,
                     device=DEV)
    ys = [torch.empty((n, h), dtype=torch.float32, device=DEV) for _ in xs]
    for xi, yi in zip(xs, ys):
        tp.tp_mlp_forward(xi, wgu, wds, mode=mode, partial_dtype=torch.float32, workspace=ws, y=yi,
                          y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    wgf, wuf, wdf = f64(wg), f64(wu), f64(wd)
    for xi, yi in zip(xs, ys):
        mlp_check(f64(yi), f64(xi), wgf, wuf, wdf, t, mode=mode)
        alone = tp.tp_mlp_forward(xi, wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
        torch.cuda.synchronize()
        _same_bits(yi, alone)


def test_row_linear_chain_then_reduce_in_every_order():
    """tp_linear_row with the reduce chained after the GEMM, in both fold
    orders, equals the GEMM's partials reduced by a separate call."""
    t, n, ks, out = 4, 40, 256, 520
    x = [synth.normal_bf16((n, ks), 1.0, 340 + r, device=DEV) for r in range(t)]
    w = [synth.normal_bf16((out, ks), 0.02, 350 + r, device=DEV) for r in range(t)]
    for mode in ("direct", "ring"):
        y = tp.tp_linear_row(x, w, mode=mode, y_dtype=torch.float32, partial_dtype=torch.float32)
        parts = tp.tp_linear_row(x, w, reduce_results=False, partial_dtype=torch.float32)
        y2 = tp.tp_shard_reduce(parts, out_dtype=torch.float32, mode=mode)
        torch.cuda.synchronize()
        _same_bits(y, y2)


def test_inputs_and_weights_written_just_before_a_call():
    """Every call's first kernel may start while the previous kernel of the
    stream drains, so it must not read anything (weights included) before
    waiting for it.  Here a torch kernel rewrites the input or the weights
    immediately before each call, with no host sync in between; every result
    must reflect the data just written."""
    t, n, k, os_ = 2, 24, 512, 384
    x = synth.int_valued((n, k), -3, 3, 360, dtype=torch.bfloat16, device=DEV)
    w = [synth.int_valued((os_, k), -3, 3, 361 + r, dtype=torch.bfloat16, device=DEV) for r in range(t)]
    xs = [synth.int_valued((n, k), -3, 3, 370 + i, dtype=torch.bfloat16, device=DEV) for i in range(3)]
    ws = [[synth.int_valued((os_, k), -3, 3, 380 + 10 * i + r, dtype=torch.bfloat16, device=DEV) for r in range(t)]
          for i in range(3)]
    outs = []
    for i in range(3):
        x.copy_(xs[i])
        for r in range(t):
            w[r].copy_(ws[i][r])
        outs.append([o.clone() for o in tp.tp_linear_col(x, w, y_dtype=torch.float32)])
        # the fused row GEMM (split-K kernel at this size) as the first kernel of a call
        x2 = [xi.contiguous() for xi in torch.chunk(x, t, dim=1)]
        outs[-1].append(tp.tp_linear_row(x2, [wr[:, :k // t].contiguous() for wr in w], mode="fused",
                                         y_dtype=torch.float32).clone())
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    for i in range(3):
        xf = f64(xs[i])
        for r in range(t):
            assert np.array_equal(f64(outs[i][r]), O.linear(xf, f64(ws[i][r])))
        ref = O.reduce_direct([O.linear(f64(xs[i][:, r * (k // t):(r + 1) * (k // t)]),
                                        f64(ws[i][r][:, :k // t])) for r in range(t)])
        assert np.array_equal(f64(outs[i][t]), ref)


def test_event_wait_still_orders_a_programmatic_launch():
    """A call's first kernel may start before the previous kernel of its
    stream ends, but a cross-stream event wait queued between them still
    holds it: here the input arrives behind a 1 GiB host-to-device copy on
    another stream, long after the short GEMM before it has finished, and
    the GEMM after the event wait must see the new input."""
    t, n, k, os_ = 2, 16, 256, 128
    w = [synth.int_valued((os_, k), -3, 3, 390 + r, dtype=torch.bfloat16, device=DEV) for r in range(t)]
    x_old = synth.int_valued((n, k), -3, 3, 393, dtype=torch.bfloat16, device=DEV)
    x_new_host = synth.int_valued((n, k), -3, 3, 394, dtype=torch.bfloat16).pin_memory()
    big_host = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    big_dev = torch.empty(1 << 30, dtype=torch.uint8, device=DEV)
    x = x_old.clone()
    copy = torch.cuda.Stream()
    ev = torch.cuda.Event()
    torch.cuda.synchronize()
    with torch.cuda.stream(copy):
        big_dev.copy_(big_host, non_blocking=True)           # about a millisecond or more
        x.copy_(x_new_host, non_blocking=True)
        ev.record(copy)
    tp.tp_linear_col(x_old, w, y_dtype=torch.float32)       # short kernel, done long before the copy
    torch.cuda.current_stream().wait_event(ev)
    y = tp.tp_linear_col(x, w, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    xf = f64(x_new_host.to(DEV))
    for r in range(t):
        assert np.array_equal(f64(y[r]), O.linear(xf, f64(w[r])))


@pytest.mark.parametrize("mode", ["direct", "ring"])
@pytest.mark.parametrize("t,n,h,f", [(3, 1, 320, 1800), (3, 5, 320, 1800), (2, 12, 512, 2176), (4, 40, 256, 4352),
                                     (4, 1, 8192, 28672), (4, 16, 8192, 28672)])
def test_mlp_forward_equals_its_two_calls(mode, t, n, h, f):
    """tp_mlp_forward's down GEMM loads its first ring of weights before it waits for
    the gate_up GEMM (its predecessor in the call writes only H); a tp_linear_row call
    loads nothing before its wait.  Same kernels and the same order of arithmetic, so
    the MLP equals the gated tp_linear_col followed by tp_linear_row bit for bit.  K of
    the down GEMM is 600 and 1088 (ragged last K blocks), 7168 at the 70B shapes; the
    rings are shorter and longer than a tile's K loop; 1 to 40 rows take the 8-, 16- and
    64-row A tiles."""
    fs = f // t
    x = synth.normal_bf16((n, h), 1.0, 400 + n, device=DEV)
    wgu = [synth.normal_bf16((2 * fs, h), 0.02, 410 + r, device=DEV) for r in range(t)]
    wds = [synth.normal_bf16((h, fs), 0.02, 420 + r, device=DEV) for r in range(t)]
    y1 = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
    hs = tp.tp_linear_col(x, wgu, act="silu")
    y2 = tp.tp_linear_row(hs, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    _same_bits(y1, y2)


def _random_mlp_shapes(count, seed):
    """Seeded shapes for tp_mlp_forward: t 1..8, f/t and h multiples of 8 (h up to 1600),
    token counts across the 8-, 16- and 64-row A tiles, the single-CTA and pair kernels."""
    rnd = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        t = int(rnd.integers(1, 9))
        fs = 8 * int(rnd.integers(1, 150))
        h = 8 * int(rnd.integers(8, 201))
        n = int(rnd.choice([rnd.integers(1, 9), rnd.integers(9, 17), rnd.integers(17, 65), rnd.integers(65, 300)]))
        out.append((t, n, h, fs * t))
    return out


@pytest.mark.parametrize("t,n,h,f", _random_mlp_shapes(16, 2026))
def test_mlp_forward_random_shapes(t, n, h, f):
    """Direct and ring: bit for bit the gated tp_linear_col followed by tp_linear_row.
    Fused: the MLP gates against the oracle."""
    fs = f // t
    x = synth.normal_bf16((n, h), 1.0, 700 + n, device=DEV)
    wgu = [synth.normal_bf16((2 * fs, h), 0.02, 710 + r, device=DEV) for r in range(t)]
    wds = [synth.normal_bf16((h, fs), 0.02, 720 + r, device=DEV) for r in range(t)]
    hs = tp.tp_linear_col(x, wgu, act="silu")
    for mode in ("direct", "ring"):
        y1 = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
        y2 = tp.tp_linear_row(hs, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
        torch.cuda.synchronize()
        _same_bits(y1, y2)
    yf = tp.tp_mlp_forward(x, wgu, wds, mode="fused", y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    wg = torch.cat([w[:fs] for w in wgu])
    wu = torch.cat([w[fs:] for w in wgu])
    wd = torch.cat(wds, dim=1)
    mlp_check(f64(yf), f64(x), f64(wg), f64(wu), f64(wd), t, mode="fused")
