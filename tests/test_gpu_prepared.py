"""Prepared calls (``prepare``) on the GPU: each entry point prepared once and
called again after new contents were written into the same input buffers gives
bit for bit what the entry point itself gives on those inputs (every kernel is
deterministic), including from a CUDA graph captured on the prepared stream."""

import pytest
import torch

from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    tp.load()
    torch.cuda.init()
    yield
    assert tp.tp_device_status() == 0


def _fill(ts, seed, std=1.0):
    for i, t in enumerate(ts):
        t.copy_(synth.normal_bf16(tuple(t.shape), std, seed * 100 + i, device=DEV).to(t.dtype))


def _same(a, b):
    if isinstance(a, (list, tuple)):
        assert len(a) == len(b)
        for u, v in zip(a, b):
            _same(u, v)
    elif a is None:
        assert b is None
    else:
        assert a.dtype == b.dtype and torch.equal(a, b)


def _check(plan, inputs, direct, std=1.0):
    """Twice: new input contents, the prepared call, the entry point itself."""
    for seed in (1, 2):
        _fill(inputs, seed, std)
        got = plan()
        want = direct()
        torch.cuda.synchronize()
        _same(got, want)
    assert tp.tp_device_status() == 0


def _mlp(t, n, h, f, seed=7):
    fs = f // t
    x = synth.normal_bf16((n, h), 1.0, seed, device=DEV)
    wgu = [synth.normal_bf16((2 * fs, h), 0.02, seed + 1 + r, device=DEV) for r in range(t)]
    wd = [synth.normal_bf16((h, fs), 0.02, seed + 20 + r, device=DEV) for r in range(t)]
    return x, wgu, wd


@pytest.mark.parametrize("mode,dt", [("direct", torch.bfloat16), ("ring", torch.float32)])
def test_prepared_shard_reduce(mode, dt):
    parts = [torch.empty(8192 * 3 + 5, dtype=dt, device=DEV) for _ in range(4)]
    out = torch.empty_like(parts[0])
    plan = tp.prepare(tp.tp_shard_reduce, parts, out=out, mode=mode)
    _check(plan, parts, lambda: tp.tp_shard_reduce(parts, mode=mode))


@pytest.mark.parametrize("gather", [False, True])
def test_prepared_linear_col(gather):
    x, wgu, _ = _mlp(2, 40, 512, 2048)
    plan = tp.prepare(tp.tp_linear_col, x, wgu, act="silu", gather_output=gather)
    _check(plan, [x], lambda: tp.tp_linear_col(x, wgu, act="silu", gather_output=gather))


@pytest.mark.parametrize("mode", ["direct", "fused"])
def test_prepared_linear_row(mode):
    t, n, k, o = 4, 300, 256, 1024
    x = [synth.normal_bf16((n, k), 1.0, 40 + r, device=DEV) for r in range(t)]
    w = [synth.normal_bf16((o, k), 0.02, 50 + r, device=DEV) for r in range(t)]
    bias = synth.normal_bf16((o,), 0.1, 60, device=DEV)
    plan = tp.prepare(tp.tp_linear_row, x, w, bias=bias, mode=mode, y_dtype=torch.float32)
    _check(plan, x, lambda: tp.tp_linear_row(x, w, bias=bias, mode=mode, y_dtype=torch.float32))


@pytest.mark.parametrize("n,mode", [(1, "direct"), (8, "fused"), (64, "ring"), (200, "fused")])
def test_prepared_mlp_forward(n, mode):
    """n = 8 fused takes the one-kernel path (h = 1024), the others the two GEMMs."""
    x, wgu, wd = _mlp(2, n, 1024, 3072)
    plan = tp.prepare(tp.tp_mlp_forward, x, wgu, wd, mode=mode, y_dtype=torch.float32)
    _check(plan, [x], lambda: tp.tp_mlp_forward(x, wgu, wd, mode=mode, y_dtype=torch.float32))


def test_prepared_mlp_forward_static():
    x, wgu, wd = _mlp(2, 16, 1024, 3072)
    plan = tp.prepare(tp.tp_mlp_forward_static, x, wgu, wd, mode="fused")
    _check(plan, [x], lambda: tp.tp_mlp_forward(x, wgu, wd, mode="fused"))


def test_prepared_mlp_forward_host():
    t, n, h, f = 2, 520, 1024, 3072
    _, wgu, wd = _mlp(t, n, h, f)

    def buffers():
        return {"y_host": torch.empty((n, h), dtype=torch.float32).pin_memory(),
                "x_dev": torch.empty((n, h), dtype=torch.bfloat16, device=DEV),
                "y_dev": torch.empty((n, h), dtype=torch.float32, device=DEV),
                "workspace": torch.empty(tp.tp_mlp_host_workspace_size(t, n, h, f, 2), dtype=torch.uint8,
                                         device=DEV)}

    x_host = torch.empty((n, h), dtype=torch.bfloat16).pin_memory()
    mine = buffers()
    plan = tp.prepare(tp.tp_mlp_forward_host, x_host, wgu, wd, chunks=2, **mine)
    for seed in (1, 2):
        x_host.copy_(synth.normal_bf16((n, h), 1.0, seed, device="cpu"))
        got = plan()
        torch.cuda.current_stream().synchronize()
        want = tp.tp_mlp_forward_host(x_host, wgu, wd, chunks=2, **buffers())
        torch.cuda.current_stream().synchronize()
        assert got is mine["y_host"] and torch.equal(got, want)


def test_prepared_embedding_and_lm_head():
    t, vocab, h, n = 4, 5003, 256, 97
    per = (vocab + t - 1) // t
    table = [synth.normal_bf16((min((r + 1) * per, vocab) - r * per, h), 1.0, 80 + r, device=DEV) for r in range(t)]
    ids = synth.uniform_ids(n, vocab, 90, device=DEV)
    plan = tp.prepare(tp.vocab_parallel_embed, ids, table, vocab)
    for seed in (1, 2):
        ids.copy_(synth.uniform_ids(n, vocab, 90 + seed, device=DEV))
        got = plan()
        want = tp.vocab_parallel_embed(ids, table, vocab)
        torch.cuda.synchronize()
        _same(got, want)
    x = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    for per_shard in (False, True):
        plan = tp.prepare(tp.lm_head_sharded, x, table, vocab, per_shard=per_shard, out_dtype=torch.float32)
        _check(plan, [x], lambda: tp.lm_head_sharded(x, table, vocab, per_shard=per_shard, out_dtype=torch.float32))


def test_prepared_gather_and_reduce_scatter_rmsnorm():
    shards = [torch.empty((33, c), dtype=torch.bfloat16, device=DEV) for c in (8, 24, 16)]
    plan = tp.prepare(tp.tp_shard_gather, shards)
    _check(plan, shards, lambda: tp.tp_shard_gather(shards))
    t, n, h = 4, 64, 1024
    parts = [torch.empty((n, h), dtype=torch.float32, device=DEV) for _ in range(t)]
    weight = synth.normal_bf16((h,), 1.0, 95, device=DEV)
    residual = torch.empty((n, h), dtype=torch.bfloat16, device=DEV)
    res_out = torch.empty_like(residual)
    plan = tp.prepare(tp.tp_reduce_scatter_rmsnorm, parts, weight, residual=residual, residual_out=res_out)
    _check(plan, parts + [residual],
           lambda: tp.tp_reduce_scatter_rmsnorm(parts, weight, residual=residual,
                                                residual_out=torch.empty_like(residual)))


def test_prepared_call_in_a_cuda_graph():
    """Prepared on a side stream, warmed up there, captured on it and replayed:
    the replay follows new contents of the input buffer."""
    x, wgu, wd = _mlp(2, 8, 1024, 3072)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    plan = tp.prepare(tp.tp_mlp_forward, x, wgu, wd, mode="direct", stream=s)
    with torch.cuda.stream(s):
        plan()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan()
    for seed in (1, 2):
        _fill([x], seed)
        g.replay()
        want = tp.tp_mlp_forward(x, wgu, wd, mode="direct")
        torch.cuda.synchronize()
        assert torch.equal(plan.result, want)
