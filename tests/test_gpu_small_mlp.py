"""The MLP of one to eight tokens in one GEMM kernel (CTA pairs over 64-column
slices of the ranks' f columns) plus an ordered reduce of the slices' fp32
partials: tp_mlp_forward takes this path for a fused reduce when the shape
allows it and the workspace holds the partials.

Checks: bit-exact results on inputs whose every intermediate is exact
(integer X, gate rows with 16 ones so that every G lies in [16, 32] and
act(G) rounds back to G in bf16, up rows with four entries of +-1, integer
W_down: H = G * U is an integer of at most 256 and every sum of Y stays below
2^24); the MLP gates against the oracle on normal inputs for both
activations, bf16 and fp32 outputs, with and without bias; agreement with the
two-GEMM path (a workspace holding H only); no write outside Y or outside the
partials' bytes of the workspace.  Reference: "6.2 Tensor-parallel inference"
section 1 (Y = sum_i act(X A_i) B_i, one all-reduce).
"""

import numpy as np
import pytest
import torch

import oracle.tp_oracle as O
from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth

from gpu_helpers import exact, f64, half_spacing_bf16, mlp_check

pytestmark = pytest.mark.gpu
DEV = "cuda"

# (t, n, h, f): the tiny TP-MLP, one slice, three ranks of three slices, the most slices
# (128), h = 768 (three down tiles per CTA), and every token count
SHAPES = [(2, 8, 1024, 3072), (1, 1, 256, 64), (3, 5, 512, 576), (8, 8, 1024, 8192), (4, 7, 768, 1024),
          (2, 2, 256, 512), (2, 3, 512, 1024), (4, 4, 1024, 2048), (2, 6, 256, 256)]


def _integer_mlp(t, n, h, f, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(1, 3, (n, h), generator=g).double()
    wg = torch.zeros((f, h), dtype=torch.float64)
    wu = torch.zeros((f, h), dtype=torch.float64)
    for row in range(f):
        wg[row, torch.randperm(h, generator=g)[:16]] = 1.0
        cols = torch.randperm(h, generator=g)[:4]
        wu[row, cols] = (torch.randint(0, 2, (4,), generator=g) * 2 - 1).double()
    wd = torch.randint(-3, 4, (h, f), generator=g).double()
    bias = torch.randint(-8, 9, (h,), generator=g).double()
    return x, wg, wu, wd, bias


def _shards(wg, wu, wd, t):
    f = wg.shape[0]
    fs = f // t
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).to(torch.bfloat16).to(DEV).contiguous()
           for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].to(torch.bfloat16).to(DEV).contiguous() for r in range(t)]
    return wgu, wds


def _small_ws(t, n, h, f):
    need = tp.tp_mlp_workspace_size(t, n, h, f, "fused", torch.bfloat16)
    assert need == (f // 64) * n * h * 4 + (-(f // 64) * n * h * 4) % 256, "shape should take the one-kernel path"
    return need


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("t,n,h,f", SHAPES)
def test_small_mlp_integer_exact(t, n, h, f, act):
    x, wg, wu, wd, bias = _integer_mlp(t, n, h, f, 1000 + n + t)
    ref = O.mlp_sharded_rounded(x.numpy(), wg.numpy(), wu.numpy(), wd.numpy(), t, bias.numpy(), act, None)
    assert np.array_equal(ref["h"][0], np.round(ref["h"][0]))        # the construction keeps H integral
    assert np.abs(ref["y"]).max() < 2 ** 24
    wgu, wds = _shards(wg, wu, wd, t)
    xd = x.to(torch.bfloat16).to(DEV)
    bd = bias.to(torch.bfloat16).to(DEV)
    ws = torch.empty(_small_ws(t, n, h, f), dtype=torch.uint8, device=DEV)
    y = tp.tp_mlp_forward(xd, wgu, wds, bias_down=bd, act=act, mode="fused", workspace=ws, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    exact(f64(y), ref["y"])


@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
@pytest.mark.parametrize("t,n,h,f", SHAPES)
def test_small_mlp_float_parity(t, n, h, f, act, ydt, bias):
    fs = f // t
    seed = 2000 + 7 * n + t
    x = synth.normal_bf16((n, h), 1.0, seed, device=DEV)
    wg = synth.normal_bf16((f, h), 0.02, seed + 1, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, seed + 2, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, seed + 3, device=DEV)
    b = synth.normal_bf16((h,), 0.5, seed + 4, device=DEV) if bias else None
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    y = tp.tp_mlp_forward(x, wgu, wds, bias_down=b, act=act, mode="fused", y_dtype=ydt)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    mlp_check(f64(y), f64(x), f64(wg), f64(wu), f64(wd), t, act=act, bias=None if b is None else f64(b),
              mode="fused", y_bf16=ydt == torch.bfloat16)


@pytest.mark.parametrize("t,n,h,f", [(2, 8, 1024, 3072), (3, 5, 512, 576), (8, 8, 1024, 8192)])
def test_small_mlp_agrees_with_the_two_gemm_path(t, n, h, f):
    """A workspace that holds H only selects the two-GEMM path; both results pass
    the gates.  They differ by the order of the fp32 sums and, where an H value
    lies next to a bf16 rounding midpoint, by that H rounding the other way:
    the two-GEMM path starts each tile's K loop at a rotated block, so its G
    and U carry other fp32 rounding.  Such H values are rare (a fraction of a
    percent at most), but each moves every output of its token: an element may
    differ by up to four H steps times the largest W_down weight of its row,
    plus the sum order."""
    fs = f // t
    x = synth.normal_bf16((n, h), 1.0, 77, device=DEV)
    wg = synth.normal_bf16((f, h), 0.02, 78, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, 79, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, 80, device=DEV)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    h_only = (n * f * 2 + 255) // 256 * 256
    assert h_only < _small_ws(t, n, h, f)
    ws_small = torch.empty(_small_ws(t, n, h, f), dtype=torch.uint8, device=DEV)
    ws_two = torch.empty(h_only, dtype=torch.uint8, device=DEV)
    y1 = tp.tp_mlp_forward(x, wgu, wds, mode="fused", workspace=ws_small, y_dtype=torch.float32)
    y2 = tp.tp_mlp_forward(x, wgu, wds, mode="fused", workspace=ws_two, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    for y in (y1, y2):
        mlp_check(f64(y), f64(x), f64(wg), f64(wu), f64(wd), t, mode="fused")
    wgf, wuf, wdf = f64(wg), f64(wu), f64(wd)
    emu = O.mlp_sharded_rounded(f64(x), wgf, wuf, wdf, t, None, "silu", None)
    allow = np.zeros((n, h))
    for r in range(t):
        step = 2.0 * half_spacing_bf16(emu["h"][r]).max(axis=1)
        allow = np.maximum(allow, np.outer(step, np.abs(O.row_shard(wdf, t, r)).max(axis=1)))
    rms = float(np.sqrt(np.mean(emu["y"] ** 2)))
    diff = np.abs(f64(y1) - f64(y2))
    assert np.all(diff <= 4.0 * allow + 1e-5 * rms), float((diff - 4.0 * allow).max() / rms)


@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_small_mlp_writes_nothing_outside(ydt):
    """Y inside a larger buffer and the workspace inside a larger buffer, both
    filled with a sentinel: only Y's [n, h] and the partials' bytes change."""
    t, n, h, f = 2, 5, 1024, 3072
    fs = f // t
    x = synth.normal_bf16((n, h), 1.0, 91, device=DEV)
    wg = synth.normal_bf16((f, h), 0.02, 92, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, 93, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, 94, device=DEV)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    need = _small_ws(t, n, h, f)
    used = (f // 64) * n * h * 4
    ws_all = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device=DEV)
    ws = ws_all[:need]
    pad = 4096 // (4 if ydt == torch.float32 else 2)
    y_all = torch.full((n * h + 2 * pad,), float("nan"), dtype=ydt, device=DEV)
    y = y_all[pad:pad + n * h].view(n, h)
    tp.tp_mlp_forward(x, wgu, wds, mode="fused", workspace=ws, y=y, y_dtype=ydt)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    assert bool(torch.isnan(y_all[:pad]).all()) and bool(torch.isnan(y_all[pad + n * h:]).all())
    assert not bool(torch.isnan(y).any())
    assert bool((ws_all[used:] == 0xA5).all())
    mlp_check(f64(y), f64(x), f64(wg), f64(wu), f64(wd), t, mode="fused", y_bf16=ydt == torch.bfloat16)


def test_small_mlp_back_to_back_on_one_workspace():
    """Calls queued without a host sync share the partials: the next call's GEMM
    kernel loads nothing before the previous call's reduce has finished."""
    t, n, h, f = 2, 8, 1024, 3072
    fs = f // t
    wg = synth.normal_bf16((f, h), 0.02, 95, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, 96, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, 97, device=DEV)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    ws = torch.empty(_small_ws(t, n, h, f), dtype=torch.uint8, device=DEV)
    xs = [synth.normal_bf16((n, h), 1.0, 100 + i, device=DEV) for i in range(6)]
    ys = [tp.tp_mlp_forward(xi, wgu, wds, mode="fused", workspace=ws, y_dtype=torch.float32) for xi in xs]
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    for xi, yi in zip(xs, ys):
        alone = tp.tp_mlp_forward(xi, wgu, wds, mode="fused", y_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(yi, alone)


@pytest.mark.parametrize("t,n,h,f", [(2, 8, 1024, 3072), (3, 5, 512, 576)])
def test_small_mlp_strided_operands(t, n, h, f):
    """X as a column view of a wider buffer (row stride h + 64) and W_down as column
    slices of the full [h, f] matrix (row stride f): the one-kernel path reads them
    through their strides and gives the contiguous call's bits."""
    fs = f // t
    x_full = synth.normal_bf16((n, h + 64), 1.0, 500, device=DEV)
    x = x_full[:, :h]
    wg = synth.normal_bf16((f, h), 0.02, 501, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, 502, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, 503, device=DEV)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds_view = [wd[:, r * fs:(r + 1) * fs] for r in range(t)]
    wds = [w.contiguous() for w in wds_view]
    ws = torch.empty(_small_ws(t, n, h, f), dtype=torch.uint8, device=DEV)
    y_strided = tp.tp_mlp_forward(x, wgu, wds_view, mode="fused", workspace=ws, y_dtype=torch.float32)
    y_plain = tp.tp_mlp_forward(x.contiguous(), wgu, wds, mode="fused", workspace=ws, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    assert torch.equal(y_strided, y_plain)
    mlp_check(f64(y_plain), f64(x), f64(wg), f64(wu), f64(wd), t, mode="fused")


def _random_shapes(count, seed):
    """Seeded eligible shapes: t in 1..8, n in 1..8, h in {256, 512, 768, 1024}, f/t a multiple
    of 64 with at most 128 slices of 64 columns in all."""
    rnd = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        t = int(rnd.integers(1, 9))
        n = int(rnd.integers(1, 9))
        h = int(rnd.choice([256, 512, 768, 1024]))
        per = int(rnd.integers(1, 128 // t + 1))          # slices per rank
        out.append((t, n, h, 64 * per * t))
    return out


@pytest.mark.parametrize("t,n,h,f", _random_shapes(12, 77))
def test_small_mlp_integer_exact_random_shapes(t, n, h, f):
    act = "silu" if (t + n) % 2 else "gelu_tanh"
    x, wg, wu, wd, bias = _integer_mlp(t, n, h, f, 3000 + 7 * t + n)
    ref = O.mlp_sharded_rounded(x.numpy(), wg.numpy(), wu.numpy(), wd.numpy(), t, bias.numpy(), act, None)
    wgu, wds = _shards(wg, wu, wd, t)
    ws = torch.empty(_small_ws(t, n, h, f), dtype=torch.uint8, device=DEV)
    y = tp.tp_mlp_forward(x.to(torch.bfloat16).to(DEV), wgu, wds, bias_down=bias.to(torch.bfloat16).to(DEV), act=act,
                          mode="fused", workspace=ws, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    exact(f64(y), ref["y"])


def test_small_mlp_smaller_h_first():
    """The kernel's shared memory grows with h; a first call with a small h must not cap
    the shared memory of later calls with a larger one (each shape in a fresh order)."""
    for (t, n, h, f) in [(2, 3, 256, 512), (2, 3, 768, 1536), (2, 3, 1024, 2048), (2, 3, 512, 1024)]:
        fs = f // t
        x = synth.normal_bf16((n, h), 1.0, 600 + h, device=DEV)
        wg = synth.normal_bf16((f, h), 0.02, 601 + h, device=DEV)
        wu = synth.normal_bf16((f, h), 0.02, 602 + h, device=DEV)
        wd = synth.normal_bf16((h, f), 0.02, 603 + h, device=DEV)
        wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
        wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
        y = tp.tp_mlp_forward(x, wgu, wds, mode="fused", y_dtype=torch.float32)
        torch.cuda.synchronize()
        assert tp.tp_device_status() == 0
        mlp_check(f64(y), f64(x), f64(wg), f64(wu), f64(wd), t, mode="fused")
