"""Parity at the full benchmark sizes, on sampled outputs.

The Llama-3.1-70B-shaped MLP (h=8192, f=28672) runs on the GPU exactly as
bench.py times it (t=4 and t=8, n=8192 prefill; n in {1,16,64} decode); the
oracle computes a seeded sample of 32 token rows (first/last rows and both
sides of a 128-row tile boundary included) in fp64 from the same bits.
Output rows depend only on their own input row, so a sample is a complete
check of those rows.  The shard reduce at its largest size is compared bit
for bit with the oracle's emulation on windows around every ring-chunk
boundary, the LM head at its configured size on sampled rows, and the
attention block's QKV and o_proj projections at the same model's shapes.
"""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

from gpu_helpers import exact, f64, gemm_gate, half_ulp_bf16

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, F, NTOK = 8192, 28672, 8192


@pytest.fixture(scope="module")
def mlp70b():
    build()
    tp.load()
    x = synth.normal_bf16((NTOK, H), 1.0, 0, device=DEV)
    wg = synth.normal_bf16((F, H), 0.02, 1, device=DEV)
    wu = synth.normal_bf16((F, H), 0.02, 2, device=DEV)
    wd = synth.normal_bf16((H, F), 0.02, 3, device=DEV)
    rng = np.random.default_rng(1234)
    rows = sorted(set([0, 127, 128, 255, 256, NTOK - 1] + rng.choice(NTOK, 26, replace=False).tolist()))
    host = {"x": f64(x[rows]), "wg": f64(wg), "wu": f64(wu), "wd": f64(wd)}
    yield {"x": x, "wg": wg, "wu": wu, "wd": wd, "rows": rows, "host": host}
    del x, wg, wu, wd
    torch.cuda.empty_cache()


def _shards(d, t):
    fs = F // t
    wgu = [torch.cat([d["wg"][r * fs:(r + 1) * fs], d["wu"][r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [d["wd"][:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    return wgu, wds


def _reference(xs, hst, t, partial_bf16):
    """fp64 rows of the unsharded MLP and the per-element allowance for the
    bf16 roundings of H (and of the partials)."""
    wg, wu, wd = hst["wg"], hst["wu"], hst["wd"]
    fs = F // t
    ref = O.mlp_unsharded(xs, wg, wu, wd, None, "silu")
    extra = 0.0
    for r in range(t):
        blk = O.merged_column_shard([wg, wu], t, r)
        h = O.glu(O.linear(xs, blk[:fs]), O.linear(xs, blk[fs:]), "silu")
        bd = O.row_shard(wd, t, r)
        extra = extra + half_ulp_bf16(h) @ np.abs(bd).T
        if partial_bf16:
            extra = extra + half_ulp_bf16(O.linear(h, bd))
    return ref, extra


@pytest.mark.parametrize("t", [4, 8])
def test_prefill_bench_launch_sequence(mlp70b, t):
    d = mlp70b
    wgu, wds = _shards(d, t)
    fs = F // t
    hbuf = torch.empty((NTOK, F), dtype=torch.bfloat16, device=DEV)
    hs = [hbuf[:, r * fs:(r + 1) * fs] for r in range(t)]
    parts = [torch.empty((NTOK, H), dtype=torch.bfloat16, device=DEV) for _ in range(t)]
    y = torch.empty((NTOK, H), dtype=torch.bfloat16, device=DEV)
    # the exact calls of one bench step
    tp.tp_linear_col(d["x"], wgu, act="silu", y=hs)
    tp.tp_linear_row(hs, wds, reduce_results=False, partials=parts)
    tp.tp_shard_reduce(parts, out=y, mode="direct")
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    ref, extra = _reference(d["host"]["x"], d["host"], t, partial_bf16=True)
    gemm_gate(f64(y[d["rows"]]), ref, bf16_out=True, extra=extra)


@pytest.mark.parametrize("mode", ["fused", "ring"])
def test_prefill_mlp_forward_modes(mlp70b, mode):
    d = mlp70b
    t = 4
    wgu, wds = _shards(d, t)
    y = tp.tp_mlp_forward(d["x"], wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    ref, extra = _reference(d["host"]["x"], d["host"], t, partial_bf16=False)
    gemm_gate(f64(y[d["rows"]]), ref, bf16_out=False, extra=extra)


@pytest.mark.parametrize("n", [1, 16, 64])
@pytest.mark.parametrize("mode", ["direct", "fused"])
def test_decode_all_rows(mlp70b, n, mode):
    d = mlp70b
    t = 4
    wgu, wds = _shards(d, t)
    x = d["x"][:n].contiguous()
    y = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    ref, extra = _reference(f64(x), d["host"], t, partial_bf16=False)
    gemm_gate(f64(y), ref, bf16_out=False, extra=extra)


@pytest.mark.parametrize("n", [200, 256, 300])
def test_mid_size_all_rows(mlp70b, n):
    """Chunked-prefill sizes between decode and the bench's 8192 tokens, where the
    kernel choice switches between CTA pairs (200, 256: one ragged or full 256-row
    tile) and single CTAs (300)."""
    d = mlp70b
    t = 4
    wgu, wds = _shards(d, t)
    x = d["x"][:n].contiguous()
    y = tp.tp_mlp_forward(x, wgu, wds, mode="direct", partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    rows = [0, 127, 128, n - 1]
    ref, extra = _reference(f64(x[rows]), d["host"], t, partial_bf16=False)
    gemm_gate(f64(y[rows]), ref, bf16_out=False, extra=extra)


@pytest.mark.parametrize("t", [2, 4, 8])
def test_shard_reduce_largest_windows(t):
    count = NTOK * H
    parts = [synth.normal_bf16((count,), 1.0, 700 + r, device=DEV) for r in range(t)]
    outs = {m: tp.tp_shard_reduce(parts, mode=m, out_dtype=torch.float32) for m in ("direct", "ring")}
    wire = tp.tp_shard_reduce(parts, mode="ring", hop_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    cs = (count + t - 1) // t
    starts = sorted(set([0, count - 4096] + [max(0, c * cs - 2048) for c in range(1, t)]))
    for s in starts:
        sl = slice(s, min(count, s + 4096))
        pf = [f64(p[sl]) for p in parts]
        exact(f64(outs["direct"][sl]), O.reduce_direct_f32(pf))
        # ring fold order of each element follows its chunk
        idx = np.arange(sl.start, sl.stop)
        ring_ref = np.empty(idx.size)
        wire_ref = np.empty(idx.size)
        for c in np.unique(idx // cs):
            m = (idx // cs) == c
            order = O.ring_fold_order(t, int(c))
            acc32 = pf[order[0]][m].astype(np.float32)
            accb = pf[order[0]][m]
            for r in order[1:]:
                acc32 = (acc32 + pf[r][m].astype(np.float32)).astype(np.float32)
                accb = O.round_to_bf16(accb + pf[r][m])
            ring_ref[m] = acc32
            wire_ref[m] = accb
        exact(f64(outs["ring"][sl]), ring_ref)
        exact(f64(wire[sl]), wire_ref)


@pytest.mark.parametrize("t", [2, 4])
def test_lm_head_config_sampled_rows(t):
    V, h, n = 151936, 1024, 4096
    x = synth.normal_bf16((n, h), 1.0, 7, device=DEV)
    table = synth.normal_bf16((V, h), 0.02, 6, device=DEV)
    per = (V + t - 1) // t
    shards = [table[r * per:min((r + 1) * per, V)].contiguous() for r in range(t)]
    logits = tp.lm_head_sharded(x, shards, V, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    rows = [0, 127, 128, n - 1] + list(np.random.default_rng(5).choice(n, 12, replace=False))
    ref, _ = O.lm_head_sharded(f64(x[rows]), f64(table), t)
    gemm_gate(f64(logits[rows]), ref, bf16_out=True)


@pytest.mark.parametrize("order", ["direct", "ring"])
def test_reduce_scatter_rmsnorm_bench_size(order):
    t, n, h = 4, 8192, 8192
    parts = [synth.normal_bf16((n, h), 1.0, 800 + r, device=DEV) for r in range(t)]
    resid = synth.normal_bf16((n, h), 1.0, 810, device=DEV)
    w = synth.normal_bf16((h,), 1.0, 811, device=DEV)
    res_out = torch.empty_like(resid)
    _, out = tp.tp_reduce_scatter_rmsnorm(parts, w, residual=resid, mode=order, residual_out=res_out)
    torch.cuda.synchronize()
    rows = [0, 2047, 2048, 4095, 4096, 6143, 6144, n - 1]          # both sides of every rank's boundary
    pf = [f64(p[rows]) for p in parts]
    full_rows = np.array(rows)
    owners = full_rows // ((n + t - 1) // t)
    x = np.zeros((len(rows), h))
    for i, r in enumerate(owners):
        seq = list(range(t)) if order == "direct" else O.reduce_scatter_fold_order(t, int(r))
        x[i] = sum(pf[j][i] for j in seq)
    xr = f64(resid[rows]) + x
    normed = O.rmsnorm(xr, f64(w), 1e-6)
    assert np.all(np.abs(f64(out[rows]) - normed) <= half_ulp_bf16(normed) + 1e-4 * np.abs(normed) + 1e-6)
    assert np.all(np.abs(f64(res_out[rows]) - xr) <= half_ulp_bf16(xr) + 1e-5 * np.abs(xr))


@pytest.mark.parametrize("n", [1, 64, 1024])
def test_attention_projections_70b_t8(n):
    """The attention block's tensor-parallel projections at Llama-3.1-70B shapes (64 query
    heads, 8 KV heads, head size 128, h = 8192) over t = 8: the head-aligned QKV
    column GEMM (each rank: 8 query heads, 1 KV head) and the o_proj row GEMM over the
    ranks' attention outputs with the reduce, on sampled rows.  The attention itself is
    not part of the path: the o_proj input is a seeded stand-in for it."""
    build()
    tp.load()
    t, nh, nkv, hd, h = 8, 64, 8, 128, 8192
    x = synth.normal_bf16((n, h), 1.0, 800, device=DEV)
    wq = synth.normal_bf16((nh * hd, h), 0.02, 801, device=DEV)
    wk = synth.normal_bf16((nkv * hd, h), 0.02, 802, device=DEV)
    wv = synth.normal_bf16((nkv * hd, h), 0.02, 803, device=DEV)
    wo = synth.normal_bf16((h, nh * hd), 0.02, 804, device=DEV)
    qh = nh // t * hd
    blocks = [torch.cat([wq[r * qh:(r + 1) * qh], wk[r * hd:(r + 1) * hd], wv[r * hd:(r + 1) * hd]]).contiguous()
              for r in range(t)]
    qkv = tp.tp_linear_col(x, blocks, y_dtype=torch.float32)
    attn = [synth.normal_bf16((n, qh), 1.0, 810 + r, device=DEV) for r in range(t)]
    wos = [wo[:, r * qh:(r + 1) * qh].contiguous() for r in range(t)]
    y = tp.tp_linear_row(attn, wos, mode="direct", partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    rows = sorted(set([0, n // 2, n - 1]))
    xf = f64(x[rows])
    wqf, wkf, wvf = f64(wq), f64(wk), f64(wv)
    for r in range(t):
        blk = O.qkv_shard(wqf, wkf, wvf, nh, nkv, hd, t, r)
        gemm_gate(f64(qkv[r][rows]), O.linear(xf, blk), bf16_out=False)
    wof = f64(wo)
    parts = [O.linear(f64(attn[r][rows]), O.row_shard(wof, t, r)) for r in range(t)]
    gemm_gate(f64(y[rows]), O.reduce_direct(parts), bf16_out=False)
