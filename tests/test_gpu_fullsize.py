"""Parity at the full benchmark sizes, on sampled outputs.

The Llama-3.1-70B-shaped MLP (h=8192, f=28672) runs on the GPU exactly as
bench.py times it (t=4 and t=8, n=8192 prefill; n in {1,16,64} decode); the
oracle computes a seeded sample of 32 token rows (first/last rows and both
sides of a 128-row tile boundary included) in fp64 from the same bits, and
the gates of ``gpu_helpers.mlp_check`` apply (2e-3 RMS against the oracle
that rounds H to bf16, 1e-2 RMS against the unrounded definition).  Output
rows depend only on their own input row, so a sample is a complete check of
those rows.  With integer-valued inputs the same GEMM launches (CTA pairs,
the raster bands, the K loop over 8192/7168 columns, bf16 partials, the
fused reduce) are compared bit for bit on rows at both sides of every
256-row tile and raster band.  The shard reduce at its largest size is compared bit
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

from gpu_helpers import exact, f64, gemm_gate, h_flip_check, half_ulp_bf16, mlp_check

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


def _check(y_rows, xs, d, t, **kw):
    hst = d["host"]
    return mlp_check(y_rows, xs, hst["wg"], hst["wu"], hst["wd"], t, **kw)


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
    _check(f64(y[d["rows"]]), d["host"]["x"], d, t, partial="bf16", y_bf16=True, row_ids=d["rows"], n_total=NTOK)
    # the gated column GEMM's H itself: the exact act(G) * U rounded to bf16, up to flips at midpoints
    xs, hst = d["host"]["x"], d["host"]
    for r in range(t):
        blk = O.merged_column_shard([hst["wg"], hst["wu"]], t, r)
        h_exact = O.glu(O.linear(xs, blk[:fs]), O.linear(xs, blk[fs:]), "silu")
        h_flip_check(f64(hs[r][d["rows"]]), h_exact)


@pytest.mark.parametrize("mode,pdt", [("fused", torch.float32), ("ring", torch.float32), ("ring", torch.bfloat16),
                                      ("direct", torch.float32)])
def test_prefill_mlp_forward_modes(mlp70b, mode, pdt):
    d = mlp70b
    t = 4
    wgu, wds = _shards(d, t)
    y = tp.tp_mlp_forward(d["x"], wgu, wds, mode=mode, partial_dtype=pdt, y_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(f64(y[d["rows"]]), d["host"]["x"], d, t, mode=mode, partial="bf16" if pdt == torch.bfloat16 else "f32",
           row_ids=d["rows"], n_total=NTOK)


@pytest.mark.parametrize("n", [1, 16, 64])
@pytest.mark.parametrize("mode", ["direct", "fused"])
def test_decode_all_rows(mlp70b, n, mode):
    d = mlp70b
    t = 4
    wgu, wds = _shards(d, t)
    x = d["x"][:n].contiguous()
    y = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=torch.float32, y_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(f64(y), f64(x), d, t, mode=mode)


@pytest.mark.parametrize("n", [1, 16, 64])
def test_decode_gated_column_h(mlp70b, n):
    """The decode gate_up GEMM (t=4, 70B shapes) writes, for every token, the exact
    act(G) * U rounded to bf16, up to flips at rounding midpoints."""
    d = mlp70b
    t = 4
    fs = F // t
    wgu, _ = _shards(d, t)
    x = d["x"][:n].contiguous()
    hs = tp.tp_linear_col(x, wgu, act="silu")
    torch.cuda.synchronize()
    xs, hst = f64(x), d["host"]
    for r in range(t):
        blk = O.merged_column_shard([hst["wg"], hst["wu"]], t, r)
        h_flip_check(f64(hs[r]), O.glu(O.linear(xs, blk[:fs]), O.linear(xs, blk[fs:]), "silu"))


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
    _check(f64(y[rows]), f64(x[rows]), d, t)


# ------------------------------------------- integer-exact at the bench's shapes

# rows at both sides of every 256-row pair tile (the raster bands of the bench's
# GEMMs hold 16 or 18 such tiles, so their edges are among these), plus the ends
TILE_EDGE_ROWS = sorted({0, NTOK - 1} | {e for k in range(1, NTOK // 256) for e in (256 * k - 1, 256 * k)})


@pytest.fixture(scope="module")
def int70b():
    build()
    tp.load()
    d = {"x": synth.int_valued((NTOK, H), -3, 3, 20, device=DEV),
         "wg": synth.int_valued((F, H), -3, 3, 21, device=DEV),
         "wu": synth.int_valued((F, H), -3, 3, 22, device=DEV),
         "wd": synth.int_valued((H, F), -3, 3, 23, device=DEV),
         "h": synth.int_valued((NTOK, F), -3, 3, 24, device=DEV),     # stands in for the activation H
         "bias": synth.int_valued((H,), -8, 8, 25, device=DEV)}
    yield d
    d.clear()
    torch.cuda.empty_cache()


def _ring_fold_bf16(pf, t, row_ids, count):
    """Ring fold of sampled rows with every hop rounded to bf16: each element is
    folded in the order of its chunk of the full [NTOK, H] buffer."""
    cs = (count + t - 1) // t
    flat = np.asarray(row_ids, np.int64)[:, None] * H + np.arange(H, dtype=np.int64)[None, :]
    chunk = flat // cs
    out = np.empty(flat.shape)
    for c in np.unique(chunk):
        m = chunk == c
        order = O.ring_fold_order(t, int(c))
        acc = pf[order[0]][m]
        for r in order[1:]:
            acc = O.round_to_bf16(acc + pf[r][m])
        out[m] = acc
    return out


@pytest.mark.parametrize("t", [4, 8])
def test_bench_gemms_integer_exact(int70b, t):
    """The bench's GEMM launches at full size with integer-valued (-3..3) inputs,
    whose every sum is an integer below 2^24 and so exact in fp32 whatever the
    order: the column GEMM over the merged gate_up blocks (K = 8192; |acc| <=
    73728), the row GEMM of each shard into bf16 partials through strided views
    of one [n, f] activation buffer (K = f/t; |P| <= 64512, rounded once to
    bf16 ties-to-even), their rank-order reduce, the ring reduce with bf16
    hops, and the fused down GEMM + reduce with the bias (|Y| <= 258048 + 8).
    Every output row listed in TILE_EDGE_ROWS is compared bit for bit."""
    d = int70b
    fs = F // t
    rows = TILE_EDGE_ROWS
    wgu = [torch.cat([d["wg"][r * fs:(r + 1) * fs], d["wu"][r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [d["wd"][:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    hs = [d["h"][:, r * fs:(r + 1) * fs] for r in range(t)]
    xs = f64(d["x"][rows])
    # column GEMM, fp32 out
    ys = tp.tp_linear_col(d["x"], wgu, act="none", y_dtype=torch.float32)
    torch.cuda.synchronize()
    for r in range(t):
        exact(f64(ys[r][rows]), O.linear(xs, f64(wgu[r])))
    del ys
    # row GEMM into bf16 partials, then the direct and ring (bf16 hops) reduces
    parts = tp.tp_linear_row(hs, wds, bias=d["bias"], reduce_results=False, partial_dtype=torch.bfloat16)
    y_direct = tp.tp_shard_reduce(parts, mode="direct")
    y_ring = tp.tp_shard_reduce(parts, mode="ring", hop_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    hrows = [f64(h[rows]) for h in hs]
    bias = f64(d["bias"])
    p_exact = [O.linear(hrows[r], f64(wds[r]), bias if r == 0 else None) for r in range(t)]
    p_bf16 = [O.round_to_bf16(p) for p in p_exact]
    for r in range(t):
        exact(f64(parts[r][rows]), p_bf16[r])
    exact(f64(y_direct[rows]), O.round_to_bf16(O.reduce_direct(p_bf16)))
    exact(f64(y_ring[rows]), _ring_fold_bf16(p_bf16, t, rows, NTOK * H))
    del parts, y_direct, y_ring
    # fused down GEMM + reduce (one accumulator over all t shards), fp32 out
    y_fused = tp.tp_linear_row(hs, wds, bias=d["bias"], mode="fused", y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    exact(f64(y_fused[rows]), O.reduce_direct(p_exact))
    # the same with scratch for the stream-K tail (the last partial wave's tiles split along K)
    scratch = torch.empty((NTOK, H), dtype=torch.bfloat16, device=DEV)
    y_sk = tp.tp_linear_row(hs, wds, bias=d["bias"], mode="fused", y_dtype=torch.float32, partials=[scratch] * t)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    exact(f64(y_sk[rows]), O.reduce_direct(p_exact))
    assert torch.equal(y_sk, y_fused)


def test_fused_stream_k_tail_bf16_out_and_graph_replay(int70b):
    """The stream-K tail through tp_mlp_forward's own workspace (flags zeroed by the
    call, ahead of its gate_up GEMM), with a bias and a bf16 output: captured once in a
    CUDA graph and replayed on new inputs, every replay gives the eager call's bits,
    and the graph with the minimal workspace (no tail split) stays within the MLP gates."""
    d = int70b
    t, n = 4, 768
    fs = F // t
    wgu = [torch.cat([d["wg"][r * fs:(r + 1) * fs], d["wu"][r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [d["wd"][:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    bias = synth.normal_bf16((H,), 1.0, 26, device=DEV)
    x = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(tp.tp_mlp_workspace_size(t, n, H, F, "fused", torch.bfloat16), dtype=torch.uint8, device=DEV)
    y = torch.empty((n, H), dtype=torch.bfloat16, device=DEV)
    x.copy_(synth.normal_bf16((n, H), 1.0, 27, device=DEV))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tp.tp_mlp_forward(x, wgu, wds, bias_down=bias, mode="fused", workspace=ws, y=y)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tp.tp_mlp_forward(x, wgu, wds, bias_down=bias, mode="fused", workspace=ws, y=y)
    for seed in (28, 29, 30):
        x.copy_(synth.normal_bf16((n, H), 1.0, seed, device=DEV))
        g.replay()
        torch.cuda.synchronize()
        from_graph = y.clone()
        eager = tp.tp_mlp_forward(x, wgu, wds, bias_down=bias, mode="fused")
        torch.cuda.synchronize()
        assert tp.tp_device_status() == 0
        assert torch.equal(from_graph, eager)
    rows = [0, 255, 256, 511, 512, n - 1]
    small_ws = torch.empty(n * F * 2, dtype=torch.uint8, device=DEV)            # H only: no tail split
    y_small = tp.tp_mlp_forward(x, wgu, wds, bias_down=bias, mode="fused", workspace=small_ws, y_dtype=torch.float32)
    torch.cuda.synchronize()
    wg, wu, wd = f64(d["wg"]), f64(d["wu"]), f64(d["wd"])
    for got, y_bf16 in ((f64(from_graph[rows]), True), (f64(y_small[rows]), False)):
        mlp_check(got, f64(x[rows]), wg, wu, wd, t, bias=f64(bias), mode="fused", y_bf16=y_bf16)


@pytest.mark.parametrize("t,n", [(4, 1280), (8, 1280), (2, 1100)])
def test_fused_stream_k_tail_integer_exact(int70b, t, n):
    """The fused down GEMM + reduce at sizes whose last wave of 256 x 256 tiles is
    short (5 row tiles by 32 column tiles, the last ragged at 1100 rows), given a
    contiguous fp32 partial buffer as scratch (n x 8192 x 4 bytes >= 32 MiB + 4 KiB):
    the tail tiles are split along K over the idle CTA pairs, the later parts park
    fp32 partials in the scratch and the first part adds them.  Integer inputs keep
    every sum exact, so the result must equal the oracle's in every row, with and
    without the split."""
    d = int70b
    fs = F // t
    wds = [d["wd"][:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    hs = [d["h"][:n, r * fs:(r + 1) * fs] for r in range(t)]
    scratch = torch.full((n, H), float("nan"), dtype=torch.float32, device=DEV)
    y_sk = tp.tp_linear_row(hs, wds, bias=d["bias"], mode="fused", y_dtype=torch.float32, partials=[scratch] * t)
    y_plain = tp.tp_linear_row(hs, wds, bias=d["bias"], mode="fused", y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    assert torch.equal(y_sk, y_plain)
    rows = sorted({0, 255, 256, n // 2, n - 257, n - 256, n - 1})
    bias = f64(d["bias"])
    ref = O.reduce_direct([O.linear(f64(hs[r][rows]), f64(wds[r]), bias if r == 0 else None) for r in range(t)])
    exact(f64(y_sk[rows]), ref)


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



# (t, n, out, K per shard): fused row GEMMs that take CTA pairs with 256 x 256 tiles and
# leave a short last wave on the 76 resident pairs, drawn by a seeded search over t 2..8,
# n 600..4096, out 8192..16384 and K a multiple of 8 (ragged last K blocks included).  The
# tail tiles split into 2 (36-tile tails), 3 (24) and 4 (4, 8, 16) K parts.
STREAM_K_SHAPES = [(7, 3962, 16384, 1976), (8, 3779, 12288, 344), (7, 3142, 8192, 680), (3, 3130, 8192, 576),
                   (7, 3824, 8192, 736), (3, 3590, 8192, 1568),
                   (2, 4002, 12288, 1856), (3, 2981, 8192, 1752), (8, 2974, 8192, 288), (2, 2481, 8192, 776)]


@pytest.mark.parametrize("t,n,o,k", STREAM_K_SHAPES)
def test_fused_stream_k_tail_shapes(t, n, o, k):
    """Integer inputs: the fused GEMM with the stream-K tail (given a contiguous fp32
    scratch of n x out x 4 >= 32 MiB + 4 KiB) equals the one without it in every element,
    and the oracle on rows at both ends and both sides of a 256-row tile edge."""
    assert tp.tp_debug_gemm_plan(n, o, k, segs=t)[:2] == ("pair", 256)
    x = [synth.int_valued((n, k), -3, 3, 800 + r, device=DEV) for r in range(t)]
    w = [synth.int_valued((o, k), -3, 3, 820 + r, device=DEV) for r in range(t)]
    scratch = torch.full((n, o), float("nan"), dtype=torch.float32, device=DEV)
    y_sk = tp.tp_linear_row(x, w, mode="fused", y_dtype=torch.float32, partials=[scratch] * t)
    y_plain = tp.tp_linear_row(x, w, mode="fused", y_dtype=torch.float32)
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    assert torch.equal(y_sk, y_plain)
    rows = sorted({0, 255, 256, n // 2, n - 257, n - 256, n - 1})
    ref = O.reduce_direct([O.linear(f64(x[r][rows]), f64(w[r])) for r in range(t)])
    exact(f64(y_sk[rows]), ref)


def _integer_mlp(t, n, h, f, seed):
    """Inputs whose every intermediate is an exact small integer: x in {1, 2}, each gate row
    sums 16 entries of x (G in [16, 32], where act(G) rounds back to G in bf16), each up row
    takes 4 entries with signs (|U| <= 8), so H = G U is an integer of at most 256; W_down
    and the bias are integers in -3..3 and -8..8, and every sum stays below 2^24."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(1, 3, (n, h), generator=g).double()
    rows = torch.arange(f)[:, None]
    wg = torch.zeros((f, h), dtype=torch.float64)
    wg[rows, torch.randint(0, h // 16, (f, 1), generator=g) + torch.arange(16)[None, :] * (h // 16)] = 1.0
    wu = torch.zeros((f, h), dtype=torch.float64)
    wu[rows, torch.randint(0, h // 4, (f, 1), generator=g) + torch.arange(4)[None, :] * (h // 4)] = \
        (torch.randint(0, 2, (f, 4), generator=g) * 2 - 1).double()
    wd = torch.randint(-3, 4, (h, f), generator=g).double()
    bias = torch.randint(-8, 9, (h,), generator=g).double()
    return x, wg, wu, wd, bias


@pytest.mark.parametrize("t,n,h,f", [(4, 200, 8192, 8192), (2, 129, 4096, 8192), (8, 256, 8192, 16384),
                                     (4, 256, 6144, 8192), (4, 160, 2048, 4096), (2, 255, 1024, 4096)])
def test_fused_stream_k_few_tiles_integer_exact(t, n, h, f):
    """A fused MLP of 129 to 256 tokens: its down GEMM has one 256-row tile by h/256 column
    tiles, fewer than the resident CTA pairs.  With the workspace's stream-K area every tile
    is split along K into S = pairs / tiles parts (at most 4: 2 for 32 tiles, 3 for 24, 4 for
    16 and fewer), one pair each; without it each tile runs whole.  Integer inputs keep
    every intermediate exact, so both must equal the oracle in every element."""
    assert tp.tp_debug_gemm_plan(n, h, f // t, segs=t)[:2] == ("pair", 256)
    x, wg, wu, wd, bias = _integer_mlp(t, n, h, f, 3000 + n + t)
    ref = O.mlp_sharded_rounded(x.numpy(), wg.numpy(), wu.numpy(), wd.numpy(), t, bias.numpy(), "silu", None)
    assert all(np.array_equal(hr, np.round(hr)) for hr in ref["h"])
    assert np.abs(ref["y"]).max() < 2 ** 24
    fs = f // t
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).to(torch.bfloat16).to(DEV).contiguous()
           for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].to(torch.bfloat16).to(DEV).contiguous() for r in range(t)]
    xd, bd = x.to(torch.bfloat16).to(DEV), bias.to(torch.bfloat16).to(DEV)
    full = tp.tp_mlp_workspace_size(t, n, h, f, "fused")
    base = -(-n * f * 2 // 256) * 256                   # H alone: no stream-K area
    assert full == base + 32 * 1024 * 1024 + 4096
    outs = []
    for size in (full, base):
        ws = torch.full((size,), 0xAB, dtype=torch.uint8, device=DEV)
        outs.append(tp.tp_mlp_forward(xd, wgu, wds, bias_down=bd, mode="fused", workspace=ws,
                                      y_dtype=torch.float32))
    torch.cuda.synchronize()
    assert tp.tp_device_status() == 0
    assert torch.equal(outs[0], outs[1])
    exact(f64(outs[0]), ref["y"])
