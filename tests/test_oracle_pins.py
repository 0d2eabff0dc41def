"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: values
printed on the pages (tests/golden, each file citing its passage), closed
forms and identities, library routines (torch, scipy) for special cases, and
brute force with Python integers on tiny inputs.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# --------------------------------------------------------------- shard layouts

def test_column_split_worked_example(golden_dir):
    g = _golden(golden_dir, "nanovllm22_column_split.json")
    w = np.repeat(np.arange(g["w_full_rows"], dtype=np.float64)[:, None], g["w_full_cols"], axis=1)
    x = np.random.default_rng(0).standard_normal((g["x_tokens"], g["w_full_cols"]))
    for r in range(g["t"]):
        shard = O.column_shard(w, g["t"], r)
        assert list(shard.shape) == g["shard_shape"]
        assert shard[:, 0].tolist() == g["rank_rows_first_column"][r]
        assert list(O.linear(x, shard).shape) == g["rank_output_shape"]


def test_row_split_worked_example(golden_dir):
    g = _golden(golden_dir, "nanovllm22_row_split.json")
    w = np.array(g["w_full"], np.float64)
    b = np.array(g["bias"], np.float64)
    x = np.array(g["x"], np.float64)
    t = g["t"]
    parts = []
    for r in range(t):
        wr = O.row_shard(w, t, r)
        assert wr.tolist() == g["rank_weights"][r]
        xr = O.row_shard(x, t, r)          # the input is cut on the same dimension
        parts.append(O.linear(xr, wr, b if r == 0 else None))
        assert parts[-1].tolist() == g["rank_partials"][r]
    assert O.reduce_direct(parts).tolist() == g["sum"]
    assert O.linear(x, w, b).tolist() == g["single_device"]


def test_merged_qkv_and_gate_up_worked_example(golden_dir):
    g = _golden(golden_dir, "nanovllm22_merged_split.json")
    hs, hid, t = g["head_size"], g["hidden"], g["t"]

    def by_head(nheads, base):
        return np.array([[float(base + h)] * hid for h in range(nheads) for _ in range(hs)])

    q, k, v = by_head(g["q_heads"], g["q_base"]), by_head(g["kv_heads"], g["k_base"]), by_head(g["kv_heads"], g["v_base"])
    for r in range(t):
        blk = O.qkv_shard(q, k, v, g["q_heads"], g["kv_heads"], hs, t, r)
        assert blk.shape == (8, hid)
        assert blk[0:4, 0].tolist() == g["rank_q_first_column"][r]
        assert blk[4:6, 0].tolist() == g["rank_k_first_column"][r]
        assert blk[6:8, 0].tolist() == g["rank_v_first_column"][r]
    f = g["gate_up_intermediate"]
    gate = np.full((f, hid), g["gate_fill"])
    up = np.full((f, hid), g["up_fill"])
    blk = O.merged_column_shard([gate, up], t, 0)
    assert blk[:2, 0].tolist() == g["rank0_gate_segment_first_column"]
    assert blk[2:4, 0].tolist() == g["rank0_up_segment_first_column"]


def test_merged_gate_up_is_double_cut_not_contiguous():
    # Rows tagged by their index: rank r must get gate rows [r f/t, (r+1) f/t)
    # followed by the SAME rows of up, not a contiguous slice of [gate; up].
    f, h, t = 8, 2, 4
    gate = np.arange(f, dtype=np.float64)[:, None].repeat(h, 1)
    up = 100 + np.arange(f, dtype=np.float64)[:, None].repeat(h, 1)
    for r in range(t):
        blk = O.merged_column_shard([gate, up], t, r)
        assert blk[:, 0].tolist() == [2 * r, 2 * r + 1, 100 + 2 * r, 100 + 2 * r + 1]


def test_divide_rejects_uneven_split():
    with pytest.raises(ValueError):
        O.column_shard(np.zeros((6, 2)), 4, 0)
    with pytest.raises(ValueError):
        O.row_shard(np.zeros((2, 6)), 4, 0)


@pytest.mark.parametrize("vocab,t,expected", [
    (10, 2, [(0, 5), (5, 10)]),
    (10, 3, [(0, 4), (4, 8), (8, 10)]),
    (10, 4, [(0, 3), (3, 6), (6, 9), (9, 10)]),
    (3, 4, [(0, 1), (1, 2), (2, 3), (3, 3)]),
    (151936, 4, [(0, 37984), (37984, 75968), (75968, 113952), (113952, 151936)]),
])
def test_vocab_range_ceil_rule(vocab, t, expected):
    assert [O.vocab_range(vocab, t, r) for r in range(t)] == expected


# ----------------------------------------------------------- number formats

def test_round_to_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    x32 = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),     # subnormal region
        np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, 1e-45], np.float32),
    ])
    ours = O.bf16_from_f64_bits(O.round_to_bf16(x32.astype(np.float64)))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_round_to_bf16_ties_and_specials():
    one = 1.0
    assert O.round_to_bf16(np.array([one + 2 ** -8]))[0] == 1.0                 # tie -> even
    assert O.round_to_bf16(np.array([one + 3 * 2 ** -8]))[0] == 1.0 + 2 ** -6   # tie -> even (up)
    assert O.round_to_bf16(np.array([one + 2 ** -8 + 2 ** -30]))[0] == 1.0 + 2 ** -7
    assert np.isinf(O.round_to_bf16(np.array([2.0 ** 128]))[0])
    assert np.isnan(O.round_to_bf16(np.array([np.nan]))[0])
    assert O.round_to_bf16(np.array([2.0 ** -140]))[0] == 0.0      # below half the subnormal quantum
    assert O.round_to_bf16(np.array([3 * 2.0 ** -134]))[0] == 2.0 ** -132


def test_bf16_bits_roundtrip():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_bits_to_f64(bits)
    finite = ~np.isnan(vals)
    assert np.array_equal(O.bf16_from_f64_bits(vals[finite]), bits[finite])


# ------------------------------------------------------------- activations

def test_silu_matches_library_and_identities():
    x = np.linspace(-40, 40, 4001)
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    assert np.allclose(O.silu(x), ref, rtol=1e-14, atol=1e-300)
    assert np.allclose(O.silu(x) - O.silu(-x), x, rtol=1e-14, atol=1e-14)
    assert O.silu(np.array([0.0]))[0] == 0.0


def test_gelu_tanh_matches_library_and_identities():
    x = np.linspace(-12, 12, 2401)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(O.gelu_tanh(x), ref, rtol=1e-13, atol=1e-15)
    assert np.allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, rtol=1e-13, atol=1e-13)


# -------------------------------------------------------------------- MLP

def _int_mats(rng, *shapes):
    return [rng.integers(-3, 4, size=s).astype(np.float64) for s in shapes]


def _brute_linear(x, w, b=None):
    n, k = len(x), len(x[0])
    out = []
    for i in range(n):
        row = []
        for j in range(len(w)):
            acc = sum(x[i][p] * w[j][p] for p in range(k))
            if b is not None:
                acc += b[j]
            row.append(acc)
        out.append(row)
    return out


def _brute_silu(v):
    return v / (1.0 + math.exp(-v)) if v >= 0 else v * math.exp(v) / (1.0 + math.exp(v))


@pytest.mark.parametrize("t", [1, 2, 3, 4])
def test_brute_force_linear_layers_integers(t):
    rng = np.random.default_rng(10 + t)
    for n, h in itertools.product([1, 3], [4 * t, 8 * t if t < 3 else 6 * t]):
        out = 2 * t
        x, w, b = _int_mats(rng, (n, h), (out, h), (out,))
        xi = x.astype(int).tolist()
        full = np.array(_brute_linear(xi, w.astype(int).tolist(), b.astype(int).tolist()), np.float64)
        # column parallel: shard outputs concatenated == full, exactly
        cols = [O.linear(x, O.column_shard(w, t, r), O.column_shard(b, t, r)) for r in range(t)]
        assert np.array_equal(O.shard_gather(cols), full)
        # row parallel: partials (bias on rank 0) summed == full, exactly
        parts = [O.linear(O.row_shard(x, t, r), O.row_shard(w, t, r), b if r == 0 else None) for r in range(t)]
        assert np.array_equal(O.reduce_direct(parts), full)
        ring, _ = O.ring_allreduce(parts, hop="f64")
        for buf in ring:
            assert np.array_equal(buf, full)


@pytest.mark.parametrize("t", [1, 2, 3, 4])
def test_brute_force_mlp_small(t):
    rng = np.random.default_rng(20 + t)
    n, h, f = 3, 5, 2 * t
    x, wg, wu, wd, b = _int_mats(rng, (n, h), (f, h), (f, h), (h, f), (h,))
    # Plain loops: g, u, silu(g) * u, then the down projection.
    g = _brute_linear(x.tolist(), wg.tolist())
    u = _brute_linear(x.tolist(), wu.tolist())
    hmid = [[_brute_silu(g[i][j]) * u[i][j] for j in range(f)] for i in range(n)]
    y = np.array(_brute_linear(hmid, wd.tolist(), b.tolist()))
    for order in ("direct", "ring"):
        ys = O.mlp_sharded(x, wg, wu, wd, t, bias=b, act="silu", order=order)
        assert np.allclose(ys, y, rtol=1e-12, atol=1e-12)
    assert np.allclose(O.mlp_unsharded(x, wg, wu, wd, b, "silu"), y, rtol=1e-12, atol=1e-12)


def test_sharded_mlp_equals_unsharded_float():
    rng = np.random.default_rng(3)
    n, h, f = 8, 64, 96
    x = rng.standard_normal((n, h))
    wg, wu, wd = (rng.standard_normal(s) * 0.1 for s in [(f, h), (f, h), (h, f)])
    ref = O.mlp_unsharded(x, wg, wu, wd, None, "silu")
    for t in (1, 2, 4, 8):
        for act in ("silu", "gelu_tanh"):
            y = O.mlp_sharded(x, wg, wu, wd, t, act=act)
            assert np.allclose(y, O.mlp_unsharded(x, wg, wu, wd, None, act), rtol=1e-12, atol=1e-12)
    assert np.abs(ref).max() > 0.1


# The MLP with H rounded to bf16 and the partials rounded to their dtype, on a
# case worked by hand.  t = 2, one token, h = 1, f = 2: x = 1, gate rows
# (1.5, -1), up rows (3, 7), down row (1.1875, 0.5).
#   rank 0: H = silu(1.5) * 3 = 3.679085...   -> bf16 3.671875 (spacing 2^-6 in [2, 4));
#           rounding silu(1.5) first would give 3.6875.
#           P = 3.671875 * 1.1875 = 4.3603515625 (exact in fp32) -> bf16 4.375 (spacing 2^-5)
#   rank 1: H = silu(-1) * 7 = -1.882589...   -> bf16 -1.8828125 (spacing 2^-7);
#           rounding silu(-1) first would give -1.890625.
#           P = -1.8828125 * 0.5 = -0.94140625 (a bf16 value)
#   bf16 partials, rank-order sum:       4.375 - 0.94140625        = 3.43359375
#   bf16 ring hop (t = 2: one rounding): bf16(3.43359375)          = 3.4375 (spacing 2^-6)
#   fp32 partials, or no partials:       4.3603515625 - 0.94140625 = 3.4189453125
#   unrounded definition:                3.4276186323648...
# With a bias of 2^-6 on rank 0, added before the partial is rounded:
#   P0 = 4.3759765625 -> bf16 4.375 (adding the bias after rounding would give
#   4.390625 and Y = 3.44921875), so Y = 3.43359375; fp32: Y = 3.4345703125.
_WORKED = dict(x=np.array([[1.0]]), wg=np.array([[1.5], [-1.0]]), wu=np.array([[3.0], [7.0]]),
               wd=np.array([[1.1875, 0.5]]))


def test_mlp_rounded_worked_example():
    x, wg, wu, wd = _WORKED["x"], _WORKED["wg"], _WORKED["wu"], _WORKED["wd"]
    e = O.mlp_sharded_rounded(x, wg, wu, wd, 2, None, "silu", "bf16", "direct")
    assert [h.item() for h in e["h"]] == [3.671875, -1.8828125]
    assert [p.item() for p in e["p"]] == [4.375, -0.94140625]
    assert [p.item() for p in e["p_exact"]] == [4.3603515625, -0.94140625]
    assert e["y"].item() == 3.43359375
    assert O.mlp_sharded_rounded(x, wg, wu, wd, 2, None, "silu", "bf16", "ring")["y"].item() == 3.4375
    for pd, order in (("f32", "direct"), ("f32", "ring"), (None, "direct")):
        assert O.mlp_sharded_rounded(x, wg, wu, wd, 2, None, "silu", pd, order)["y"].item() == 3.4189453125
    assert abs(O.mlp_unsharded(x, wg, wu, wd, None, "silu").item() - 3.4276186323648) < 1e-12
    b = np.array([2.0 ** -6])
    assert O.mlp_sharded_rounded(x, wg, wu, wd, 2, b, "silu", "bf16", "direct")["y"].item() == 3.43359375
    assert O.mlp_sharded_rounded(x, wg, wu, wd, 2, b, "silu", "f32", "direct")["y"].item() == 3.4345703125
    assert O.mlp_sharded_rounded(x, wg, wu, wd, 2, b, "silu", None, "direct")["y"].item() == 3.4345703125


def test_mlp_rounded_within_the_rounding_bounds():
    """On random inputs every rounding the function takes stays within half a
    spacing of the value it rounds: the result differs from the unrounded
    definition by at most sum_f |W_down[j, f]| * spacing(H[i, f]) / 2 (plus
    half a spacing per bf16 partial), and the H rounding does change it."""
    rng = np.random.default_rng(11)
    n, h, f, t = 6, 48, 64, 4
    bf = lambda a: O.round_to_bf16(a)
    x = bf(rng.standard_normal((n, h)))
    wg, wu, wd = (bf(rng.standard_normal(s) * 0.1) for s in [(f, h), (f, h), (h, f)])

    def half_spacing(v):
        _, e = np.frexp(np.maximum(np.abs(v), 2.0 ** -126))
        return np.ldexp(1.0, e.astype(np.int64) - 9)

    ref = O.mlp_unsharded(x, wg, wu, wd, None, "silu")
    fused = O.mlp_sharded_rounded(x, wg, wu, wd, t, None, "silu", None)
    hbound = sum(half_spacing(fused["h_exact"][r]) @ np.abs(O.row_shard(wd, t, r)).T for r in range(t))
    assert np.all(np.abs(fused["y"] - ref) <= hbound * (1 + 1e-12))
    assert np.any(fused["y"] != ref)
    for r in range(t):
        assert np.all(np.abs(fused["h"][r] - fused["h_exact"][r]) <= half_spacing(fused["h_exact"][r]))
    wire = O.mlp_sharded_rounded(x, wg, wu, wd, t, None, "silu", "bf16")
    pbound = sum(half_spacing(p) for p in wire["p_exact"])
    assert np.all(np.abs(wire["y"] - fused["y"]) <= pbound * (1 + 1e-12))
    assert np.any(wire["y"] != fused["y"])
    for r in range(t):                         # partials are bf16 values
        O.bf16_from_f64_bits(wire["p"][r])


def test_round_to_f32_matches_torch():
    rng = np.random.default_rng(12)
    v = np.concatenate([rng.standard_normal(1000) * 10.0 ** rng.integers(-30, 30, 1000),
                        [1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, -(1.0 + 2.0 ** -24), 0.0, -0.0]])
    ours = O.round_to_f32(v)
    lib = torch.tensor(v, dtype=torch.float64).to(torch.float32).to(torch.float64).numpy()
    assert np.array_equal(ours, lib)
    assert ours[-5] == 1.0 and ours[-4] == 1.0 + 2.0 ** -22      # ties to even


def test_bias_counted_once():
    rng = np.random.default_rng(4)
    x, wg, wu, wd = _int_mats(rng, (2, 8), (8, 8), (8, 8), (8, 8))
    b = np.full(8, 7.0)
    parts = O.mlp_shard_partials(x, wg, wu, wd, 4, bias=b)
    nob = O.mlp_shard_partials(x, wg, wu, wd, 4, bias=None)
    assert np.allclose(parts[0] - nob[0], 7.0)
    for p, q in zip(parts[1:], nob[1:]):
        assert np.array_equal(p, q)


def test_activation_before_reduce_is_wrong():
    # vLLM source analysis 13, section 2.2.2: GeLU(X1A1 + X2A2) != GeLU(X1A1) + GeLU(X2A2),
    # so a row split of the FIRST matmul would need the reduce before the activation.
    rng = np.random.default_rng(42)
    x = rng.standard_normal((4, 8))
    a = rng.standard_normal((8, 4))
    right = O.gelu_tanh(x @ a)
    p1, p2 = x[:, :4] @ a[:4], x[:, 4:] @ a[4:]
    assert np.allclose(O.gelu_tanh(p1 + p2), right, rtol=1e-12, atol=1e-12)
    assert np.abs(O.gelu_tanh(p1) + O.gelu_tanh(p2) - right).max() > 0.1


# -------------------------------------------------------------------- ring

def test_ring_step_counts_and_volume(golden_dir):
    g = _golden(golden_dir, "vllm13_ring_costs.json")
    for case in g["cases"]:
        n = case["n"]
        sched = O.ring_schedule(n)
        rs = {s for (ph, s, *_r) in sched if ph == "reduce_scatter"}
        ag = {s for (ph, s, *_r) in sched if ph == "all_gather"}
        assert len(rs) == case["reduce_scatter_steps"] and len(ag) == case["all_gather_steps"]
        k = 6 * n * 5
        parts = [np.full(k, float(r + 1)) for r in range(n)]
        _, stats = O.ring_allreduce(parts)
        assert stats["steps"] == case["total_steps"]
        assert stats["sent_per_rank"] == [2 * (n - 1) * k // n] * n
    # every step, every rank sends exactly one chunk to its right neighbour
    for n in (2, 3, 4, 8):
        for (ph, s, src, dst, c) in O.ring_schedule(n):
            assert dst == (src + 1) % n


@pytest.mark.parametrize("n,k", [(2, 10), (3, 10), (4, 16), (4, 13), (8, 64), (8, 5), (5, 3)])
def test_ring_ownership_and_all_gather(n, k):
    rng = np.random.default_rng(n * 100 + k)
    parts = [rng.integers(-50, 50, k).astype(np.float64) for _ in range(n)]
    total = sum(parts)
    bufs, stats = O.ring_allreduce(parts)
    chunks = stats["chunks"]
    after = stats["after_reduce_scatter"]
    owners = {}
    for r in range(n):
        c = (r + 1) % n
        lo, hi = chunks[c]
        assert np.array_equal(after[r][lo:hi], total[lo:hi])      # rank r finished chunk r+1
        owners.setdefault(c, []).append(r)
    assert sorted(owners) == list(range(n)) and all(len(v) == 1 for v in owners.values())
    for b in bufs:
        assert np.array_equal(b, total)
    assert sum(hi - lo for lo, hi in chunks) == k


def test_ring_fold_order_visible_in_bf16():
    # With bfloat16 hops the order of additions shows in the result:
    # (1 + 2^-8) rounds to 1 (tie to even), while 2^-8 + 2^-8 = 2^-7 is exact.
    # N=3, one element per chunk.  Following the schedule by hand:
    # chunk c is folded as P_c, then P_{c+1}, then P_{c+2} (mod 3).
    a, e = 1.0, 2.0 ** -8
    p = [np.array([a, e, e]), np.array([e, a, e]), np.array([e, e, a])]
    bufs, _ = O.ring_allreduce(p, hop="bf16")
    # chunk 0: (P0=1 + P1=e) -> 1 ; + P2=e -> 1
    # chunk 1: (P1=a + P2=e) -> 1 ; + P0=e -> 1
    # chunk 2: (P2=a + P0=e) -> 1 ; + P1=e -> 1
    assert bufs[0].tolist() == [1.0, 1.0, 1.0]
    # Now put the large value at the LAST rank of each chunk's fold: rank
    # (c + 2) mod 3 holds a at element c.  The two small values meet first
    # (e + e = 2^-7, exact) and 1 + 2^-7 is a bfloat16 number, so every chunk
    # gives 1 + 2^-7.  A rank-order fold (0, 1, 2) would give 1 for
    # chunks 1 and 2, and a ring turning the other way would give 1 for all.
    q = [np.array([e, a, e]), np.array([e, e, a]), np.array([a, e, e])]
    bufs, _ = O.ring_allreduce(q, hop="bf16")
    for b in bufs:
        assert b.tolist() == [1.0 + 2 ** -7] * 3
    direct = O.round_to_bf16(O.round_to_bf16(q[0] + q[1]) + q[2])
    assert direct.tolist() == [1.0 + 2 ** -7, 1.0, 1.0]
    assert O.ring_fold_order(3, 1) == [1, 2, 0]
    assert O.ring_fold_order(4, 3) == [3, 0, 1, 2]


def test_reduce_f32_matches_torch_sequential_sum():
    rng = np.random.default_rng(5)
    parts = [(rng.standard_normal(5000) * 10.0 ** rng.integers(-3, 4)).astype(np.float32) for _ in range(8)]
    acc = torch.from_numpy(parts[0].copy())
    for p in parts[1:]:
        acc = acc + torch.from_numpy(p)
    ours = O.reduce_direct_f32([p.astype(np.float64) for p in parts])
    assert np.array_equal(ours, acc.numpy().astype(np.float64))
    # ring with f32 hops: chunk c folded from rank c, so it differs from the
    # direct order on some elements, but every element equals a float32 fold
    bufs, _ = O.ring_allreduce([p.astype(np.float64) for p in parts], hop="f32")
    chunks = O.ring_chunks(5000, 8)
    for c, (lo, hi) in enumerate(chunks):
        order = O.ring_fold_order(8, c)
        acc = torch.from_numpy(parts[order[0]][lo:hi].copy())
        for r in order[1:]:
            acc = acc + torch.from_numpy(parts[r][lo:hi])
        assert np.array_equal(bufs[0][lo:hi], acc.numpy().astype(np.float64))


# -------------------------------------------------------------- embedding

def test_embedding_worked_example_structure(golden_dir):
    g = _golden(golden_dir, "vllm13_embedding_example.json")
    rng = np.random.default_rng(42)
    table = rng.standard_normal((g["vocab"], g["hidden"]))
    ids = np.array(g["ids"])
    total, parts = O.vocab_parallel_embedding(ids, table, g["t"])
    assert [list(O.vocab_range(g["vocab"], g["t"], r)) for r in range(g["t"])] == g["ranges"]
    for i in range(ids.shape[0]):
        for j in range(ids.shape[1]):
            nz = [r for r in range(g["t"]) if np.any(parts[r][i, j] != 0)]
            assert nz == [g["owner_rank"][i][j]]
    assert np.array_equal(total, table[ids])


def test_embedding_out_of_range_and_specials():
    v, h, t = 12, 3, 4
    table = np.arange(v * h, dtype=np.float64).reshape(v, h) + 1
    table[1] = [np.nan, np.inf, -0.0]            # rank 0 row with specials
    ids = np.array([-1, 12, 1000, 5, 1, 11, -7])
    total, parts = O.vocab_parallel_embedding(ids, table, t)
    for k in (0, 1, 2, 6):
        assert np.all(total[k] == 0.0) and not np.any(np.signbit(total[k]))
    assert np.array_equal(total[3], table[5]) and np.array_equal(total[5], table[11])
    assert np.isnan(total[4, 0]) and total[4, 1] == np.inf
    assert total[4, 2] == 0.0 and not np.signbit(total[4, 2])     # -0 + (+0) = +0 (t > 1)
    # specials of rank 0's row never leak into other ranks' tokens
    assert np.all(np.isfinite(total[[3, 5]]))
    single, _ = O.vocab_parallel_embedding(np.array([1]), table, 1)
    assert np.signbit(single[0, 2])                                # t = 1: the lookup itself


# ---------------------------------------------------------------- LM head

@pytest.mark.parametrize("vocab,t", [(16, 2), (15, 4), (12, 3), (7, 8)])
def test_lm_head_concat_equals_unsharded(vocab, t):
    rng = np.random.default_rng(vocab * t)
    x, table = _int_mats(rng, (5, 6), (vocab, 6))
    logits, parts = O.lm_head_sharded(x, table, t)
    assert logits.shape == (5, vocab)
    assert np.array_equal(logits, np.array(_brute_linear(x.tolist(), table.tolist())))
    assert sum(p.shape[1] for p in parts) == vocab


# ------------------------------------------------------------ cost model

def test_allreduce_cost_table(golden_dir):
    g = _golden(golden_dir, "aiinfra62_allreduce_table.json")
    for row in g["rows"]:
        us = O.allreduce_time(row["bytes"], g["t"], g["bandwidth_bytes_per_s"]) * 1e6
        assert abs(us - row["approx_us"]) <= row["rel_tol"] * row["approx_us"] + 0.005
        assert row["bytes"] == row["tokens"] * 8192 * 2


# ------------------------------------------------------- sequence parallelism

def test_rmsnorm_matches_library_and_closed_forms():
    rng = np.random.default_rng(60)
    x = rng.standard_normal((7, 33)) * 3
    w = rng.standard_normal(33)
    for eps in (0.0, 1e-6, 1e-2):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(w), eps=eps).numpy()
        assert np.allclose(O.rmsnorm(x, w, eps), ref, rtol=1e-13, atol=1e-13)
    # a constant row c normalises to sign(c) * weight (eps = 0)
    c = np.full((2, 5), -2.5)
    assert np.allclose(O.rmsnorm(c, np.arange(1.0, 6.0), 0.0), -np.arange(1.0, 6.0)[None, :].repeat(2, 0))
    # scale invariance for eps = 0
    assert np.allclose(O.rmsnorm(7.0 * x, w, 0.0), O.rmsnorm(x, w, 0.0), rtol=1e-13)


def test_reduce_scatter_ownership_and_volume(golden_dir):
    g = _golden(golden_dir, "tpscratch_sequence_parallel.json")
    for case in g["cases"]:
        n, k = case["n"], case["k"]
        rng = np.random.default_rng(n * k)
        parts = [rng.integers(-20, 20, k).astype(np.float64) for _ in range(n)]
        total = sum(parts)
        bufs, st = O.ring_reduce_scatter(parts)
        assert st["steps"] == n - 1
        assert st["sent_per_rank"] == [case["rs_per_rank"]] * n
        for r, (lo, hi) in enumerate(st["chunks"]):
            assert np.array_equal(bufs[r][lo:hi], total[lo:hi])          # rank r owns chunk r
        _, ar = O.ring_allreduce(parts)
        assert ar["sent_per_rank"] == [case["ar_per_rank"]] * n
        ag = [a - b for a, b in zip(ar["sent_per_rank"], st["sent_per_rank"])]
        assert ag == [case["ag_per_rank"]] * n                            # RS + AG = AR, equal halves
        # all-gather of the owned chunks gives every rank the all-reduce result
        gathered = np.concatenate([bufs[r][lo:hi] for r, (lo, hi) in enumerate(st["chunks"])])
        assert np.array_equal(gathered, total)


def test_reduce_scatter_fold_order_visible_in_bf16():
    # chunk c is folded c+1, c+2, ..., c (mod 3): put 1.0 on rank c (the last
    # one to add) and 2^-8 elsewhere, so every chunk gives 1 + 2^-7 exactly.
    a, e = 1.0, 2.0 ** -8
    p = [np.array([a, e, e]), np.array([e, a, e]), np.array([e, e, a])]
    bufs, _ = O.ring_reduce_scatter(p, hop="bf16")
    for r in range(3):
        assert bufs[r][r] == 1.0 + 2 ** -7
    assert O.reduce_scatter_fold_order(3, 0) == [1, 2, 0]
    assert O.reduce_scatter_fold_order(4, 3) == [0, 1, 2, 3]
    # the all-reduce convention (chunk c starts at rank c) gives 1 for these inputs
    ar, _ = O.ring_allreduce(p, hop="bf16")
    assert ar[0].tolist() == [1.0, 1.0, 1.0]


@pytest.mark.parametrize("t,n", [(1, 5), (2, 8), (3, 10), (4, 9), (8, 3)])
def test_sequence_parallel_equals_allreduce_then_norm(t, n):
    rng = np.random.default_rng(70 + t)
    h = 12
    parts = [rng.standard_normal((n, h)) for _ in range(t)]
    resid = rng.standard_normal((n, h))
    w = rng.standard_normal(h)
    full = resid + O.reduce_direct(parts)
    for order in ("direct", "ring"):
        res, normed, blocks = O.sequence_parallel_residual_norm(parts, resid, w, 1e-6, order)
        assert np.allclose(res, full, rtol=1e-13, atol=1e-13)
        assert np.allclose(normed, O.rmsnorm(full, w, 1e-6), rtol=1e-12, atol=1e-12)
        assert sum(b[0].shape[0] for b in blocks) == n
        assert [b[0].shape[0] for b in blocks] == [hi - lo for lo, hi in O.token_chunks(n, t)]
    res0, _, _ = O.sequence_parallel_residual_norm(parts, None, w, 1e-6)
    assert np.allclose(res0, O.reduce_direct(parts))


# ----------------------------------------------------- GQA KV-head replication

def test_gqa_kv_replication_counts(golden_dir):
    g = _golden(golden_dir, "aiinfra62_gqa_replication.json")
    nh, nkv = g["num_heads"], g["num_kv_heads"]
    for case in g["cases"]:
        t = case["t"]
        held = [O.kv_head_of_rank(nkv, t, r) for r in range(t)]
        assert all(len(hs) == case["kv_heads_per_rank"] for hs in held)
        copies = {h: sum(h in hs for hs in held) for h in range(nkv)}
        assert set(copies.values()) == {case["copies_per_kv_head"]}
        assert sum(len(hs) for hs in held) == case["total_kv_copies"]
        assert all(len(hs) / nkv == case["kv_fraction_per_rank"] for hs in held)
        for r in range(t):
            q_heads = range(r * nh // t, (r + 1) * nh // t)
            assert len(q_heads) == case["q_heads_per_rank"]
            # every query head of the rank attends to a KV head the rank holds (GQA grouping)
            assert all(q // (nh // nkv) in held[r] for q in q_heads)
    q = g["qwen3_0_6b"]
    for t in q["tp_without_replication"]:
        held = [O.kv_head_of_rank(q["num_kv_heads"], t, r) for r in range(t)]
        assert sorted(h for hs in held for h in hs) == list(range(q["num_kv_heads"]))


def test_qkv_shard_gqa_layout():
    hs, hid = 2, 3
    nh, nkv = 8, 2

    def by_head(n, base):
        return np.array([[float(base + h)] * hid for h in range(n) for _ in range(hs)])

    wq, wk, wv = by_head(nh, 0), by_head(nkv, 100), by_head(nkv, 200)
    # t divides the KV heads: same as the plain double cut
    for r in range(2):
        assert np.array_equal(O.qkv_shard_gqa(wq, wk, wv, nh, nkv, hs, 2, r), O.qkv_shard(wq, wk, wv, nh, nkv, hs, 2, r))
    # t = 4 > 2 KV heads: ranks 0,1 hold KV head 0, ranks 2,3 hold KV head 1
    for r in range(4):
        blk = O.qkv_shard_gqa(wq, wk, wv, nh, nkv, hs, 4, r)
        assert blk[:, 0].tolist() == [2 * r, 2 * r, 2 * r + 1, 2 * r + 1] + [100 + r // 2] * 2 + [200 + r // 2] * 2
    with pytest.raises(ValueError):
        O.qkv_shard_gqa(wq, wk, wv, nh, nkv, hs, 3, 0)        # 3 does not divide 8 query heads
