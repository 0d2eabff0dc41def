"""Helpers shared by the GPU parity tests: move bit patterns from the CUDA
path's tensors into the oracle's float64 arrays, and the tolerance gates.

Tolerances (derived from the arithmetic):
* A bf16-in / fp32-accumulate GEMM output: max |err| <= 1e-2 * RMS(Y_oracle),
  plus half a bf16 spacing of |Y_oracle| per element when the output is
  stored in bf16 (the final rounding alone can reach that).
* The two-GEMM MLP (:func:`mlp_check`) passes two gates:
  A. against the oracle that rounds H to bf16 where the GPU stores it
     (``mlp_sharded_rounded``): max |err| <= 3e-3 * RMS(Y) plus one H flip.
     The GPU's fp32 value of H (tensor-core accumulation of G and U, fast
     exponential) is not the exact one, so a small fraction of H values
     round to the other bf16 neighbour of a nearby rounding midpoint
     (:func:`h_flip_check` measures that fraction: at most ~1 % at K=8192).
     Each flip moves an output by |W_down[j, f]| * spacing(H[i, f]).  Many
     small flips add up like a random walk, which the 3e-3 RMS term covers
     at the sizes tested; at small f one flip can exceed it, so the gate
     adds, per element, the largest single flip the row can make
     (max_f spacing(H[i, f]) * max_f |W_down[j, f]|, per shard).
  B. against the plain unrounded definition (``mlp_unsharded``), max |err|
     <= 1e-2 * RMS(Y) (the bf16 rounding of H is part of this budget).
  Each explicit bf16 rounding the path takes after H (a bf16 partial, a
  bf16 ring hop, a bf16 output) adds half a bf16 spacing of the value it
  rounds to both gates: one rounding to nearest moves a value by at most
  that much.
* fp32 shard reduce vs the fp64 sum: |err| <= 1e-6 * max|Y| (the rank-order
  float32 fold of <= 8 terms is within (t-1) * 2^-24 * sum|P_r|); vs the
  oracle's float32 emulation of the same order: bit-exact.
"""

import json
import os

import numpy as np
import torch

import oracle as O
from megatron_tensor_layers_gb300 import synth


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 value of a bf16 or fp32 CUDA/CPU tensor."""
    if t.dtype == torch.bfloat16:
        return O.bf16_bits_to_f64(synth.bits_u16(t))
    if t.dtype == torch.float32:
        return O.f32_bits_to_f64(synth.bits_u32(t))
    raise TypeError(t.dtype)


def half_ulp_bf16(y: np.ndarray) -> np.ndarray:
    """Bound on one bf16 rounding of a value near y: with |y| in
    [2^(e-1), 2^e), bf16 numbers are 2^(e-8) apart, so rounding moves a value
    by at most 2^(e-9); 2^(e-8) also covers a value that crossed into the
    binade above."""
    a = np.abs(y)
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))
    return np.ldexp(1.0, e.astype(np.int64) - 8)


def gemm_gate(y_gpu: np.ndarray, y_ref: np.ndarray, bf16_out: bool, extra=None, rel=1e-2):
    """Assert the GEMM tolerance; returns (max_err, rms)."""
    err = np.abs(y_gpu - y_ref)
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    bound = rel * rms + (half_ulp_bf16(y_ref) if bf16_out else 0.0)
    if extra is not None:
        bound = bound + extra
    bad = err > bound
    if np.any(bad):
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{int(bad.sum())} of {bad.size} elements exceed the tolerance; max err {err.max():.3e}, "
            f"rms {rms:.3e}; first at {idx.tolist()}: gpu {y_gpu[tuple(idx[0])]!r} ref {y_ref[tuple(idx[0])]!r}")
    return float(err.max()) if err.size else 0.0, rms


def exact(y_gpu: np.ndarray, y_ref: np.ndarray):
    """Bit-for-bit equality of two float64 arrays holding the same format
    (NaNs compared as NaN, signed zeros distinguished)."""
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    nan_g, nan_r = np.isnan(y_gpu), np.isnan(y_ref)
    assert np.array_equal(nan_g, nan_r), "NaN positions differ"
    ok = ~nan_g
    same = (y_gpu[ok] == y_ref[ok]) & (np.signbit(y_gpu[ok]) == np.signbit(y_ref[ok]))
    if not np.all(same):
        bad = np.argwhere(~same)[:5]
        raise AssertionError(f"{int((~same).sum())} elements differ; first flat idx {bad.ravel().tolist()}: "
                             f"gpu {y_gpu[ok][~same][:5]} ref {y_ref[ok][~same][:5]}")


def half_spacing_bf16(v: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |v| * (1 + 2^-7): the most one round-to-nearest
    bf16 rounding moves a value within 2^-7 (relative) of v.  Where the GPU
    rounds its own value of a quantity whose exact value the oracle knows,
    the two differ by far less than 2^-7 relative (so this bounds the GPU's
    rounding even where its value crossed into the next binade), except near
    zero, where the difference is a tiny absolute one whose rounding the
    gate's RMS term covers."""
    a = np.abs(v) * (1.0 + 2.0 ** -7)
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))
    return np.ldexp(1.0, e.astype(np.int64) - 9)


def ring_hop_allowance(p_exact, t, row_ids, h, count):
    """Sum, over the hops of the ring fold, of the bf16 rounding bound of each
    running sum, for output rows ``row_ids`` of a buffer of ``count`` elements
    whose rows are ``h`` long (each element's chunk fixes its fold order)."""
    cs = (count + t - 1) // t
    flat = np.asarray(row_ids, np.int64)[:, None] * h + np.arange(h, dtype=np.int64)[None, :]
    chunk = flat // cs
    allow = np.zeros(flat.shape)
    for c in np.unique(chunk):
        m = chunk == c
        order = O.ring_fold_order(t, int(c))
        acc = p_exact[order[0]][m]
        for r in order[1:]:
            acc = acc + p_exact[r][m]
            allow[m] += half_spacing_bf16(acc)
    return allow


MLP_GATE_A = 3e-3      # RMS fraction against the oracle that rounds H to bf16
MLP_GATE_B = 1e-2      # RMS fraction against the unrounded definition


def mlp_check(y_gpu, x, wg, wu, wd, t, act="silu", bias=None, partial="f32", mode="direct", y_bf16=False,
              row_ids=None, n_total=None):
    """Gates A and B of the module docstring for a tensor-parallel MLP output.

    x, wg, wu, wd: float64 arrays holding the exact bf16 values the GPU got
    (x may be a sample of rows: ``row_ids`` are then their indices in the
    full [n_total, h] output, used for the ring's chunk boundaries).
    partial: "bf16" or "f32" partials (ignored when mode == "fused").
    Returns (max err / RMS against the rounding oracle, max err / RMS against
    the unrounded definition).
    """
    n, h = x.shape[0], wd.shape[0]
    emu = O.mlp_sharded_rounded(x, wg, wu, wd, t, bias, act, None)
    ref = O.mlp_unsharded(x, wg, wu, wd, bias, act)
    allow_a = np.zeros((n, h))
    allow_b = np.zeros((n, h))
    for r in range(t):                      # the largest single H flip of each output element
        s_max = 2.0 * half_spacing_bf16(emu["h"][r]).max(axis=1)
        w_max = np.abs(O.row_shard(wd, t, r)).max(axis=1)
        allow_a = np.maximum(allow_a, np.outer(s_max, w_max))
    if partial == "bf16" and mode != "fused":
        for p in emu["p_exact"]:
            allow_a += half_spacing_bf16(p)
        if mode == "ring":
            rows = np.arange(n) if row_ids is None else np.asarray(row_ids)
            allow_a += ring_hop_allowance(emu["p_exact"], t, rows, h, (n if n_total is None else n_total) * h)
        allow_b = allow_b + allow_a
    if y_bf16:
        allow_a = allow_a + half_spacing_bf16(emu["y"])
        allow_b = allow_b + half_spacing_bf16(ref)
    rms_a = float(np.sqrt(np.mean(emu["y"] ** 2)))
    rms_b = float(np.sqrt(np.mean(ref ** 2)))
    _log_parity(y_gpu, emu["y"], ref, allow_a, allow_b, rms_a, rms_b, t, partial, mode, y_bf16)
    ea, _ = gemm_gate(y_gpu, emu["y"], bf16_out=False, extra=allow_a, rel=MLP_GATE_A)
    eb, _ = gemm_gate(y_gpu, ref, bf16_out=False, extra=allow_b, rel=MLP_GATE_B)
    return ea / rms_a, eb / rms_b


def h_flip_check(h_gpu: np.ndarray, h_exact: np.ndarray, max_fraction=0.02):
    """The gated column GEMM's bf16 output against the exact act(G) * U.

    The GPU rounds its own fp32 value of H, which differs slightly from the
    exact one (fp32 tensor-core accumulation of G and U, fast exponential),
    so an element may round to the other bf16 neighbour of a nearby midpoint.
    Checked: every GPU value lies within one bf16 step of the exact value's
    rounding (plus 2^-12 * RMS(H), for values near zero, where the fp32
    error is absolute rather than relative); such one-step flips are rare
    (at most max_fraction of the elements); and among the elements far from
    zero (|H| >= RMS(H) / 64) every flip moves towards the exact value.
    Returns the fraction of elements that differ from the exact rounding."""
    h_rnd = O.round_to_bf16(h_exact)
    diff = h_gpu != h_rnd
    frac = float(diff.mean()) if diff.size else 0.0
    if np.any(diff):
        rms = float(np.sqrt(np.mean(h_exact ** 2)))
        g, e, r = h_gpu[diff], h_exact[diff], h_rnd[diff]
        step = 2.0 * half_spacing_bf16(np.maximum(np.abs(g), np.abs(r)))
        far = np.abs(g - r) > step + 2.0 ** -12 * rms
        assert not np.any(far), (f"{int(far.sum())} H values lie more than one bf16 step from the exact rounding; "
                                 f"first gpu {g[far][:3]} exact {e[far][:3]}")
        big = np.abs(e) >= rms / 64
        wrong_way = big & ((g - r) * (e - r) <= 0)
        assert not np.any(wrong_way), f"{int(wrong_way.sum())} H values moved away from the exact value"
    assert frac <= max_fraction, f"{frac:.3%} of H values differ from the exact rounding"
    path = os.environ.get("TP_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0],
                                "h_flip_fraction": frac, "elements": int(diff.size)}) + "\n")
    return frac


def _log_parity(y_gpu, y_a, y_b, allow_a, allow_b, rms_a, rms_b, t, partial, mode, y_bf16):
    """With TP_PARITY_LOG set, append one JSON line per MLP check: the max
    error against each oracle over RMS, and the same after subtracting each
    element's rounding allowance (the part the RMS term must cover)."""
    path = os.environ.get("TP_PARITY_LOG")
    if not path:
        return
    ea = np.abs(y_gpu - y_a)
    eb = np.abs(y_gpu - y_b)
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], "t": t, "shape": list(y_gpu.shape),
           "partial": partial, "mode": mode, "y_bf16": bool(y_bf16),
           "err_a_rms": float(ea.max() / rms_a), "err_b_rms": float(eb.max() / rms_b),
           "excess_a_rms": float(np.max(ea - allow_a) / rms_a), "excess_b_rms": float(np.max(eb - allow_b) / rms_b)}
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")
