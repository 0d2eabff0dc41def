"""Helpers shared by the GPU parity tests: move bit patterns from the CUDA
path's tensors into the oracle's float64 arrays, and the tolerance gates.

Tolerances (derived from the arithmetic):
* A bf16-in / fp32-accumulate GEMM output: max |err| <= 1e-2 * RMS(Y_oracle),
  plus half a bf16 ulp of |Y_oracle| per element when the output is stored
  in bf16 (the final rounding alone can reach that).
* The two-GEMM MLP stores its intermediate H in bf16 and, unless fused, its
  partials in the partial dtype; each rounding adds at most half an ulp of
  the rounded value, which propagates through the down projection as
  sum_f |W_down[j, f]| * ulp(H[i, f]) / 2 and as sum_r ulp(P_r[i, j]) / 2.
  The MLP gate adds these per-element bounds (computed from the oracle's own
  H and partials) to the GEMM gate above.
* fp32 shard reduce vs the fp64 sum: |err| <= 1e-6 * max|Y| (the rank-order
  float32 fold of <= 8 terms is within (t-1) * 2^-24 * sum|P_r|); vs the
  oracle's float32 emulation of the same order: bit-exact.
"""

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


def mlp_rounding_allowance(xf, wg, wu, wd, t, act, partial_bf16):
    """Per-element bound of the bf16 roundings inside the sharded MLP
    (intermediate H, partials), from the oracle's own values."""
    fs = wg.shape[0] // t
    extra = 0.0
    parts = []
    for r in range(t):
        blk = O.merged_column_shard([wg, wu], t, r)
        h = O.glu(O.linear(xf, blk[:fs]), O.linear(xf, blk[fs:]), act)
        bd = O.row_shard(wd, t, r)
        extra = extra + half_ulp_bf16(h) @ np.abs(bd).T
        parts.append(O.linear(h, bd))
    if partial_bf16:
        for p in parts:
            extra = extra + half_ulp_bf16(p)
    return extra
