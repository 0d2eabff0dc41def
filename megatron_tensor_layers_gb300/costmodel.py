"""Analytic cost model of tensor-parallel inference, with measured inputs.

The pages estimate what tensor parallelism costs with two simple models:

* one all-reduce of S bytes over t ranks takes alpha + 2(t-1)/t * S / B
  ("6.2 Tensor-parallel inference", §3.1; "Tensor parallelism from
  scratch", "the cost of communication"), and a transformer layer needs two
  of them (after the attention output projection and after the MLP);
* a decode step is bounded by reading the weights and the KV cache from HBM
  plus that communication ("6.2 Tensor-parallel inference", §7); prefill by
  the GEMM FLOPs at some fraction of peak.

This module restates both models as plain functions (the page prints its
H100 numbers; the tests reproduce them), and adds the same estimates for
the simulated-rank path of this library on one GB300, whose "all-reduce" of
t partials is one HBM pass of (t + 1) * S bytes plus a kernel launch.
Feed it measured numbers (``bench.py`` prints them) to see where the time
goes.  Run ``python -m megatron_tensor_layers_gb300.costmodel`` for the
tables.
"""

from __future__ import annotations

import json
import sys
from dataclasses import dataclass
from typing import Dict, List, Optional


def allreduce_time(size_bytes: float, t: int, link_bytes_per_s: float, alpha_s: float) -> float:
    """alpha + 2 (t-1)/t * S / B: a ring (or bus) all-reduce of S bytes."""
    if t <= 1:
        return 0.0
    return alpha_s + 2.0 * (t - 1) / t * size_bytes / link_bytes_per_s


@dataclass
class DecodeModel:
    """A dense decoder for the decode-step model (weights and KV read once
    per step; two all-reduces of batch x hidden x 2 bytes per layer)."""
    layers: int = 80
    hidden: int = 8192
    weight_bytes: float = 70.6e9 * 2
    kv_bytes_per_token: float = 320 * 1024
    ctx: int = 4096
    kv_rank_limit: int = 8           # the KV cache stops shrinking past the KV head count


def decode_step(model: DecodeModel, t: int, batch: int, hbm_bytes_per_s: float, link_bytes_per_s: float,
                alpha_s: float) -> Dict[str, float]:
    """Seconds of one decode step: weight read + KV read + communication."""
    weight = model.weight_bytes / t / hbm_bytes_per_s
    kv = batch * model.ctx * model.kv_bytes_per_token / min(t, model.kv_rank_limit) / hbm_bytes_per_s
    msg = batch * model.hidden * 2
    comm = 2 * model.layers * allreduce_time(msg, t, link_bytes_per_s, alpha_s) if t > 1 else 0.0
    total = weight + kv + comm
    return {"step_s": total, "comm_s": comm, "tokens_per_s": batch / total, "tokens_per_s_per_gpu": batch / total / t}


def allreduces_per_forward(layers: int) -> int:
    """All-reduces in one forward of a TP transformer: one after each
    layer's attention output projection and one after its MLP, plus one for
    the vocab-parallel embedding (the LM head gathers instead)."""
    return 2 * layers + 1


def comm_per_forward(layers: int, hidden: int, tokens: int, t: int, busbw: float, alpha_s: float) -> float:
    """Seconds of all-reduce in one forward of `tokens` tokens (2 per layer)."""
    return 2 * layers * allreduce_time(tokens * hidden * 2, t, busbw, alpha_s)


def prefill_compute(params: float, tokens: int, t: int, peak_flops: float, mfu: float) -> float:
    """Seconds of 2 * params * tokens FLOP spread over t GPUs at mfu of peak."""
    return 2.0 * params * tokens / (t * peak_flops * mfu)


# -------------------------------------------------------------- this library

def simulated_allreduce_time(size_bytes: float, t: int, hbm_bytes_per_s: float, launch_s: float) -> float:
    """The one-GPU stand-in: a reduce of t partials of S bytes into one
    output reads t*S and writes S bytes of HBM, plus one kernel launch."""
    return launch_s + (t + 1) * size_bytes / hbm_bytes_per_s


def gb300_table(measured: Dict[str, float], tokens: List[int] = (1, 64, 8192), t: int = 4,
                hidden: int = 8192) -> List[Dict[str, float]]:
    """Per-message estimates for the simulated-rank all-reduce on one GB300
    next to the pages' NVLink estimate, from measured HBM bandwidth (bytes/s)
    and launch time (s)."""
    rows = []
    for n in tokens:
        s = n * hidden * 2
        rows.append({"tokens": n, "bytes": s,
                     "nvlink_tp8_us": allreduce_time(s, 8, 450e9, 0.0) * 1e6,
                     "gb300_sim_us": simulated_allreduce_time(s, t, measured["hbm_bytes_per_s"],
                                                              measured["launch_s"]) * 1e6})
    return rows


def _main(argv: Optional[List[str]] = None) -> None:
    argv = sys.argv[1:] if argv is None else argv
    print("Decode step model of '6.2 Tensor-parallel inference' (H100 assumptions):")
    print(f"{'TP':>3} {'batch':>5} {'step ms':>8} {'comm ms':>8} {'tok/s':>8} {'tok/s/GPU':>10}")
    m = DecodeModel()
    for batch in (1, 64):
        for t in (1, 2, 4, 8):
            r = decode_step(m, t, batch, 3.35e12, 450e9, 10e-6)
            print(f"{t:>3} {batch:>5} {r['step_s'] * 1e3:>8.2f} {r['comm_s'] * 1e3:>8.2f} "
                  f"{r['tokens_per_s']:>8.0f} {r['tokens_per_s_per_gpu']:>10.0f}")
    measured = {"hbm_bytes_per_s": 6.5e12, "launch_s": 3e-6}
    if argv:
        with open(argv[0]) as f:
            line = json.loads(f.read().splitlines()[0])
        measured["hbm_bytes_per_s"] = line["shard_reduce"]["value"] * 1e9
        sweep = line.get("detail", {}).get("shard_reduce_sweep", {})
        n1 = sweep.get("bf16_t4_n1_direct", {}).get("graph_us")
        if n1:   # a one-token reduce is all latency: take it as the per-reduce fixed cost
            measured["launch_s"] = n1 * 1e-6
    print("\nOne all-reduce of n tokens x 8192 x 2 bytes: NVLink TP=8 bandwidth term vs this library's")
    print(f"simulated t=4 reduce on one GB300 (one HBM pass at {measured['hbm_bytes_per_s'] / 1e12:.2f} TB/s "
          f"+ {measured['launch_s'] * 1e6:.2f} us fixed):")
    for r in gb300_table(measured):
        print(f"  n={r['tokens']:>5}  {r['bytes'] / 2**20:8.3f} MiB  NVLink {r['nvlink_tp8_us']:9.2f} us   "
              f"GB300 simulated {r['gb300_sim_us']:9.2f} us")


if __name__ == "__main__":
    _main()
