"""Benchmark of the tensor-parallel hot path on GB300.

One step = one forward of the Llama-3.1-70B-shaped tensor-parallel MLP
prefill with t = 4 simulated ranks (n = 8192 tokens, h = 8192, f = 28672,
SiLU-gated): per rank the merged gate_up column GEMM with the activation in
its epilogue, per rank the down-projection row GEMM into a bf16 partial, then
the all-reduce of the 4 partials (direct order).  `value` is the MLP's
6*n*h*f FLOP divided by the device time of the step (inputs resident in HBM,
all larger than L2).  The shard reduce inside the same step gives the
second half of the metric (GB/s).  After the timed steps the other rows of
the hot path (fused reduce, t=8, decode, embedding, LM head, the reduce
sweep) are timed once each and reported under "detail".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the pages publish no implementation to run).  Under torchrun
(N > 1) every rank runs an independent replica (weak scaling); rank 0
prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TP-MLP TFLOP/s (% bf16 tensor peak); shard-reduce GB/s (% HBM peak)"
T, N_TOK, H, F = 4, 8192, 8192, 28672
FLOPS = 6.0 * N_TOK * H * F                 # gate + up + down GEMMs
WORKLOAD = ("Llama-3.1-70B-shaped TP-MLP prefill: t=4 simulated ranks, n=8192 tokens, h=8192, f=28672 "
            "(per-rank gate_up [14336,8192], down [8192,7168]), SiLU-gated, bf16 partials reduced in rank order")
E2E_CHUNKS = 2                              # row blocks of the host-buffer entry point
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) of one launch of the gate_up GEMM at the bench
# size, from ncu (dram__bytes_read.sum + dram__bytes_write.sum); None until
# taken for the current kernel.
TRAFFIC_GLU_FULL = 8332345344 + 467087872
TRAFFIC_NOTE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch of the CTA-pair gate_up "
                "GEMM at the bench size (1-pass capture); 5.6x the algorithmic bytes: weights streamed once "
                "per 64 MB raster band of X rows, band rows re-read from DRAM between waves")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running.

    Every sample carries nvidia-smi's timestamp; ``mark_start`` / ``mark_end``
    record the host clock around the timed region, and the summary describes
    only the samples that fall inside it (with how many there were)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None
        self.t0 = None
        self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __enter__(self):
        try:
            self.out = open(os.path.join("/tmp", f"tp_bench_clocks_{os.getpid()}.csv"), "w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        # Wait for the first sample: nvidia-smi's first NVML initialisation on a fresh machine
        # can hold the driver for a while, and must not fall into the timed region.
        t0 = time.time()
        while self.proc is not None and time.time() - t0 < 10.0:
            self.out.flush()
            if os.path.getsize(self.out.name) > 0:
                break
            time.sleep(0.05)
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def _rows(self):
        from datetime import datetime
        self.out.flush()
        self.out.seek(0)
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, smax, power = float(parts[2]), float(parts[3]), float(parts[4])
            except ValueError:
                continue
            active = {nm for nm, v in zip(names, parts[6:10]) if v.lower().startswith("active")}
            rows.append((ts, sm, smax, power, active))
        return rows

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = self._rows()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        sm = [r[1] for r in use]
        reasons = sorted(set().union(*(r[4] for r in use)))
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[2] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_in_timed_region": len(inside),
                "sample_period_ms": self.PERIOD_MS,
                "power_cap_samples_in_timed_region": sum(1 for r in inside if "sw_power_cap" in r[4]),
                "power_w_max": max(r[3] for r in use),
                "basis": ("samples inside the timed region" if inside else
                          "no sample fell inside the timed region: all samples of the run")}


# ------------------------------------------------------------------ ours

def make_mlp(torch, synth, t, n, h, f, dev, seed=0):
    fs = f // t
    x = synth.normal_bf16((n, h), 1.0, seed, device=dev)
    wg = synth.normal_bf16((f, h), 0.02, seed + 1, device=dev)
    wu = synth.normal_bf16((f, h), 0.02, seed + 2, device=dev)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    del wg, wu
    wd = synth.normal_bf16((h, f), 0.02, seed + 3, device=dev)
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    del wd
    return x, wgu, wds


def max_over_ranks(dist, seconds: float, device) -> float:
    """The slowest rank's timed region (all ranks get the same value)."""
    import torch
    tt = torch.tensor([seconds], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units processed by all ranks per second of the slowest rank (weak
    scaling: every rank runs its own replica of the workload)."""
    return units_per_rank * world / max_seconds


def time_fn(torch, fn, iters, warm=2, stream=None, repeats=3):
    """Device time (s) of one fn() call: CUDA events on the stream around
    `iters` back-to-back calls, the median over `repeats` such windows."""
    stream = stream or torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(repeats):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / 1e3 / iters)
    return sorted(times)[len(times) // 2]


def run_ours(args, rank, world, local_rank):
    import torch
    from megatron_tensor_layers_gb300 import _lib as tp
    from megatron_tensor_layers_gb300 import synth
    from megatron_tensor_layers_gb300.build import build

    build()
    tp.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    stream = torch.cuda.current_stream()
    x, wgu, wds = make_mlp(torch, synth, T, N_TOK, H, F, dev, seed=0)
    fs = F // T
    hbuf = torch.empty((N_TOK, F), dtype=torch.bfloat16, device=dev)
    h_slices = [hbuf[:, r * fs:(r + 1) * fs] for r in range(T)]
    parts = [torch.empty((N_TOK, H), dtype=torch.bfloat16, device=dev) for _ in range(T)]
    y = torch.empty((N_TOK, H), dtype=torch.bfloat16, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        tp.tp_linear_col(x, wgu, act="silu", y=h_slices, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        tp.tp_linear_row(h_slices, wds, reduce_results=False, partials=parts, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        tp.tp_shard_reduce(parts, out=y, mode="direct", stream=stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if tp.tp_device_status() != 0:
        raise RuntimeError("device status error after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank if world > 1 else (dev.index or 0)) as clocks:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        clocks.mark_start()
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        if dist is not None:
            dist.barrier()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    if tp.tp_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    col_t = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3 / args.steps
    row_t = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3 / args.steps
    red_t = sum(e[2].elapsed_time(e[3]) for e in evs) / 1e3 / args.steps
    if dist is not None:
        elapsed = max_over_ranks(dist, elapsed, dev)
    ms_per_step = elapsed / args.steps * 1e3
    value = whole_job_value(FLOPS * args.steps, world, elapsed) / 1e12

    col_flops = 4.0 * N_TOK * H * F
    red_bytes = (T + 1) * N_TOK * H * 2
    # The denominator follows the regime the step ran in, as the clock samples
    # taken inside the timed region show it: a region in which some sample saw
    # the power cap is compared with the sustained GEMM peak, which was measured
    # under the same cap; otherwise (no cap seen, or no sample inside a region
    # shorter than the sampling period) with the higher burst peak.
    clk = clocks.summary()
    capped = clk.get("power_cap_samples_in_timed_region", 0) > 0
    tpeak = peaks["bf16_tflops_sustained"] if capped else peaks["bf16_tflops"]
    n_in = clk.get("samples_in_timed_region", 0)
    seen = (f"power cap seen in {clk.get('power_cap_samples_in_timed_region', 0)} of {n_in} clock samples inside the "
            f"{elapsed:.2f} s timed region" if n_in else
            f"no clock sample inside the {elapsed:.2f} s timed region (period {ClockSampler.PERIOD_MS} ms)")
    tkind = f"bf16 {'sustained' if capped else 'burst'} ({peak_src}; {seen})"
    roofline = {"bound": "tensor", "kernel": "tp_gemm_pair_kernel<6,GLU> (gate_up column GEMM + SiLU*up, CTA pairs)",
                "achieved": col_flops / col_t / 1e12, "peak": tpeak, "unit": "TFLOP/s",
                "frac": col_flops / col_t / 1e12 / tpeak, "peak_kind": tkind,
                "frac_of_burst": col_flops / col_t / 1e12 / peaks["bf16_tflops"], "traffic": TRAFFIC_GLU_FULL,
                "traffic_note": TRAFFIC_NOTE, "algorithmic_per_launch": col_flops,
                "algorithmic_bytes_per_launch": 2.0 * (N_TOK * H + 2 * F * H + N_TOK * F),
                "launch_ms": col_t * 1e3}
    shard_reduce = {"value": red_bytes / red_t / 1e9, "unit": "GB/s",
                    "frac": red_bytes / red_t / 1e9 / peaks["hbm_gbs"], "peak": peaks["hbm_gbs"],
                    "peak_kind": f"HBM copy ({peak_src})", "ms": red_t * 1e3, "bytes": red_bytes,
                    "config": "t=4 bf16 partials of 8192 x 8192 (128 MiB each) -> 128 MiB, direct order"}
    row_flops = 2.0 * N_TOK * H * F
    detail = {"col_gate_up_ms": col_t * 1e3, "row_down_partials_ms": row_t * 1e3, "shard_reduce_ms": red_t * 1e3,
              "row_down_tflops": row_flops / row_t / 1e12}

    # ---------------- e2e: host buffers through tp_mlp_forward
    xh = torch.empty((N_TOK, H), dtype=torch.bfloat16, pin_memory=True)
    xh.copy_(x)
    yh = torch.empty((N_TOK, H), dtype=torch.bfloat16, pin_memory=True)
    xd = torch.empty_like(x)
    ws = torch.empty(tp.tp_mlp_workspace_size(T, N_TOK, H, F, "direct", torch.bfloat16), dtype=torch.uint8,
                     device=dev)

    copy_stream = torch.cuda.Stream(device=dev)
    e2e_runs = {}
    for chunks in (1, 2, 3, 4, 8):
        def e2e_step(chunks=chunks):
            tp.tp_mlp_forward_host(xh, wgu, wds, y_host=yh, x_dev=xd, y_dev=y, workspace=ws, mode="direct",
                                   chunks=chunks, stream=stream, copy_stream=copy_stream)
        e2e_runs[chunks] = (time_fn(torch, e2e_step, max(3, args.steps // 10), warm=2)
                            if not args.no_e2e else float("nan"))
    e2e_s = e2e_runs[E2E_CHUNKS]
    blocks = tp.tp_mlp_host_blocks(N_TOK, E2E_CHUNKS)
    e2e = {"value": FLOPS / e2e_s / 1e12 * world, "unit": "TFLOP/s", "h2d_bytes_per_step": N_TOK * H * 2,
           "d2h_bytes_per_step": N_TOK * H * 2, "ms_per_step": e2e_s * 1e3,
           "path": (f"pinned host X -> tp_mlp_forward_host (C ABI; chunks={E2E_CHUNKS}: row blocks of "
                    f"{[b - a for a, b in zip(blocks, blocks[1:])]} tokens, copies overlapped with compute on a "
                    "second stream) -> pinned host Y"),
           "ms_by_chunks": {str(k): v * 1e3 for k, v in e2e_runs.items()}}
    if args.no_e2e:                     # profiling runs: no end-to-end number (null, not NaN, in the JSON)
        e2e.update({"value": None, "ms_per_step": None, "ms_by_chunks": None})

    if not args.no_detail:
        rows = tuple(args.detail_rows.split(",")) if args.detail_rows else DETAIL_ROWS
        detail.update(bench_detail(torch, tp, synth, dev, peaks, wgu, wds, x, rows))
    del wgu, wds, hbuf, parts

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(torch, synth, dev)
    gpu_launches = 3 * args.steps
    res = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic: seeded N(0,1) activations, N(0,0.02) weights",
           "config": {"workload": WORKLOAD, "t": T, "n": N_TOK, "h": H, "f": F, "reduce": "direct",
                      "partials": "bf16", "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                      "l2": "inputs larger than L2 (X 128 MiB, weights 1.41 GB, partials 512 MiB)"},
           "tensor_frac_of_peak": value / tpeak, "tensor_peak_kind": tkind,
           "tensor_frac_of_burst": value / peaks["bf16_tflops"],
           "shard_reduce": shard_reduce, "roofline": roofline, "e2e": e2e, "gpu_launches": gpu_launches,
           "clocks": clk, "peaks": {**peaks, "source": peak_src}, "detail": detail}
    if cpu is not None:
        res["cpu_baseline"] = cpu
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return res


DETAIL_ROWS = ("prefill", "decode", "chunked", "prefill_t8", "reduce_sweep", "seqpar", "embed", "lm_head", "tiny",
               "attn", "host")


def bench_detail(torch, tp, synth, dev, peaks, wgu4, wds4, x, rows=DETAIL_ROWS):
    """Every other row of the hot path, timed once each (not part of value).
    `rows` selects sections (all by default; single rows serve profiling)."""
    out = {}
    hbm = peaks["hbm_gbs"]
    ten = peaks["bf16_tflops"]
    # fused down-GEMM + reduce, t=4 (reuses the step's weights)
    y = torch.empty((N_TOK, H), dtype=torch.bfloat16, device=dev)
    if "prefill" in rows:
        out.update(_detail_prefill(torch, tp, dev, ten, wgu4, wds4, x, y))
    if "decode" in rows:
        out.update(_detail_decode(torch, tp, dev, hbm, wgu4, wds4, x))
    if "chunked" in rows:
        out.update(_detail_chunked(torch, tp, dev, ten, wgu4, wds4, x))
    if "prefill_t8" in rows:
        out.update(_detail_prefill_t8(torch, tp, synth, dev, ten, y))
    if "reduce_sweep" in rows:
        out["shard_reduce_sweep"] = _detail_reduce_sweep(torch, tp, dev, hbm)
    if "seqpar" in rows:
        out.update(_detail_seqpar(torch, tp, dev, hbm))
    if "embed" in rows or "lm_head" in rows:
        out.update(_detail_vocab(torch, tp, synth, dev, hbm, ten, rows))
    if "tiny" in rows:
        out.update(_detail_tiny(torch, tp, synth, dev))
    if "attn" in rows:
        out.update(_detail_attn(torch, tp, synth, dev, hbm, ten))
    if "host" in rows:
        out["host_overhead"] = _detail_host_overhead(torch, tp, synth, dev)
    return out


def _detail_host_overhead(torch, tp, synth, dev):
    """Host cost per call of the C-ABI entry points: from C (a probe program
    with no Python in the loop), through the Python binding, and through the
    binding's prepared calls (checks and marshalling done once), all timed on
    the host clock from entry to return, calls enqueued back to back with a
    stream sync every 16 calls so none blocks on the device."""
    out = {}
    try:
        from megatron_tensor_layers_gb300.build import build_abi_overhead
        exe = build_abi_overhead()
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        out["c_abi"] = json.loads(r.stdout) if r.returncode == 0 else {"error": (r.stdout + r.stderr)[-300:]}
    except Exception as e:  # the probe is optional: report why it did not run
        out["c_abi"] = {"error": str(e)[-300:]}
    t, n, h, f = 2, 8, 1024, 3072
    x, wgu, wds = make_mlp(torch, synth, t, n, h, f, dev, seed=300)
    y = torch.empty((n, h), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tp.tp_mlp_workspace_size(t, n, h, f, "direct", torch.bfloat16), dtype=torch.uint8, device=dev)
    parts = [torch.zeros((8192,), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    red = torch.empty((8192,), dtype=torch.bfloat16, device=dev)
    hbuf = torch.empty((n, f), dtype=torch.bfloat16, device=dev)
    hs = [hbuf[:, r * (f // t):(r + 1) * (f // t)] for r in range(t)]
    calls = {
        "tp_shard_reduce_t4_n1": lambda: tp.tp_shard_reduce(parts, out=red, mode="direct"),
        "tp_linear_col_tiny_gated": lambda: tp.tp_linear_col(x, wgu, act="silu", y=hs),
        "tp_linear_row_tiny_fused": lambda: tp.tp_linear_row(hs, wds, mode="fused", y=y),
        "tp_mlp_forward_tiny_direct": lambda: tp.tp_mlp_forward(x, wgu, wds, mode="direct", workspace=ws, y=y),
    }
    prepared = {
        "tp_shard_reduce_t4_n1": tp.prepare(tp.tp_shard_reduce, parts, out=red, mode="direct"),
        "tp_linear_col_tiny_gated": tp.prepare(tp.tp_linear_col, x, wgu, act="silu", y=hs),
        "tp_linear_row_tiny_fused": tp.prepare(tp.tp_linear_row, hs, wds, mode="fused", y=y),
        "tp_mlp_forward_tiny_direct": tp.prepare(tp.tp_mlp_forward, x, wgu, wds, mode="direct", workspace=ws, y=y),
    }

    def host_times(fns):
        res = {}
        for name, fn in fns.items():
            for _ in range(20):
                fn()
            torch.cuda.synchronize()
            ts = []
            for i in range(200):
                t0 = time.perf_counter()
                fn()
                ts.append((time.perf_counter() - t0) * 1e6)
                if i % 16 == 15:
                    torch.cuda.synchronize()
            torch.cuda.synchronize()
            res[name] = {"host_us_median": statistics.median(ts), "host_us_mean": statistics.fmean(ts)}
        return res

    out["python_binding"] = host_times(calls)
    # the same calls checked and marshalled once (tp.prepare), then made again and again
    out["python_prepared"] = host_times(prepared)
    return out


def _detail_attn(torch, tp, synth, dev, hbm, ten):
    """The attention block's tensor-parallel projections at Llama-3.1-70B shapes, t=8
    (64 query heads, 8 KV heads, head size 128, h=8192): the head-aligned QKV column GEMM
    (rank r: 8 query heads and 1 KV head, [1280, 8192]) and the o_proj row GEMM ([8192,
    1024] per rank) into bf16 partials with the direct reduce, or with the reduce fused into
    the o_proj GEMM (rows tagged "_fused").  The attention between them
    is not part of the path; o_proj reads a seeded stand-in.  Decode (n=1, 64) is weight
    streaming, timed as CUDA graphs over two weight copies (2 x 302 MB, beyond the L2);
    prefill (n=8192) is compared with the tensor peak."""
    out = {}
    t, nh, nkv, hd, h = 8, 64, 8, 128, 8192
    qh = nh // t * hd
    wbytes = (t * (qh + 2 * hd) * h + h * nh * hd) * 2

    def weights(seed):
        blocks = [synth.normal_bf16((qh + 2 * hd, h), 0.02, seed + r, device=dev) for r in range(t)]
        wos = [synth.normal_bf16((h, qh), 0.02, seed + 20 + r, device=dev) for r in range(t)]
        return blocks, wos

    copies = [weights(900), weights(950)]
    for n in (1, 64, 8192):
        x = synth.normal_bf16((n, h), 1.0, 990, device=dev)
        attn = [synth.normal_bf16((n, qh), 1.0, 991 + r, device=dev) for r in range(t)]
        qkv = [torch.empty((n, qh + 2 * hd), dtype=torch.bfloat16, device=dev) for _ in range(t)]
        parts = [torch.empty((n, h), dtype=torch.bfloat16, device=dev) for _ in range(t)]
        y = torch.empty((n, h), dtype=torch.bfloat16, device=dev)

        def proj(c, mode="direct"):
            def run():
                tp.tp_linear_col(x, c[0], y=qkv)
                if mode == "fused":
                    tp.tp_linear_row(attn, c[1], mode="fused", y=y)
                else:
                    tp.tp_linear_row(attn, c[1], partials=parts, y=y)
            return run

        if n < 8192:
            for mode, tag in (("direct", ""), ("fused", "_fused")):
                gs = graph_time_cold(torch, [proj(c, mode) for c in copies], 5)
                if gs:
                    out[f"attn_proj_t8_n{n}{tag}"] = {"graph_us": gs * 1e6, "weight_GBps": wbytes / gs / 1e9,
                                                      "graph_hbm_frac": wbytes / gs / 1e9 / hbm}
        else:
            fl = 2.0 * n * h * (t * (qh + 2 * hd)) + 2.0 * n * h * (nh * hd)
            for mode, tag in (("direct", ""), ("fused", "_fused")):
                s = time_fn(torch, proj(copies[0], mode), 10)
                out[f"attn_proj_t8_n{n}{tag}"] = {"ms": s * 1e3, "tflops": fl / s / 1e12, "frac": fl / s / 1e12 / ten}
        del x, attn, qkv, parts, y
    del copies
    torch.cuda.empty_cache()
    return out


def time_modes_interleaved(torch, fns, rounds=6, iters=3):
    """Median device time (s) per call of each fn in `fns` (name -> fn), timed in
    alternation (round r times every fn once, `iters` calls each), so that every
    mode sees the same clock and power state."""
    for fn in fns.values():
        fn()
    torch.cuda.synchronize()
    times = {k: [] for k in fns}
    for _ in range(rounds):
        for k, fn in fns.items():
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(iters):
                fn()
            b.record()
            torch.cuda.synchronize()
            times[k].append(a.elapsed_time(b) / 1e3 / iters)
    return {k: statistics.median(v) for k, v in times.items()}


def _prefill_modes(torch, tp, dev, ten, t, x, wgu, wds, y):
    """tp_mlp_forward at n=8192 in direct (separate reduce), fused (down GEMM + reduce in one
    accumulator) and ring order, timed in alternation.  These rows are bursts of a few launches,
    nearer boost clock than the long timed step, so they are compared with the burst peak."""
    ws = {m: torch.empty(tp.tp_mlp_workspace_size(t, N_TOK, H, F, m, torch.bfloat16), dtype=torch.uint8, device=dev)
          for m in ("direct", "fused", "ring")}
    fns = {m: (lambda m=m: tp.tp_mlp_forward(x, wgu, wds, mode=m, workspace=ws[m], y=y)) for m in ws}
    med = time_modes_interleaved(torch, fns)
    out = {f"prefill_t{t}_{m}": {"ms": s * 1e3, "tflops": FLOPS / s / 1e12, "frac": FLOPS / s / 1e12 / ten}
           for m, s in med.items()}
    out[f"prefill_t{t}_fused_vs_direct"] = med["direct"] / med["fused"]
    del ws
    return out


def _detail_prefill(torch, tp, dev, ten, wgu4, wds4, x, y):
    return _prefill_modes(torch, tp, dev, ten, T, x, wgu4, wds4, y)


def _detail_decode(torch, tp, dev, hbm, wgu4, wds4, x):
    """Decode, t=4, n in {1, 16, 64}: weight streaming."""
    out = {}
    wbytes = 3.0 * H * F * 2
    for n in (1, 16, 64):
        xs = x[:n].contiguous()
        yd = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
        for mode in ("direct", "fused"):
            wsn = torch.empty(max(256, tp.tp_mlp_workspace_size(T, n, H, F, mode, torch.bfloat16)),
                              dtype=torch.uint8, device=dev)
            fn = lambda: tp.tp_mlp_forward(xs, wgu4, wds4, mode=mode, workspace=wsn, y=yd)
            s = time_fn(torch, fn, 20)
            rec = {"us": s * 1e6, "tflops": 6.0 * n * H * F / s / 1e12, "weight_GBps": wbytes / s / 1e9,
                   "hbm_frac": wbytes / s / 1e9 / hbm}
            gs = graph_time(torch, fn, 10)          # replayed from a CUDA graph, as a serving loop runs it
            if gs:
                rec.update({"graph_us": gs * 1e6, "graph_hbm_frac": wbytes / gs / 1e9 / hbm})
            out[f"decode_t4_n{n}_{mode}"] = rec
    return out


def _detail_chunked(torch, tp, dev, ten, wgu4, wds4, x):
    """Chunked-prefill sizes of the same MLP (t=4): 200, 256 and 384 tokens, direct (separate
    reduce) and fused (down GEMM + reduce; at 129-256 tokens every down-GEMM tile split along K
    over two CTA pairs), timed in alternation.  Weights 1.41 GB (beyond the L2)."""
    out = {}
    for n in (200, 256, 384):
        xs = x[:n].contiguous()
        yd = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
        ws = {m: torch.empty(tp.tp_mlp_workspace_size(T, n, H, F, m, torch.bfloat16), dtype=torch.uint8, device=dev)
              for m in ("direct", "fused")}
        fns = {m: (lambda m=m: tp.tp_mlp_forward(xs, wgu4, wds4, mode=m, workspace=ws[m], y=yd)) for m in ws}
        med = time_modes_interleaved(torch, fns, rounds=6, iters=5)
        fl = 6.0 * n * H * F
        for m, s in med.items():
            out[f"chunked_t4_n{n}_{m}"] = {"us": s * 1e6, "tflops": fl / s / 1e12, "frac": fl / s / 1e12 / ten}
    return out


def _detail_prefill_t8(torch, tp, synth, dev, ten, y):
    """t=8 prefill, separate and fused."""
    out = {}
    x8, wgu8, wds8 = make_mlp(torch, synth, 8, N_TOK, H, F, dev, seed=50)
    out.update(_prefill_modes(torch, tp, dev, ten, 8, x8, wgu8, wds8, y))
    del x8, wgu8, wds8
    torch.cuda.empty_cache()
    return out


def _detail_tiny(torch, tp, synth, dev):
    """The tiny TP-MLP (t=2, h=1024, f=3072, n=8): a latency row, in us per MLP
    (gate_up GEMM + down GEMM + reduce, or the fused down+reduce)."""
    out = {}
    t, n, h, f = 2, 8, 1024, 3072
    x, wgu, wds = make_mlp(torch, synth, t, n, h, f, dev, seed=90)
    y = torch.empty((n, h), dtype=torch.bfloat16, device=dev)
    wbytes = 3.0 * h * f * 2
    # Cold: each launch of the graph runs its own copy of the weights (and input), the copies
    # together twice the L2.  Warm (context only): one copy, L2-resident across launches.
    sets = cold_set_count(torch, wbytes, 64)
    copies = [(x, wgu, wds)] + [make_mlp(torch, synth, t, n, h, f, dev, seed=90 + 10 * j) for j in range(1, sets)]
    for mode in ("direct", "ring", "fused"):
        ws = torch.empty(max(256, tp.tp_mlp_workspace_size(t, n, h, f, mode, torch.bfloat16)), dtype=torch.uint8,
                         device=dev)
        fn = lambda: tp.tp_mlp_forward(x, wgu, wds, mode=mode, workspace=ws, y=y)
        rec = {"us": time_fn(torch, fn, 100) * 1e6, "weight_MB": wbytes / 1e6}
        fns = [(lambda c: (lambda: tp.tp_mlp_forward(c[0], c[1], c[2], mode=mode, workspace=ws, y=y)))(c)
               for c in copies]
        gs = graph_time_cold(torch, fns, 4)
        if gs:
            rec.update({"graph_us": gs * 1e6, "graph_weight_GBps": wbytes / gs / 1e9, "graph_sets": sets})
        gw = graph_time(torch, fn, 100)
        if gw:
            rec["graph_us_l2_warm"] = gw * 1e6
        out[f"tiny_t2_n8_{mode}"] = rec
    del copies
    return out


def _detail_reduce_sweep(torch, tp, dev, hbm):
    """Shard-reduce sweep: t in {2,4,8}, n in {1,64,8192}, h=8192, bf16 and fp32, direct and ring."""
    sweep = {}
    for dt in (torch.bfloat16, torch.float32):
        es = 2 if dt == torch.bfloat16 else 4
        for t in (2, 4, 8):
            base = [torch.randn((N_TOK * H,), device=dev).to(dt) for _ in range(t)]
            o_all = torch.empty((N_TOK * H,), dtype=dt, device=dev)
            for n in (1, 64, 8192):
                ps = [b[: n * H] for b in base]
                o = o_all[: n * H]
                for mode in ("direct", "ring"):
                    iters = 20 if n == 8192 else 200
                    fn = lambda: tp.tp_shard_reduce(ps, out=o, mode=mode)
                    s = time_fn(torch, fn, iters)
                    byts = (t + 1) * n * H * es
                    rec = {"us": s * 1e6, "GBps": byts / s / 1e9, "hbm_frac": byts / s / 1e9 / hbm}
                    if n < 8192:
                        # small messages: eager calls time the host's launch rate; a CUDA-graph
                        # replay gives the device latency of one reduce (the all-reduce's alpha).
                        # Cold: each launch reduces its own slices of the buffers, the slices of
                        # all launches together twice the L2.  Warm: the same slices every launch,
                        # as when the partials come straight from the GEMM that wrote them.
                        sets = cold_set_count(torch, byts, N_TOK // n)
                        fns = [(lambda j: (lambda: tp.tp_shard_reduce(
                            [b[j * n * H:(j + 1) * n * H] for b in base], out=o_all[j * n * H:(j + 1) * n * H],
                            mode=mode)))(j) for j in range(sets)]
                        gs = graph_time_cold(torch, fns)
                        if gs:
                            rec.update({"graph_us": gs * 1e6, "graph_GBps": byts / gs / 1e9,
                                        "graph_hbm_frac": byts / gs / 1e9 / hbm, "graph_sets": sets})
                        gw = graph_time(torch, fn, 50)
                        if gw:
                            rec["graph_us_l2_warm"] = gw * 1e6
                    sweep[f"{'bf16' if es == 2 else 'f32'}_t{t}_n{n}_{mode}"] = rec
            del base, o_all
    return sweep


def _detail_seqpar(torch, tp, dev, hbm):
    """Sequence parallelism: reduce-scatter + residual + RMSNorm (all-gather in place), t=4, bf16."""
    out = {}
    parts4 = [torch.randn((N_TOK, H), device=dev).to(torch.bfloat16) for _ in range(4)]
    resid = torch.randn((N_TOK, H), device=dev).to(torch.bfloat16)
    wn = torch.randn((H,), device=dev).to(torch.bfloat16)
    res_out = torch.empty_like(resid)
    nrm = torch.empty_like(resid)
    for mode in ("direct", "ring"):
        s = time_fn(torch, lambda: tp.tp_reduce_scatter_rmsnorm(parts4, wn, residual=resid, mode=mode,
                                                                residual_out=res_out, out=nrm), 20)
        byts = (4 + 1 + 2) * N_TOK * H * 2
        out[f"rs_rmsnorm_t4_n{N_TOK}_{mode}"] = {"us": s * 1e6, "GBps": byts / s / 1e9,
                                                 "hbm_frac": byts / s / 1e9 / hbm}
    del parts4, resid, res_out, nrm
    return out


def _detail_vocab(torch, tp, synth, dev, hbm, ten, rows):
    """Vocab-parallel embedding + LM head, V=151936, h=1024, 4096 ids."""
    out = {}
    V, hh, nt = 151936, 1024, 4096
    table = synth.normal_bf16((V, hh), 0.02, 6, device=dev)
    ids = synth.uniform_ids(nt, V, 5, device=dev)
    xh = synth.normal_bf16((nt, hh), 1.0, 7, device=dev)
    logits = torch.empty((nt, V), dtype=torch.bfloat16, device=dev)
    ids_big = synth.uniform_ids(65536, V, 15, device=dev)
    for t in (2, 4):
        per = (V + t - 1) // t
        shards = [table[r * per:min((r + 1) * per, V)].contiguous() for r in range(t)]
        for tag, idv in ((("", ids), ("_65536ids", ids_big)) if "embed" in rows else ()):
            m = idv.numel()
            e = torch.empty((m, hh), dtype=torch.bfloat16, device=dev)
            s = time_fn(torch, lambda: tp.vocab_parallel_embed(idv, shards, V, out=e), 200 if m == nt else 50)
            byts = m * 4 + 2 * m * hh * 2
            rec = {"us": s * 1e6, "GBps": byts / s / 1e9, "hbm_frac": byts / s / 1e9 / hbm, "bytes": byts}
            # Cold: a CUDA graph of lookups, each with its own seeded ids (so its own table rows) and
            # its own output, the sets together twice the L2.  Warm (context only): the same ids and
            # output every launch, so rows, ids and output stay in L2.
            sets = cold_set_count(torch, byts, 64)
            idss = [idv] + [synth.uniform_ids(m, V, 500 + 7 * j + m, device=dev) for j in range(1, sets)]
            outs = [e] + [torch.empty((m, hh), dtype=torch.bfloat16, device=dev) for _ in range(1, sets)]
            fns = [(lambda j: (lambda: tp.vocab_parallel_embed(idss[j], shards, V, out=outs[j])))(j)
                   for j in range(sets)]
            graph_s = graph_time_cold(torch, fns, 4 if m == nt else 1)
            if graph_s:
                rec.update({"graph_us": graph_s * 1e6, "graph_GBps": byts / graph_s / 1e9,
                            "graph_hbm_frac": byts / graph_s / 1e9 / hbm, "graph_sets": sets})
            gw = graph_time(torch, lambda: tp.vocab_parallel_embed(idv, shards, V, out=e), 100 if m == nt else 20)
            if gw:
                rec["graph_us_l2_warm"] = gw * 1e6
            if m == nt:
                # The floor for a lookup this small: one launch of a contiguous copy of the same
                # bytes (the rows' 8 MB read, 8 MB written), cold L2, timed the same way.  A lookup
                # adds the dependent id load before its row loads.
                srcs = [torch.empty((m, hh), dtype=torch.bfloat16, device=dev) for _ in range(sets)]
                dsts = [torch.empty((m, hh), dtype=torch.bfloat16, device=dev) for _ in range(sets)]
                cs = graph_time_cold(torch, [(lambda j: (lambda: dsts[j].copy_(srcs[j])))(j) for j in range(sets)], 4)
                if cs:
                    rec["copy_same_bytes_graph_us"] = cs * 1e6
                del srcs, dsts
            del idss, outs, fns
            out[f"embed_t{t}{tag}"] = rec
        if "lm_head" not in rows:
            continue
        s = time_fn(torch, lambda: tp.lm_head_sharded(xh, shards, V, logits=logits), 10)
        fl = 2.0 * nt * hh * V
        out[f"lm_head_t{t}"] = {"ms": s * 1e3, "tflops": fl / s / 1e12, "frac": fl / s / 1e12 / ten,
                                "store_GBps": nt * V * 2 / s / 1e9}
        per_shard = tp.lm_head_sharded(xh, shards, V, per_shard=True)
        s = time_fn(torch, lambda: tp.tp_shard_gather(per_shard, out=logits), 10)
        byts = 2 * nt * V * 2
        out[f"gather_t{t}"] = {"ms": s * 1e3, "GBps": byts / s / 1e9, "hbm_frac": byts / s / 1e9 / hbm}
        del per_shard
    return out


def graph_time(torch, fn, reps):
    """Per-launch time of fn replayed from a CUDA graph of `reps` launches
    (median of three timed windows)."""
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(3):                       # median of three windows of 5 replays
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(5):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) / 1e3 / (5 * reps))
        return sorted(times)[1]
    except Exception:
        return None


def l2_bytes(torch):
    return int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0)) or 126 * 2**20


def cold_set_count(torch, set_bytes, cap):
    """How many disjoint buffer sets a rotation needs so that the sets together
    hold at least twice the L2: each set is then evicted before its next use."""
    return max(2, min(cap, -(-2 * l2_bytes(torch) // max(1, int(set_bytes)))))


def graph_time_cold(torch, fns, passes=1):
    """Per-launch time of a CUDA graph that calls fns[0], fns[1], ... in turn
    (`passes` times), each on its own buffers, with the buffers of all sets
    together larger than twice the L2: every launch starts with its inputs out
    of L2, as with an L2 flush between launches but without timing the flush.
    Median of three timed windows."""
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fns[0]()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(passes):
                for fn in fns:
                    fn()
        g.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(3):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) / 1e3 / (3 * passes * len(fns)))
        del g
        return sorted(times)[1]
    except Exception:
        return None


# ------------------------------------------------------------------ oracle

def oracle_sample(torch, synth, dev, rows, seed=0):
    """fp64 inputs of the bench workload for the first `rows` token rows."""
    import oracle as O
    fs = F // T
    x = synth.normal_bf16((N_TOK, H), 1.0, seed, device=dev)[:rows]
    wg = synth.normal_bf16((F, H), 0.02, seed + 1, device=dev)
    wu = synth.normal_bf16((F, H), 0.02, seed + 2, device=dev)
    wd = synth.normal_bf16((H, F), 0.02, seed + 3, device=dev)
    cv = lambda a: O.bf16_bits_to_f64(synth.bits_u16(a))
    out = (cv(x), cv(wg), cv(wu), cv(wd))
    del wg, wu, wd
    return out


def cpu_baseline(torch, synth, dev, rows=16):
    """The oracle as it stands (fp64 numpy, all host cores), on `rows` token
    rows of the bench workload: the sharded MLP of the pages with the
    partials summed in rank order."""
    import oracle as O
    xf, wg, wu, wd = oracle_sample(torch, synth, dev, rows)
    O.mlp_sharded(xf[:1], wg, wu, wd, T)                  # touch the pages once
    t0 = time.perf_counter()
    O.mlp_sharded(xf, wg, wu, wd, T)
    s = time.perf_counter() - t0
    return {"value": 6.0 * rows * H * F / s / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows} of 8192 token rows of the bench workload (all weights), fp64 numpy, "
                      f"{s:.2f} s", "seconds": s}


REF_TIMED_BUDGET_S = 120.0   # the reference arm's K timed steps together


def run_reference(args, rank, world):
    """Time the oracle on the host cores (rank 0 only).

    Each step is the oracle's sharded MLP (all t ranks, partials summed in
    rank order) on the first `ref_rows` token rows.  The MLP separates over
    the intermediate dimension, so when K full-width steps would run past
    the budget, every step takes the same leading slice of f (a multiple of
    128 per rank, gate/up rows and down columns alike) and the value counts
    only the flops of that slice.  The slice is set from one untimed
    full-width step."""
    if rank != 0:
        return None
    import torch
    from megatron_tensor_layers_gb300 import synth
    import oracle as O
    dev = "cpu"
    rows = args.ref_rows
    xf, wg, wu, wd = oracle_sample(torch, synth, dev, rows)
    t0 = time.perf_counter()
    O.mlp_sharded(xf, wg, wu, wd, T)
    full_s = time.perf_counter() - t0
    unit = 128 * T
    frac = min(1.0, REF_TIMED_BUDGET_S / max(args.steps, 1) / max(full_s, 1e-9))
    fs = max(unit, int(F * frac) // unit * unit)
    wg_s, wu_s, wd_s = wg[:fs], wu[:fs], wd[:, :fs]
    for _ in range(args.warmup):
        O.mlp_sharded(xf, wg_s, wu_s, wd_s, T)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.mlp_sharded(xf, wg_s, wu_s, wd_s, T)
    s = time.perf_counter() - t0
    v = 6.0 * rows * H * fs * args.steps / s / 1e12
    sample = (f"{rows} of {N_TOK} token rows per step, intermediate slice f'={fs} of {F} "
              f"(all of h), fp64 numpy on {os.cpu_count()} cores")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded N(0,1) activations, N(0,0.02) weights",
            "config": {"workload": WORKLOAD, "t": T, "n": N_TOK, "h": H, "f": F, "reduce": "direct"},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-detail", action="store_true", help="skip the per-row detail timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--tokens", type=int, default=8192,
                    help="token count of the step (8192 is the bench workload; smaller only for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--detail-rows", default="",
                    help="comma-separated subset of " + ",".join(DETAIL_ROWS) + " (default: all)")
    args = ap.parse_args()
    global N_TOK, FLOPS
    N_TOK = args.tokens
    FLOPS = 6.0 * N_TOK * H * F
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
