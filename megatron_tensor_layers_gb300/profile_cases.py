"""One small case per kernel, for single-kernel profiler captures.

    python -m megatron_tensor_layers_gb300.profile_cases <case>

Each case runs the kernel it names twice on seeded synthetic inputs larger
than the L2 but of a few GB at most, so that a capture of one launch
(``-s 1 -c 1``) sees cold data and ends in seconds.  Cases: reduce, embed,
gather, seqpar, decode (70B MLP, t=4, 16 tokens, direct then fused, twice),
pair2048 (prefill MLP, 2048 tokens: the CTA-pair gate_up and down GEMMs),
fused1280 (fused down GEMM + reduce of 1280 rows given scratch: its last wave
split along K), tiny (the tiny TP-MLP fused, t=2, h=1024, f=3072, 8 tokens: the
one-kernel path, over 15 weight copies so that each call starts cold), qkv
(the 70B attention QKV column GEMM at t=8, one token, two weight copies),
decode64 (70B MLP decode, t=4, 64 tokens, fused: the split-K down GEMM with five
stages and its staging in the ring), fused200 (70B MLP, t=4, 200 tokens, fused:
every tile of the down GEMM split along K over two CTA pairs).
"""

import sys

import torch

from . import _lib as tp
from . import synth
from .build import build

H, F = 8192, 28672


def run(mode: str, dev: str = "cuda") -> None:
    if mode == "reduce":                      # t=4, 2048 tokens: 4 x 32 MiB bf16 -> 32 MiB
        parts = [torch.randn(2048 * H, device=dev).to(torch.bfloat16) for _ in range(4)]
        out = torch.empty(2048 * H, dtype=torch.bfloat16, device=dev)
        for _ in range(2): tp.tp_shard_reduce(parts, out=out)
    elif mode == "embed":                     # 65536 ids, t=2, V=151936, h=1024 (269 MB moved)
        V = 151936
        table = synth.normal_bf16((V, 1024), 0.02, 6, device=dev)
        shards = [table[:V // 2].contiguous(), table[V // 2:].contiguous()]
        ids = synth.uniform_ids(65536, V, 5, device=dev)
        for _ in range(2): tp.vocab_parallel_embed(ids, shards, V)
    elif mode == "gather":                    # logits all-gather, t=2, 1024 rows of V=151936
        V = 151936
        sh = [synth.normal_bf16((1024, V // 2), 1.0, 3 + r, device=dev) for r in range(2)]
        out = torch.empty((1024, V), dtype=torch.bfloat16, device=dev)
        for _ in range(2): tp.tp_shard_gather(sh, out=out)
    elif mode == "seqpar":                    # t=4, 2048 tokens
        parts = [torch.randn((2048, H), device=dev).to(torch.bfloat16) for _ in range(4)]
        resid = torch.randn((2048, H), device=dev).to(torch.bfloat16)
        w = torch.randn((H,), device=dev).to(torch.bfloat16)
        for _ in range(2): tp.tp_reduce_scatter_rmsnorm(parts, w, residual=resid, residual_out=resid)
    elif mode == "decode":                    # 70B MLP decode, t=4, n=16: direct, then fused
        t = 4; fs = F // t
        x = synth.normal_bf16((16, H), 1.0, 0, device=dev)
        wgu = [synth.normal_bf16((2 * fs, H), 0.02, 10 + r, device=dev) for r in range(t)]
        wds = [synth.normal_bf16((H, fs), 0.02, 20 + r, device=dev) for r in range(t)]
        for m in ("direct", "fused", "direct", "fused"):
            tp.tp_mlp_forward(x, wgu, wds, mode=m, partial_dtype=torch.bfloat16)
    elif mode in ("decode64", "fused200"):   # 70B MLP, t=4, fused reduce
        t = 4; fs = F // t
        n = 64 if mode == "decode64" else 200
        x = synth.normal_bf16((n, H), 1.0, 0, device=dev)
        wgu = [synth.normal_bf16((2 * fs, H), 0.02, 10 + r, device=dev) for r in range(t)]
        wds = [synth.normal_bf16((H, fs), 0.02, 20 + r, device=dev) for r in range(t)]
        ws = torch.empty(tp.tp_mlp_workspace_size(t, n, H, F, "fused"), dtype=torch.uint8, device=dev)
        for _ in range(2): tp.tp_mlp_forward(x, wgu, wds, mode="fused", workspace=ws)
    elif mode == "pair2048":                  # prefill n=2048, t=4: gate_up + down (CTA pairs)
        t = 4; fs = F // t
        x = synth.normal_bf16((2048, H), 1.0, 0, device=dev)
        wgu = [synth.normal_bf16((2 * fs, H), 0.02, 10 + r, device=dev) for r in range(t)]
        wds = [synth.normal_bf16((H, fs), 0.02, 20 + r, device=dev) for r in range(t)]
        for _ in range(2): tp.tp_mlp_forward(x, wgu, wds, mode="direct")
    elif mode == "tiny":                      # one-kernel fused MLP, 15 x 18.9 MB of weights
        t, n, h, f = 2, 8, 1024, 3072
        fs = f // t
        sets = [(synth.normal_bf16((n, h), 1.0, 90 + 10 * j, device=dev),
                 [synth.normal_bf16((2 * fs, h), 0.02, 91 + 10 * j + r, device=dev) for r in range(t)],
                 [synth.normal_bf16((h, fs), 0.02, 95 + 10 * j + r, device=dev) for r in range(t)]) for j in range(15)]
        for x, wgu, wds in sets:
            tp.tp_mlp_forward(x, wgu, wds, mode="fused")
    elif mode == "qkv":                       # 70B QKV, t=8, n=1: 8 x [1280, 8192], two weight copies
        t = 8
        copies = [[synth.normal_bf16((1280, H), 0.02, 900 + 50 * c + r, device=dev) for r in range(t)] for c in range(2)]
        x = synth.normal_bf16((1, H), 1.0, 990, device=dev)
        for _ in range(2):
            for w in copies:
                tp.tp_linear_col(x, w)
    elif mode == "fused1280":                 # fused down + reduce, 1280 rows: its last wave split along K
        t = 4; fs = F // t
        hs = [synth.normal_bf16((1280, fs), 1.0, 30 + r, device=dev) for r in range(t)]
        wds = [synth.normal_bf16((H, fs), 0.02, 20 + r, device=dev) for r in range(t)]
        scratch = torch.empty((1280, H), dtype=torch.float32, device=dev)      # contiguous: lent as scratch
        for _ in range(2): tp.tp_linear_row(hs, wds, mode="fused", y_dtype=torch.float32, partials=[scratch] * t)
    else:
        raise ValueError(f"unknown case {mode}")
    torch.cuda.synchronize()
    if tp.tp_device_status() != 0:
        raise RuntimeError("device status error")
    print("ok", mode)


if __name__ == "__main__":
    build()
    tp.load()
    run(sys.argv[1])
