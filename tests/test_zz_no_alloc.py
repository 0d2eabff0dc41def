"""tp_mlp_forward_static: the MLP entry point for callers that cannot allocate.

A host application that owns the device memory pool may forbid its plugins
to call cudaMalloc, and a latency-critical decode loop cannot afford
cudaMalloc/cudaFree (they can synchronise the device).  Such callers use
tp_mlp_forward_static, whose scratch is a fixed 16 MiB array inside the
library.  This test calls it through the C ABI twice in a row, with
different inputs each time (the array keeps the previous call's contents).
Each output must be bit-identical to the regular workspace entry point's on
the same inputs (same kernels, same order of arithmetic) and pass the MLP
gates against the oracle.  After a first call, a call given its own output
buffer must leave torch's allocated bytes and the device's free bytes
unchanged.  A request larger than the array is refused.

This file is named so that pytest collects it last.
"""

import gc

import pytest
import torch

from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

from gpu_helpers import f64, mlp_check

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _weights(t, h, f, seed):
    fs = f // t
    wg = synth.normal_bf16((f, h), 0.02, seed + 1, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, seed + 2, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, seed + 3, device=DEV)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    return (wg, wu, wd), wgu, wds


def _call_static(lib, t, n, h, f, x, wgu, wds, mode, pdt, y):
    return lib.tp_mlp_forward_static(t, n, h, f, x.data_ptr(), h, tp._ptrs(wgu), tp._ptrs(wds), f // t, None,
                                     tp.ACTS["silu"], tp.MODES[mode], tp.DTYPES[pdt], y.data_ptr(),
                                     tp.DTYPES[torch.float32], torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("t,n,h,f,mode,pdt", [
    (2, 8, 1024, 3072, "direct", torch.bfloat16),     # the tiny TP-MLP config
    (2, 8, 1024, 3072, "fused", torch.bfloat16),      # the same, one-kernel path (1.5 MB of slice partials)
    (4, 64, 8192, 28672, "direct", torch.float32),    # 70B-shaped decode, 12.1 MB of scratch
    (4, 64, 8192, 28672, "ring", torch.bfloat16),
    (8, 16, 8192, 28672, "fused", torch.bfloat16),
])
def test_static_scratch_matches_workspace_entry_point(t, n, h, f, mode, pdt):
    build()
    lib = tp.load()
    full, wgu, wds = _weights(t, h, f, 40)
    host_w = [f64(w) for w in full]
    for call in range(2):
        x = synth.normal_bf16((n, h), 1.0, 100 + call, device=DEV)
        y_ref = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=pdt, y_dtype=torch.float32)
        y = torch.full((n, h), float("nan"), dtype=torch.float32, device=DEV)
        code = _call_static(lib, t, n, h, f, x, wgu, wds, mode, pdt, y)
        assert code == 0, tp.STATUS_NAMES.get(code, code)
        torch.cuda.synchronize()
        assert tp.tp_device_status() == 0
        assert torch.equal(y, y_ref), "static-scratch output differs from the workspace entry point's"
        mlp_check(f64(y), f64(x), *host_w, t, mode=mode, partial="bf16" if pdt == torch.bfloat16 else "f32")


def test_static_scratch_allocates_nothing():
    build()
    lib = tp.load()
    t, n, h, f = 4, 64, 8192, 28672
    full, wgu, wds = _weights(t, h, f, 50)
    x = synth.normal_bf16((n, h), 1.0, 120, device=DEV)
    y = torch.empty((n, h), dtype=torch.float32, device=DEV)
    # first call: loads the module and its kernels on this device if that has not happened yet
    assert _call_static(lib, t, n, h, f, x, wgu, wds, "direct", torch.float32, y) == 0
    torch.cuda.synchronize()
    y2 = torch.empty((n, h), dtype=torch.float32, device=DEV)
    # Earlier tests' tensors that sit in reference cycles are freed whenever Python's cycle
    # collector runs; collect them now and keep the collector off while measuring, so that
    # only the call itself can change the counts.
    gc.collect()
    gc.disable()
    try:
        torch.cuda.synchronize()
        allocated = torch.cuda.memory_allocated()
        free_before = torch.cuda.mem_get_info()[0]
        code = _call_static(lib, t, n, h, f, x, wgu, wds, "direct", torch.float32, y2)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        allocated_after = torch.cuda.memory_allocated()
    finally:
        gc.enable()
    assert code == 0
    assert allocated_after == allocated
    assert free_after == free_before
    assert torch.equal(y, y2)
    assert tp.tp_device_status() == 0


def test_static_scratch_refuses_oversized_requests():
    build()
    lib = tp.load()
    t, n, h, f = 4, 8192, 8192, 28672          # prefill: far beyond 16 MiB of scratch
    need = lib.tp_mlp_workspace_size(t, n, h, f, tp.MODES["direct"], tp.DTYPES[torch.bfloat16])
    assert need > tp.STATIC_SCRATCH_BYTES
    dummy = (tp.P * t)(*([0x10000] * t))
    code = lib.tp_mlp_forward_static(t, n, h, f, 0x10000, h, dummy, dummy, f // t, None, tp.ACTS["silu"],
                                     tp.MODES["direct"], tp.DTYPES[torch.bfloat16], 0x10000,
                                     tp.DTYPES[torch.bfloat16], None)
    assert code == 7                            # TP_ERR_WORKSPACE, nothing launched
