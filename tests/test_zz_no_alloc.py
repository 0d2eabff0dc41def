"""tp_mlp_forward_static: the MLP entry point for callers that cannot allocate.

A host application that owns the device memory pool may forbid its plugins
to call cudaMalloc, and a latency-critical decode loop cannot afford
cudaMalloc/cudaFree (they can synchronise the device).  Such callers use
tp_mlp_forward_static, whose scratch is a fixed 16 MiB array inside the
library.  This test calls it through the C ABI twice in a row, with
different inputs each time (the array keeps the previous call's contents),
and checks each output against the regular workspace entry point on the same
inputs.  It also checks that a request larger than the array is refused.

This file is named so that pytest collects it last.
"""

import numpy as np
import pytest
import torch

from megatron_tensor_layers_gb300 import _lib as tp
from megatron_tensor_layers_gb300 import synth
from megatron_tensor_layers_gb300.build import build

from gpu_helpers import f64, gemm_gate

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _weights(t, h, f, seed):
    fs = f // t
    wg = synth.normal_bf16((f, h), 0.02, seed + 1, device=DEV)
    wu = synth.normal_bf16((f, h), 0.02, seed + 2, device=DEV)
    wd = synth.normal_bf16((h, f), 0.02, seed + 3, device=DEV)
    wgu = [torch.cat([wg[r * fs:(r + 1) * fs], wu[r * fs:(r + 1) * fs]]).contiguous() for r in range(t)]
    wds = [wd[:, r * fs:(r + 1) * fs].contiguous() for r in range(t)]
    return wgu, wds


@pytest.mark.parametrize("t,n,h,f,mode,pdt", [
    (2, 8, 1024, 3072, "direct", torch.bfloat16),     # the tiny TP-MLP config
    (4, 64, 8192, 28672, "direct", torch.float32),    # 70B-shaped decode, 12.1 MB of scratch
    (4, 64, 8192, 28672, "ring", torch.bfloat16),
    (8, 16, 8192, 28672, "fused", torch.bfloat16),
])
def test_static_scratch_matches_workspace_entry_point(t, n, h, f, mode, pdt):
    build()
    lib = tp.load()
    wgu, wds = _weights(t, h, f, 40)
    for call in range(2):
        x = synth.normal_bf16((n, h), 1.0, 100 + call, device=DEV)
        y_ref = tp.tp_mlp_forward(x, wgu, wds, mode=mode, partial_dtype=pdt, y_dtype=torch.float32)
        y = torch.empty((n, h), dtype=torch.float32, device=DEV)
        code = lib.tp_mlp_forward_static(t, n, h, f, x.data_ptr(), h, tp._ptrs(wgu), tp._ptrs(wds), f // t, None,
                                         tp.ACTS["silu"], tp.MODES[mode], tp.DTYPES[pdt], y.data_ptr(),
                                         tp.DTYPES[torch.float32], torch.cuda.current_stream().cuda_stream)
        assert code == 0, tp.STATUS_NAMES.get(code, code)
        torch.cuda.synchronize()
        assert tp.tp_device_status() == 0
        ref = f64(y_ref)
        gemm_gate(f64(y), ref, bf16_out=False)
        assert np.sqrt(np.mean(ref ** 2)) > 0.0


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
