"""The Python binding checks every tensor argument before it reaches the C
ABI (which sees only raw pointers and one row stride per list of shards):
shapes, dtypes, per-shard strides and contiguity first, then that every
tensor is a CUDA tensor.  Runs on the CPU: each case fails in the binding,
before any library call."""

import pytest
import torch

from megatron_tensor_layers_gb300 import _lib as tp

B = torch.bfloat16


def z(*shape, dtype=B):
    return torch.zeros(shape, dtype=dtype)


def test_host_tensors_are_refused_before_any_call():
    with pytest.raises(ValueError, match="CUDA"):
        tp.tp_linear_col(z(4, 64), [z(32, 64), z(32, 64)], y=[z(4, 32), z(4, 32)])
    with pytest.raises(ValueError, match="CUDA"):
        tp.tp_linear_row([z(4, 32), z(4, 32)], [z(64, 32), z(64, 32)], partials=[z(4, 64), z(4, 64)], y=z(4, 64))
    with pytest.raises(ValueError, match="CUDA"):
        tp.tp_shard_reduce([z(100), z(100)], out=z(100))
    with pytest.raises(ValueError, match="CUDA"):
        tp.tp_mlp_forward(z(4, 64), [z(64, 64), z(64, 64)], [z(64, 32), z(64, 32)],
                          workspace=torch.zeros(256, dtype=torch.uint8), y=z(4, 64))
    with pytest.raises(ValueError, match="CUDA"):
        tp.vocab_parallel_embed(torch.zeros(5, dtype=torch.int32), [z(5, 16), z(5, 16)], 10, out=z(5, 16))
    with pytest.raises(ValueError, match="CUDA"):
        tp.lm_head_sharded(z(4, 16), [z(5, 16), z(5, 16)], 10, logits=z(4, 10))
    with pytest.raises(ValueError, match="CUDA"):
        tp.tp_shard_gather([z(3, 4), z(3, 5)], out=z(3, 9))
    with pytest.raises(ValueError, match="CUDA"):
        tp.tp_reduce_scatter_rmsnorm([z(4, 16), z(4, 16)], z(16), out=z(4, 16))


def test_shapes_that_disagree_are_refused():
    with pytest.raises(ValueError, match="shape"):       # second shard narrower than the first
        tp.tp_linear_col(z(4, 64), [z(32, 64), z(16, 64)])
    with pytest.raises(ValueError, match="shape"):       # K of the weight differs from x
        tp.tp_linear_col(z(4, 64), [z(32, 48), z(32, 48)])
    with pytest.raises(ValueError, match="shape"):       # output of the wrong width
        tp.tp_linear_col(z(4, 64), [z(32, 64), z(32, 64)], y=[z(4, 32), z(4, 16)])
    with pytest.raises(ValueError, match="shape"):       # gated: y holds half the weight rows
        tp.tp_linear_col(z(4, 64), [z(32, 64), z(32, 64)], act="silu", y=[z(4, 32), z(4, 32)])
    with pytest.raises(ValueError, match="shape"):
        tp.tp_linear_row([z(4, 32), z(4, 16)], [z(64, 32), z(64, 32)])
    with pytest.raises(ValueError, match="shape"):       # partial buffers smaller than n x out
        tp.tp_linear_row([z(4, 32), z(4, 32)], [z(64, 32), z(64, 32)], partials=[z(4, 64), z(2, 64)])
    with pytest.raises(ValueError, match="shape"):
        tp.tp_shard_reduce([z(100), z(99)])
    with pytest.raises(ValueError, match="shape"):       # w_down[r] must be [h, f/t]
        tp.tp_mlp_forward(z(4, 64), [z(64, 64), z(64, 64)], [z(64, 16), z(64, 16)])
    with pytest.raises(ValueError, match="shape"):       # rank 1 owns ids 5..9: 5 rows
        tp.vocab_parallel_embed(torch.zeros(5, dtype=torch.int32), [z(5, 16), z(4, 16)], 10)
    with pytest.raises(ValueError, match="shape"):
        tp.lm_head_sharded(z(4, 16), [z(5, 16), z(5, 8)], 10)
    with pytest.raises(ValueError, match="shape"):
        tp.tp_reduce_scatter_rmsnorm([z(4, 16), z(4, 16)], z(8))
    with pytest.raises(ValueError, match="owns"):
        tp.vocab_parallel_embed(torch.zeros(5, dtype=torch.int32), [z(5, 16), None], 10)


def test_layouts_dtypes_and_counts_are_checked():
    w = z(64, 128)[:, :64]                                  # row stride 128
    with pytest.raises(ValueError, match="row stride"):    # one row stride serves every shard
        tp.tp_linear_col(z(4, 64), [z(32, 64), w[:32]])
    with pytest.raises(ValueError, match="row-major"):
        tp.tp_linear_col(z(64, 4).t(), [z(32, 64)])
    with pytest.raises(ValueError, match="contiguous"):    # gate_up blocks have no row stride in the ABI
        tp.tp_mlp_forward(z(4, 64), [w, w], [z(64, 32), z(64, 32)])
    with pytest.raises(TypeError, match="dtype"):
        tp.tp_linear_col(z(4, 64, dtype=torch.float32), [z(32, 64)])
    with pytest.raises(TypeError, match="dtype"):
        tp.vocab_parallel_embed(torch.zeros(5, dtype=torch.int64), [z(10, 16)], 10)
    with pytest.raises(ValueError, match="shards"):
        tp.tp_linear_col(z(4, 64), [])
    with pytest.raises(ValueError, match="shards"):
        tp.tp_shard_reduce([z(8)] * 9)
    with pytest.raises(ValueError, match="even"):
        tp.tp_mlp_forward(z(4, 64), [z(63, 64)], [z(64, 31)])
    with pytest.raises(ValueError, match="mode"):
        tp.tp_shard_reduce([z(8), z(8)], mode="fused")
    with pytest.raises(ValueError, match="gated"):
        tp.tp_mlp_forward(z(4, 64), [z(64, 64)], [z(64, 32)], act="none")
