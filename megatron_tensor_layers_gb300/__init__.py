"""GB300-native tensor-parallel layers of an LLM serving stack, on one GPU.

The t ranks of a Megatron-style tensor-parallel group are simulated as t
shards in this GPU's memory; the column/row-parallel GEMMs, the shard
all-reduce, the vocab-parallel embedding and the vocab-sharded LM head run
as hand-written sm_103a kernels behind a C ABI (include/tp.h).  This package
is the Python binding of that ABI; the kernels are in ``csrc/``.
"""

from ._lib import (  # noqa: F401
    PreparedCall,
    TPError,
    lm_head_sharded,
    load,
    prepare,
    tp_abi_version,
    tp_collective_count,
    tp_debug_expire_wait,
    tp_device_status,
    tp_linear_col,
    tp_linear_row,
    tp_mlp_forward,
    tp_mlp_forward_host,
    tp_mlp_forward_static,
    tp_mlp_host_blocks,
    tp_mlp_host_workspace_size,
    tp_mlp_workspace_size,
    tp_reduce_scatter_rmsnorm,
    tp_reset_collective_count,
    tp_set_gemm_cta_pair,
    tp_set_gemm_split,
    tp_set_gemm_tile_n,
    tp_shard_gather,
    tp_shard_reduce,
    vocab_parallel_embed,
)
