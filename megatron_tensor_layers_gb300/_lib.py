"""ctypes binding of ``libtp_gb300.so`` (the C ABI declared in include/tp.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors; their data
pointers, row strides and the current CUDA stream are passed through.  If
the library is not built, or a call is made on a machine without a CUDA
device, the call raises: there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtp_gb300.so")

TP_OK = 0
STATUS_NAMES = {
    0: "TP_OK", 1: "TP_ERR_INVALID_ARG", 2: "TP_ERR_NOT_DIVISIBLE", 3: "TP_ERR_ALIGNMENT",
    4: "TP_ERR_UNSUPPORTED", 5: "TP_ERR_CUDA", 6: "TP_ERR_TIMEOUT", 7: "TP_ERR_WORKSPACE",
}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}
MODES = {"direct": 0, "ring": 1, "fused": 2}
ACTS = {"none": 0, "silu": 1, "gelu_tanh": 2}
MAX_SHARDS = 8

EXPORTED = [
    "tp_status_string", "tp_abi_version", "tp_linear_col", "tp_linear_row", "tp_shard_reduce",
    "tp_mlp_workspace_size", "tp_mlp_forward", "vocab_parallel_embed", "lm_head_sharded",
    "tp_shard_gather", "tp_device_status", "tp_collective_count", "tp_reset_collective_count",
    "tp_debug_expire_wait", "tp_set_gemm_tile_n", "tp_mlp_forward_static", "tp_set_gemm_cta_pair", "tp_mlp_forward_host",
    "tp_reduce_scatter_rmsnorm", "tp_set_gemm_split",
]
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024


class TPError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")


_lib = None
P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int


def load() -> ctypes.CDLL:
    """Load the library (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "tp_status_string": (ctypes.c_char_p, [I32]),
        "tp_abi_version": (I32, []),
        "tp_linear_col": (I32, [I32, I64, I64, I64, P, I64, P, I64, P, I32, I32, P, I64, I32, P]),
        "tp_linear_row": (I32, [I32, I64, I64, I64, P, I64, P, I64, P, I32, I32, I32, P, I64, P, I64, I32, P]),
        "tp_shard_reduce": (I32, [I32, I64, I32, P, P, I32, I32, I32, I32, P]),
        "tp_mlp_workspace_size": (ctypes.c_size_t, [I32, I64, I64, I64, I32, I32]),
        "tp_mlp_forward": (I32, [I32, I64, I64, I64, P, I64, P, P, I64, P, I32, I32, I32, P, ctypes.c_size_t, P, I32, P]),
        "vocab_parallel_embed": (I32, [I32, I64, I64, P, I64, P, I32, P, P, P]),
        "lm_head_sharded": (I32, [I32, I64, I64, I64, P, I64, P, P, I64, P, I32, P]),
        "tp_shard_gather": (I32, [I32, I64, P, I32, P, P, P]),
        "tp_device_status": (I32, [P]),
        "tp_collective_count": (ctypes.c_uint64, []),
        "tp_reset_collective_count": (None, []),
        "tp_debug_expire_wait": (I32, [ctypes.c_uint64, P]),
        "tp_set_gemm_tile_n": (I32, [I32]),
        "tp_set_gemm_cta_pair": (I32, [I32]),
        "tp_set_gemm_split": (I32, [I32, I32]),
        "tp_reduce_scatter_rmsnorm": (I32, [I32, I64, I64, I32, P, P, P, ctypes.c_float, I32, P, P, P]),
        "tp_mlp_forward_host": (I32, [I32, I64, I64, I64, P, P, P, I64, P, I32, I32, I32, P, P, ctypes.c_size_t, P, P,
                                      I32, I32, P, P]),
        "tp_mlp_forward_static": (I32, [I32, I64, I64, I64, P, I64, P, P, I64, P, I32, I32, I32, P, I32, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, code: int) -> None:
    if code != TP_OK:
        raise TPError(fn, code)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _ptrs(ts: Optional[Sequence[Optional[torch.Tensor]]]):
    if ts is None:
        return None
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = None if t is None else t.data_ptr()
    return arr


def _ld(t: torch.Tensor) -> int:
    assert t.dim() == 2 and t.stride(1) == 1, "matrices must be row-major with unit column stride"
    return t.stride(0)


def _dt(dtype) -> int:
    if dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {dtype}")
    return DTYPES[dtype]


# ----------------------------------------------------------------- entry points

def tp_abi_version() -> int:
    return load().tp_abi_version()


def tp_linear_col(x: torch.Tensor, w: Sequence[torch.Tensor], *, act: str = "none",
                  bias: Optional[Sequence[torch.Tensor]] = None, gather_output: bool = False,
                  y=None, y_dtype=torch.bfloat16, stream=None):
    """ColumnParallelLinear over t shards.  w[r] is [out/t, in] (act="none") or
    rank r's merged [gate; up] block [2*out/t, in].  Returns the list of
    per-shard outputs, or the gathered [n, out] tensor if gather_output."""
    t = len(w)
    n, k = x.shape
    os_ = w[0].shape[0] // (2 if act != "none" else 1)
    out_full = os_ * t
    if y is None:
        if gather_output:
            y = torch.empty((n, out_full), dtype=y_dtype, device=x.device)
        else:
            y = [torch.empty((n, os_), dtype=y_dtype, device=x.device) for _ in range(t)]
    ys = [y] if gather_output else list(y)
    ldy = _ld(ys[0])
    code = load().tp_linear_col(t, n, k, out_full, _ptr(x), _ld(x), _ptrs(w), _ld(w[0]), _ptrs(bias),
                                ACTS[act], int(gather_output), _ptrs(ys), ldy, _dt(ys[0].dtype), _stream(stream))
    _check("tp_linear_col", code)
    return y


def tp_linear_row(x: Sequence[torch.Tensor], w: Sequence[torch.Tensor], *, bias: Optional[torch.Tensor] = None,
                  reduce_results: bool = True, mode: str = "direct", partial_dtype=torch.bfloat16,
                  partials: Optional[List[torch.Tensor]] = None, y: Optional[torch.Tensor] = None,
                  y_dtype=torch.bfloat16, stream=None):
    """RowParallelLinear: x[r] [n, in/t], w[r] [out, in/t].  Returns y (the
    all-reduced sum) when reduce_results, else the list of partials."""
    t = len(w)
    n, ks = x[0].shape
    out = w[0].shape[0]
    dev = x[0].device
    if mode != "fused" and partials is None:
        partials = [torch.empty((n, out), dtype=partial_dtype, device=dev) for _ in range(t)]
    if reduce_results and y is None:
        y = torch.empty((n, out), dtype=y_dtype, device=dev)
    ldp = _ld(partials[0]) if partials is not None else out
    pdt = partials[0].dtype if partials is not None else partial_dtype
    code = load().tp_linear_row(t, n, ks * t, out, _ptrs(x), _ld(x[0]), _ptrs(w), _ld(w[0]), _ptr(bias),
                                int(reduce_results), MODES[mode], _dt(pdt), _ptrs(partials), ldp,
                                _ptr(y), _ld(y) if y is not None else out, _dt(y.dtype) if y is not None else 0,
                                _stream(stream))
    _check("tp_linear_row", code)
    return y if reduce_results else partials


def tp_shard_reduce(partials: Sequence[torch.Tensor], *, out: Optional[torch.Tensor] = None, out_dtype=None,
                    mode: str = "direct", hop_dtype=torch.float32, replicate: bool = False,
                    alloc_out: bool = True, stream=None):
    """All-reduce (sum) of t equally shaped partial buffers."""
    t = len(partials)
    p0 = partials[0]
    if out is None and alloc_out and not replicate:
        out = torch.empty(p0.shape, dtype=out_dtype or p0.dtype, device=p0.device)
    code = load().tp_shard_reduce(t, p0.numel(), _dt(p0.dtype), _ptrs(partials), _ptr(out),
                                  _dt(out.dtype) if out is not None else 0, MODES[mode], _dt(hop_dtype),
                                  int(replicate), _stream(stream))
    _check("tp_shard_reduce", code)
    return out


def tp_mlp_workspace_size(t: int, n: int, h: int, f: int, mode: str = "direct", partial_dtype=torch.bfloat16) -> int:
    return load().tp_mlp_workspace_size(t, n, h, f, MODES[mode], _dt(partial_dtype))


def tp_mlp_forward(x: torch.Tensor, w_gate_up: Sequence[torch.Tensor], w_down: Sequence[torch.Tensor], *,
                   bias_down: Optional[torch.Tensor] = None, act: str = "silu", mode: str = "direct",
                   partial_dtype=torch.bfloat16, workspace: Optional[torch.Tensor] = None,
                   y: Optional[torch.Tensor] = None, y_dtype=torch.bfloat16, stream=None):
    """Tensor-parallel MLP block Y = sum_r act(X A_r) B_r.  w_gate_up[r] is
    [2f/t, h] (gate rows then up rows), w_down[r] is [h, f/t]."""
    t = len(w_gate_up)
    n, h = x.shape
    f = w_gate_up[0].shape[0] // 2 * t
    need = tp_mlp_workspace_size(t, n, h, f, mode, partial_dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    if y is None:
        y = torch.empty((n, h), dtype=y_dtype, device=x.device)
    code = load().tp_mlp_forward(t, n, h, f, _ptr(x), _ld(x), _ptrs(w_gate_up), _ptrs(w_down), _ld(w_down[0]),
                                 _ptr(bias_down), ACTS[act], MODES[mode], _dt(partial_dtype), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(y), _dt(y.dtype), _stream(stream))
    _check("tp_mlp_forward", code)
    return y


def vocab_parallel_embed(ids: torch.Tensor, table: Sequence[Optional[torch.Tensor]], vocab: int, *,
                         out: Optional[torch.Tensor] = None, partials: Optional[List[torch.Tensor]] = None,
                         stream=None):
    """Vocab-parallel embedding: table[r] holds rank r's rows (ceil rule)."""
    t = len(table)
    ref = next(tb for tb in table if tb is not None)
    h = ref.shape[1]
    n = ids.numel()
    if out is None:
        out = torch.empty((n, h), dtype=ref.dtype, device=ids.device)
    code = load().vocab_parallel_embed(t, vocab, h, _ptr(ids), n, _ptrs(table), _dt(ref.dtype), _ptr(out),
                                       _ptrs(partials), _stream(stream))
    _check("vocab_parallel_embed", code)
    return out


def lm_head_sharded(x: torch.Tensor, table: Sequence[Optional[torch.Tensor]], vocab: int, *,
                    logits: Optional[torch.Tensor] = None, per_shard: bool = False,
                    shard_logits: Optional[List[torch.Tensor]] = None, out_dtype=torch.bfloat16, stream=None):
    """Vocab-sharded LM head.  Returns the concatenated [n, vocab] logits, or
    the per-shard logits when per_shard=True."""
    t = len(table)
    n, h = x.shape
    if per_shard:
        if shard_logits is None:
            per = (vocab + t - 1) // t
            widths = [max(0, min((r + 1) * per, vocab) - min(r * per, vocab)) for r in range(t)]
            shard_logits = [torch.empty((n, wd), dtype=out_dtype, device=x.device) for wd in widths]
        code = load().lm_head_sharded(t, n, h, vocab, _ptr(x), _ld(x), _ptrs(table), None, 0,
                                      _ptrs(shard_logits), _dt(shard_logits[0].dtype), _stream(stream))
        _check("lm_head_sharded", code)
        return shard_logits
    if logits is None:
        logits = torch.empty((n, vocab), dtype=out_dtype, device=x.device)
    code = load().lm_head_sharded(t, n, h, vocab, _ptr(x), _ld(x), _ptrs(table), _ptr(logits), _ld(logits),
                                  None, _dt(logits.dtype), _stream(stream))
    _check("lm_head_sharded", code)
    return logits


def tp_shard_gather(shards: Sequence[torch.Tensor], *, out: Optional[torch.Tensor] = None, stream=None):
    """Concatenate t [rows, cols_r] shards along the last dimension."""
    t = len(shards)
    rows = shards[0].shape[0]
    cols = (ctypes.c_int64 * t)(*[s.shape[1] for s in shards])
    if out is None:
        out = torch.empty((rows, sum(s.shape[1] for s in shards)), dtype=shards[0].dtype, device=shards[0].device)
    code = load().tp_shard_gather(t, rows, cols, _dt(shards[0].dtype), _ptrs(shards), _ptr(out), _stream(stream))
    _check("tp_shard_gather", code)
    return out


def tp_device_status(stream=None) -> int:
    return load().tp_device_status(_stream(stream))


def tp_collective_count() -> int:
    return load().tp_collective_count()


def tp_reset_collective_count() -> None:
    load().tp_reset_collective_count()


def tp_debug_expire_wait(limit_ns: int, stream=None) -> None:
    _check("tp_debug_expire_wait", load().tp_debug_expire_wait(limit_ns, _stream(stream)))


def tp_set_gemm_cta_pair(mode: int) -> None:
    """1: always use the CTA-pair GEMM kernel, -1: never, 0: automatic."""
    _check("tp_set_gemm_cta_pair", load().tp_set_gemm_cta_pair(mode))


def tp_set_gemm_split(mode: int, max_clusters: int = 0) -> None:
    """Split-K kernel of the fused reduce at decode sizes: 1 always (when the
    shape allows it), -1 never, 0 automatic; max_clusters > 0 caps the
    clusters resident at once."""
    _check("tp_set_gemm_split", load().tp_set_gemm_split(mode, max_clusters))


def tp_set_gemm_tile_n(n: int) -> None:
    """Force the GEMM tile width (64/128/256) for later launches; 0 = automatic."""
    _check("tp_set_gemm_tile_n", load().tp_set_gemm_tile_n(n))


def tp_mlp_forward_static(x: torch.Tensor, w_gate_up: Sequence[torch.Tensor], w_down: Sequence[torch.Tensor], *,
                          bias_down: Optional[torch.Tensor] = None, act: str = "silu", mode: str = "direct",
                          partial_dtype=torch.bfloat16, y: Optional[torch.Tensor] = None,
                          y_dtype=torch.bfloat16, stream=None):
    """tp_mlp_forward without a workspace argument, for callers that must not
    allocate device memory: the scratch is the library's own fixed 16 MiB
    device array (see include/tp.h).  Pass `y` to keep this call free of
    allocations as well; requests larger than the array raise TPError
    (TP_ERR_WORKSPACE)."""
    t = len(w_gate_up)
    n, h = x.shape
    f = w_gate_up[0].shape[0] // 2 * t
    if y is None:
        y = torch.empty((n, h), dtype=y_dtype, device=x.device)
    code = load().tp_mlp_forward_static(t, n, h, f, _ptr(x), _ld(x), _ptrs(w_gate_up), _ptrs(w_down),
                                        _ld(w_down[0]), _ptr(bias_down), ACTS[act], MODES[mode], _dt(partial_dtype),
                                        _ptr(y), _dt(y.dtype), _stream(stream))
    _check("tp_mlp_forward_static", code)
    return y


def tp_mlp_forward_host(x_host: torch.Tensor, w_gate_up: Sequence[torch.Tensor], w_down: Sequence[torch.Tensor], *,
                        y_host: torch.Tensor, x_dev: torch.Tensor, y_dev: torch.Tensor, workspace: torch.Tensor,
                        bias_down: Optional[torch.Tensor] = None, act: str = "silu", mode: str = "direct",
                        partial_dtype=torch.bfloat16, chunks: int = 2, stream=None, copy_stream=None):
    """tp_mlp_forward on pinned host activations with chunked, overlapped
    copies (see include/tp.h).  Returns y_host; the work is complete when
    `stream` is."""
    assert x_host.is_pinned() and y_host.is_pinned(), "host buffers must be page-locked"
    t = len(w_gate_up)
    n, h = x_host.shape
    f = w_gate_up[0].shape[0] // 2 * t
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=x_dev.device)
    code = load().tp_mlp_forward_host(t, n, h, f, _ptr(x_host), _ptrs(w_gate_up), _ptrs(w_down), _ld(w_down[0]),
                                      _ptr(bias_down), ACTS[act], MODES[mode], _dt(partial_dtype), _ptr(x_dev),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(y_dev),
                                      _ptr(y_host), _dt(y_host.dtype), chunks, _stream(stream), _stream(copy_stream))
    _check("tp_mlp_forward_host", code)
    return y_host


def tp_reduce_scatter_rmsnorm(partials: Sequence[torch.Tensor], weight: torch.Tensor, *,
                              residual: Optional[torch.Tensor] = None, eps: float = 1e-6, mode: str = "direct",
                              residual_out: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                              stream=None):
    """Sequence-parallel reduce-scatter + residual add + RMSNorm (all-gather
    in place).  Returns (residual_out or None, out)."""
    t = len(partials)
    n, h = partials[0].shape
    if out is None:
        out = torch.empty((n, h), dtype=torch.bfloat16, device=partials[0].device)
    code = load().tp_reduce_scatter_rmsnorm(t, n, h, _dt(partials[0].dtype), _ptrs(partials), _ptr(residual),
                                            _ptr(weight), eps, MODES[mode], _ptr(residual_out), _ptr(out),
                                            _stream(stream))
    _check("tp_reduce_scatter_rmsnorm", code)
    return residual_out, out
