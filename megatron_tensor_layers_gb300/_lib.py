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
import threading
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
    "tp_reduce_scatter_rmsnorm", "tp_set_gemm_split", "tp_debug_gemm_plan", "tp_mlp_host_blocks",
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
        "tp_debug_gemm_plan": (I32, [I64, I64, I64, I32, I32, I32, I32, P, P, P]),
        "tp_set_gemm_tile_n": (I32, [I32]),
        "tp_set_gemm_cta_pair": (I32, [I32]),
        "tp_set_gemm_split": (I32, [I32, I32]),
        "tp_reduce_scatter_rmsnorm": (I32, [I32, I64, I64, I32, P, P, P, ctypes.c_float, I32, P, P, P]),
        "tp_mlp_forward_host": (I32, [I32, I64, I64, I64, P, P, P, I64, P, I32, I32, I32, P, P, ctypes.c_size_t, P, P,
                                      I32, I32, P, P]),
        "tp_mlp_forward_static": (I32, [I32, I64, I64, I64, P, I64, P, P, I64, P, I32, I32, I32, P, I32, P]),
        "tp_mlp_host_blocks": (I32, [I64, I32, P, I32]),
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


# The current stream as a raw handle, without building a torch Stream object
# (torch's own kernel launchers use the same entry point); older builds fall
# back to torch.cuda.current_stream().
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_raw_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream) -> Optional[int]:
    if stream is None:
        if _raw_stream is not None and _raw_device is not None:
            return _raw_stream(_raw_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


# Host arrays of per-shard device pointers.  The C ABI reads them during the
# call only, so each thread reuses a small ring of arrays instead of building
# new ctypes objects on every call (a call passes at most three lists).  An
# array returned by _ptrs is therefore valid only until this thread's next
# _PTR_RING calls of _ptrs: pass it straight to the C function.  While
# `prepare` records a call, every array is new (the recording keeps it).
_PTR_RING = 8
_tls = threading.local()


def _ptrs(ts: Optional[Sequence[Optional[torch.Tensor]]]):
    if ts is None:
        return None
    n = len(ts)
    if n > MAX_SHARDS or getattr(_tls, "rec", None) is not None:   # a recorded call keeps its own array
        arr = (ctypes.c_void_p * n)()
    else:
        ring = getattr(_tls, "ring", None)
        if ring is None:
            ring = _tls.ring = [(ctypes.c_void_p * MAX_SHARDS)() for _ in range(_PTR_RING)]
            _tls.next = 0
        i = _tls.next
        _tls.next = (i + 1) % _PTR_RING
        arr = ring[i]
    arr[:n] = [None if t is None else t.data_ptr() for t in ts]
    return arr


def _ld(t: torch.Tensor) -> int:
    assert t.dim() == 2 and t.stride(1) == 1, "matrices must be row-major with unit column stride"
    return t.stride(0)


def _dt(dtype) -> int:
    if dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {dtype}")
    return DTYPES[dtype]


# ----------------------------------------------------------------- launches and prepared calls
#
# Every entry point below checks its arguments, marshals them and then makes
# its C calls through _launch.  A serving loop makes the same calls on the same
# buffers step after step, and in Python the checks and the marshalling cost
# several times what the C ABI itself does.  `prepare(entry, ...)` runs an
# entry point once with its launches recorded instead of made; the returned
# PreparedCall then makes exactly those C calls, with arguments converted to
# ctypes objects once, each time it is called.


def _launch(name: str, *args) -> None:
    rec = getattr(_tls, "rec", None)
    fn = getattr(load(), name)
    if rec is not None:
        rec.append((name, fn, args))
        return
    code = fn(*args)
    if code != TP_OK:
        raise TPError(name, code)


def _frozen(name: str, fn, args):
    """A fresh handle of C function `name` that does no argument conversion,
    and `args` converted once to ctypes objects of the declared types (ctypes
    arrays pass as pointers to their first element, None as a null pointer)."""
    if len(fn.argtypes) != len(args):
        raise TypeError(f"{name} takes {len(fn.argtypes)} arguments, {len(args)} were recorded")
    raw = load()[name]
    raw.restype = fn.restype
    return name, raw, tuple(a if isinstance(a, ctypes.Array) else ty(a) for ty, a in zip(fn.argtypes, args))


class PreparedCall:
    """An entry point's C calls with their arguments checked and marshalled once.

    Calling it makes the same calls again, on the stream that was current (or
    given) when it was prepared, and returns what the entry point returned then
    (the same output tensors).  It keeps the tensors it was prepared with alive;
    their contents may change between calls (that is the use: new inputs written
    into the same buffers), but their storage must not be replaced or resized.
    Ownership, layout and error behaviour are those of the entry point: a C call
    that fails raises TPError, and later calls of the same PreparedCall are not
    made."""

    __slots__ = ("_calls", "_keep", "result")

    def __init__(self, calls, keep, result):
        self._calls = tuple(_frozen(name, fn, args) for name, fn, args in calls)
        self._keep = keep
        self.result = result

    def __call__(self):
        for name, raw, args in self._calls:
            code = raw(*args)
            if code != TP_OK:
                raise TPError(name, code)
        return self.result

    def __len__(self) -> int:
        return len(self._calls)


def prepare(entry, *args, **kwargs) -> PreparedCall:
    """Check and marshal `entry(*args, **kwargs)` (an entry point of this
    module) once, without launching anything, and return the PreparedCall that
    launches it.  Outputs the entry point would allocate are allocated now."""
    if getattr(_tls, "rec", None) is not None:
        raise RuntimeError("prepare() does not nest")
    rec = []
    _tls.rec = rec
    try:
        result = entry(*args, **kwargs)
    finally:
        _tls.rec = None
    if not rec:
        raise ValueError(f"{getattr(entry, '__name__', entry)!s} made no launch to prepare")
    return PreparedCall(rec, (args, kwargs), result)


# ----------------------------------------------------------------- argument checks
#
# The C ABI takes raw device pointers with one row stride per list of shards,
# so it cannot see a tensor's size, device or layout.  The binding checks them
# before any call: shapes, dtypes and strides first, then that every tensor is
# on the GPU (a host pointer handed to a kernel would be an illegal address).


# Each check takes a fast path (plain comparisons) and builds its message only
# when it fails.  `name` is a string or a (list name, index) pair, formatted
# only for the message.

def _nm(name) -> str:
    return f"{name[0]}[{name[1]}]" if isinstance(name, tuple) else name


def _tensor(name, t, shape=None, dtypes=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{_nm(name)} must be a torch.Tensor, got {type(t).__name__}")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{_nm(name)} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{_nm(name)} has dtype {t.dtype}, expected one of {list(dtypes)}")
    return t


def _matrix(name, t, shape=None, dtypes=None) -> torch.Tensor:
    """A row-major 2-D tensor (unit column stride, any row stride)."""
    _tensor(name, t, shape, dtypes)
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1) or t.stride(0) < t.shape[1]:
        raise ValueError(f"{_nm(name)} must be a row-major matrix with unit column stride")
    return t


def _dense(name, t, shape=None, dtypes=None) -> torch.Tensor:
    _tensor(name, t, shape, dtypes)
    if not t.is_contiguous():
        raise ValueError(f"{_nm(name)} must be contiguous")
    return t


def _matrices(name: str, ts, shape, dtypes) -> int:
    """Every ts[r] is a row-major matrix of `shape` and one of `dtypes`, all
    with one row stride, which is returned (the ABI takes one per list)."""
    ld = None
    for r, t in enumerate(ts):
        if not (isinstance(t, torch.Tensor) and t.shape == shape and t.dtype in dtypes and t.dim() == 2):
            _matrix((name, r), t, shape, dtypes)
        s0, s1 = t.stride()
        if (s1 != 1 and shape[1] > 1) or s0 < shape[1]:
            _matrix((name, r), t, shape, dtypes)
        if ld is None:
            ld = s0
        elif s0 != ld:
            _same_ld(name, ts)
    return ld


def _denses(name: str, ts, shape, dtypes) -> None:
    """Every ts[r] is a contiguous tensor of `shape` and one of `dtypes`."""
    for r, t in enumerate(ts):
        if not (isinstance(t, torch.Tensor) and t.shape == shape and t.dtype in dtypes and t.is_contiguous()):
            _dense((name, r), t, shape, dtypes)


def _same_ld(name: str, ts: Sequence[torch.Tensor]) -> None:
    ld = ts[0].stride(0)
    for t in ts:
        if t.stride(0) != ld:
            lds = {u.stride(0) for u in ts}
            raise ValueError(f"every {name}[r] must have the same row stride (got {sorted(lds)})")


def _shard_count(name: str, ts) -> int:
    if ts is None or len(ts) < 1 or len(ts) > MAX_SHARDS:
        raise ValueError(f"{name} must hold 1..{MAX_SHARDS} shards")
    return len(ts)


def _on_gpu(*groups) -> None:
    """Every tensor (or list of tensors; None entries skipped) is a CUDA tensor of one device."""
    dev = None
    for g in groups:
        if g is None:
            continue
        for t in ((g,) if isinstance(g, torch.Tensor) else g):
            if t is None:
                continue
            d = t.get_device()
            if d < 0:
                raise ValueError("every tensor argument must be a CUDA tensor (the library has no CPU path)")
            if dev is None:
                dev = d
            elif d != dev:
                raise ValueError(f"tensor arguments span devices cuda:{dev} and cuda:{d}")


BF16 = (torch.bfloat16,)
BF16_F32 = (torch.bfloat16, torch.float32)


# ----------------------------------------------------------------- entry points

def tp_abi_version() -> int:
    return load().tp_abi_version()


def tp_linear_col(x: torch.Tensor, w: Sequence[torch.Tensor], *, act: str = "none",
                  bias: Optional[Sequence[torch.Tensor]] = None, gather_output: bool = False,
                  y=None, y_dtype=torch.bfloat16, stream=None):
    """ColumnParallelLinear over t shards.  w[r] is [out/t, in] (act="none") or
    rank r's merged [gate; up] block [2*out/t, in].  Returns the list of
    per-shard outputs, or the gathered [n, out] tensor if gather_output."""
    t = _shard_count("w", w)
    n, k = _matrix("x", x, dtypes=BF16).shape
    if act not in ACTS:
        raise ValueError(f"act must be one of {list(ACTS)}")
    rows = w[0].shape[0] if w[0].dim() == 2 else -1
    ldw = _matrices("w", w, (rows, k), BF16)
    gated = act != "none"
    if gated and rows % 2:
        raise ValueError("a gated weight block holds gate rows then as many up rows: its row count must be even")
    os_ = rows // (2 if gated else 1)
    out_full = os_ * t
    if bias is not None:
        if len(bias) != t:
            raise ValueError("bias must hold one vector per shard")
        for r in range(t):
            _dense(("bias", r), bias[r], (os_,), BF16)
    if y is None:
        if gather_output:
            y = torch.empty((n, out_full), dtype=y_dtype, device=x.device)
        else:
            y = [torch.empty((n, os_), dtype=y_dtype, device=x.device) for _ in range(t)]
    ys = [y] if gather_output else list(y)
    if len(ys) != (1 if gather_output else t):
        raise ValueError("y must be one tensor with gather_output, else one per shard")
    ldy = _matrices("y", ys, (n, out_full if gather_output else os_), BF16_F32)
    for yi in ys:
        if yi.dtype is not ys[0].dtype:
            raise TypeError("every y[r] must have the same dtype")
    _on_gpu(x, w, bias, ys)
    _launch("tp_linear_col", t, n, k, out_full, _ptr(x), _ld(x), _ptrs(w), ldw, _ptrs(bias),
            ACTS[act], int(gather_output), _ptrs(ys), ldy, _dt(ys[0].dtype), _stream(stream))
    return y


def tp_linear_row(x: Sequence[torch.Tensor], w: Sequence[torch.Tensor], *, bias: Optional[torch.Tensor] = None,
                  reduce_results: bool = True, mode: str = "direct", partial_dtype=torch.bfloat16,
                  partials: Optional[List[torch.Tensor]] = None, y: Optional[torch.Tensor] = None,
                  y_dtype=torch.bfloat16, stream=None):
    """RowParallelLinear: x[r] [n, in/t], w[r] [out, in/t].  Returns y (the
    all-reduced sum) when reduce_results, else the list of partials."""
    t = _shard_count("w", w)
    if len(x) != t:
        raise ValueError("x and w must hold the same number of shards")
    n, ks = _matrix("x[0]", x[0], dtypes=BF16).shape
    out = _matrix("w[0]", w[0], dtypes=BF16).shape[0]
    ldx = _matrices("x", x, (n, ks), BF16)
    ldw = _matrices("w", w, (out, ks), BF16)
    if mode not in MODES:
        raise ValueError(f"mode must be one of {list(MODES)}")
    if bias is not None:
        _dense("bias", bias, (out,), BF16)
    dev = x[0].device
    if mode != "fused" and partials is None:
        partials = [torch.empty((n, out), dtype=partial_dtype, device=dev) for _ in range(t)]
    if reduce_results and y is None:
        y = torch.empty((n, out), dtype=y_dtype, device=dev)
    if partials is not None:
        if len(partials) != t:
            raise ValueError("partials must hold one buffer per shard")
        _matrix(("partials", 0), partials[0], (n, out), BF16_F32)
        _matrices("partials", partials, (n, out), (partials[0].dtype,))
    if y is not None:
        _matrix("y", y, (n, out), BF16_F32)
    _on_gpu(x, w, bias, partials, y)
    ldp = _ld(partials[0]) if partials is not None else out
    pdt = partials[0].dtype if partials is not None else partial_dtype
    _launch("tp_linear_row", t, n, ks * t, out, _ptrs(x), ldx, _ptrs(w), ldw, _ptr(bias),
            int(reduce_results), MODES[mode], _dt(pdt), _ptrs(partials), ldp,
            _ptr(y), _ld(y) if y is not None else out, _dt(y.dtype) if y is not None else 0,
            _stream(stream))
    return y if reduce_results else partials


def tp_shard_reduce(partials: Sequence[torch.Tensor], *, out: Optional[torch.Tensor] = None, out_dtype=None,
                    mode: str = "direct", hop_dtype=torch.float32, replicate: bool = False,
                    alloc_out: bool = True, stream=None):
    """All-reduce (sum) of t equally shaped partial buffers."""
    t = _shard_count("partials", partials)
    p0 = _dense("partials[0]", partials[0], dtypes=BF16_F32)
    shape, dt = p0.shape, p0.dtype
    for r, p in enumerate(partials):
        if not (isinstance(p, torch.Tensor) and p.shape == shape and p.dtype is dt and p.is_contiguous()):
            _dense(("partials", r), p, shape, (dt,))
    if mode not in ("direct", "ring"):
        raise ValueError("mode must be 'direct' or 'ring'")
    if out is None and alloc_out and not replicate:
        out = torch.empty(p0.shape, dtype=out_dtype or p0.dtype, device=p0.device)
    if out is not None:
        _dense("out", out, dtypes=BF16_F32)
        if out.numel() != p0.numel():
            raise ValueError(f"out holds {out.numel()} elements, the partials {p0.numel()}")
    _on_gpu(partials, out)
    _launch("tp_shard_reduce", t, p0.numel(), _dt(p0.dtype), _ptrs(partials), _ptr(out),
            _dt(out.dtype) if out is not None else 0, MODES[mode], _dt(hop_dtype),
            int(replicate), _stream(stream))
    return out


def _mlp_args(x, w_gate_up, w_down, bias_down, act, mode):
    """Shapes of the MLP entry points: returns (t, n, h, f)."""
    t = _shard_count("w_gate_up", w_gate_up)
    if len(w_down) != t:
        raise ValueError("w_gate_up and w_down must hold the same number of shards")
    if act not in ACTS or act == "none":
        raise ValueError("act must be 'silu' or 'gelu_tanh' (the MLP is gated)")
    if mode not in MODES:
        raise ValueError(f"mode must be one of {list(MODES)}")
    n, h = _matrix("x", x, dtypes=BF16).shape
    rows = w_gate_up[0].shape[0] if w_gate_up[0].dim() == 2 else -1
    if rows % 2:
        raise ValueError("w_gate_up[r] holds gate rows then as many up rows: its row count must be even")
    fs = rows // 2
    _denses("w_gate_up", w_gate_up, (2 * fs, h), BF16)
    _matrices("w_down", w_down, (h, fs), BF16)
    if bias_down is not None:
        _dense("bias_down", bias_down, (h,), BF16)
    return t, n, h, fs * t


def tp_mlp_workspace_size(t: int, n: int, h: int, f: int, mode: str = "direct", partial_dtype=torch.bfloat16) -> int:
    return load().tp_mlp_workspace_size(t, n, h, f, MODES[mode], _dt(partial_dtype))


def tp_mlp_forward(x: torch.Tensor, w_gate_up: Sequence[torch.Tensor], w_down: Sequence[torch.Tensor], *,
                   bias_down: Optional[torch.Tensor] = None, act: str = "silu", mode: str = "direct",
                   partial_dtype=torch.bfloat16, workspace: Optional[torch.Tensor] = None,
                   y: Optional[torch.Tensor] = None, y_dtype=torch.bfloat16, stream=None):
    """Tensor-parallel MLP block Y = sum_r act(X A_r) B_r.  w_gate_up[r] is
    [2f/t, h] (gate rows then up rows), w_down[r] is [h, f/t]."""
    t, n, h, f = _mlp_args(x, w_gate_up, w_down, bias_down, act, mode)
    if workspace is None:
        need = tp_mlp_workspace_size(t, n, h, f, mode, partial_dtype)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    if y is None:
        y = torch.empty((n, h), dtype=y_dtype, device=x.device)
    _dense("workspace", workspace)
    _dense("y", y, (n, h), BF16_F32)
    _on_gpu(x, w_gate_up, w_down, bias_down, workspace, y)
    _launch("tp_mlp_forward", t, n, h, f, _ptr(x), _ld(x), _ptrs(w_gate_up), _ptrs(w_down), _ld(w_down[0]),
            _ptr(bias_down), ACTS[act], MODES[mode], _dt(partial_dtype), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(y), _dt(y.dtype), _stream(stream))
    return y


def vocab_parallel_embed(ids: torch.Tensor, table: Sequence[Optional[torch.Tensor]], vocab: int, *,
                         out: Optional[torch.Tensor] = None, partials: Optional[List[torch.Tensor]] = None,
                         stream=None):
    """Vocab-parallel embedding: table[r] holds rank r's rows (ceil rule)."""
    t = _shard_count("table", table)
    _dense("ids", ids, dtypes=(torch.int32,))
    if ids.dim() != 1:
        raise ValueError("ids must be a 1-D int32 tensor")
    ref = next((tb for tb in table if tb is not None), None)
    if ref is None:
        raise ValueError("table holds no shard")
    h = _dense("table shard", ref, dtypes=BF16_F32).shape[1] if ref.dim() == 2 else -1
    per = (vocab + t - 1) // t
    for r in range(t):
        rows_r = max(0, min((r + 1) * per, vocab) - min(r * per, vocab))
        if table[r] is None:
            if rows_r:
                raise ValueError(f"table[{r}] is None but rank {r} owns {rows_r} ids")
            continue
        _dense(("table", r), table[r], (rows_r, h), (ref.dtype,))
    n = ids.numel()
    if out is None:
        out = torch.empty((n, h), dtype=ref.dtype, device=ids.device)
    _dense("out", out, (n, h), (ref.dtype,))
    if partials is not None:
        if len(partials) != t:
            raise ValueError("partials must hold one buffer per shard")
        for r in range(t):
            _dense(("partials", r), partials[r], (n, h), (ref.dtype,))
    _on_gpu(ids, table, out, partials)
    _launch("vocab_parallel_embed", t, vocab, h, _ptr(ids), n, _ptrs(table), _dt(ref.dtype), _ptr(out),
            _ptrs(partials), _stream(stream))
    return out


def lm_head_sharded(x: torch.Tensor, table: Sequence[Optional[torch.Tensor]], vocab: int, *,
                    logits: Optional[torch.Tensor] = None, per_shard: bool = False,
                    shard_logits: Optional[List[torch.Tensor]] = None, out_dtype=torch.bfloat16, stream=None):
    """Vocab-sharded LM head.  Returns the concatenated [n, vocab] logits, or
    the per-shard logits when per_shard=True."""
    t = _shard_count("table", table)
    n, h = _matrix("x", x, dtypes=BF16).shape
    per = (vocab + t - 1) // t
    widths = [max(0, min((r + 1) * per, vocab) - min(r * per, vocab)) for r in range(t)]
    for r in range(t):
        if table[r] is None:
            if widths[r]:
                raise ValueError(f"table[{r}] is None but rank {r} owns {widths[r]} ids")
            continue
        _dense(("table", r), table[r], (widths[r], h), BF16)
    if per_shard:
        if shard_logits is None:
            shard_logits = [torch.empty((n, wd), dtype=out_dtype, device=x.device) for wd in widths]
        if len(shard_logits) != t:
            raise ValueError("shard_logits must hold one buffer per shard")
        for r in range(t):
            _dense(("shard_logits", r), shard_logits[r], (n, widths[r]), (shard_logits[0].dtype,) if r else BF16_F32)
        _on_gpu(x, table, shard_logits)
        _launch("lm_head_sharded", t, n, h, vocab, _ptr(x), _ld(x), _ptrs(table), None, 0,
                _ptrs(shard_logits), _dt(shard_logits[0].dtype), _stream(stream))
        return shard_logits
    if logits is None:
        logits = torch.empty((n, vocab), dtype=out_dtype, device=x.device)
    _matrix("logits", logits, (n, vocab), BF16_F32)
    _on_gpu(x, table, logits)
    _launch("lm_head_sharded", t, n, h, vocab, _ptr(x), _ld(x), _ptrs(table), _ptr(logits), _ld(logits),
            None, _dt(logits.dtype), _stream(stream))
    return logits


def tp_shard_gather(shards: Sequence[torch.Tensor], *, out: Optional[torch.Tensor] = None, stream=None):
    """Concatenate t [rows, cols_r] shards along the last dimension."""
    t = _shard_count("shards", shards)
    s0 = _dense("shards[0]", shards[0], dtypes=BF16_F32)
    if s0.dim() != 2:
        raise ValueError("shards must be 2-D")
    rows = s0.shape[0]
    for r in range(t):
        _dense(("shards", r), shards[r], dtypes=(s0.dtype,))
        if shards[r].dim() != 2 or shards[r].shape[0] != rows:
            raise ValueError(f"shards[{r}] must be [{rows}, cols_r]")
    cols = (ctypes.c_int64 * t)(*[s.shape[1] for s in shards])
    if out is None:
        out = torch.empty((rows, sum(s.shape[1] for s in shards)), dtype=shards[0].dtype, device=shards[0].device)
    _dense("out", out, (rows, sum(s.shape[1] for s in shards)), (s0.dtype,))
    _on_gpu(shards, out)
    _launch("tp_shard_gather", t, rows, cols, _dt(shards[0].dtype), _ptrs(shards), _ptr(out), _stream(stream))
    return out


def tp_device_status(stream=None) -> int:
    return load().tp_device_status(_stream(stream))


def tp_collective_count() -> int:
    return load().tp_collective_count()


def tp_reset_collective_count() -> None:
    load().tp_reset_collective_count()


def tp_debug_gemm_plan(m: int, n: int, k: int, *, groups: int = 1, segs: int = 1, gated: bool = False,
                       sms: int = 152):
    """The GEMM kernel the library would choose (host logic only): returns
    (kind, tile_n, cluster) with kind "single", "pair" or "split"."""
    kind, bn, cs = I32(), I32(), I32()
    _check("tp_debug_gemm_plan", load().tp_debug_gemm_plan(m, n, k, groups, segs, int(gated), sms, ctypes.byref(kind),
                                                           ctypes.byref(bn), ctypes.byref(cs)))
    return ("single", "pair", "split")[kind.value], bn.value, cs.value


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
    """Force the GEMM tile width (64/96/128/256) for later launches; 0 = automatic."""
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
    t, n, h, f = _mlp_args(x, w_gate_up, w_down, bias_down, act, mode)
    if y is None:
        y = torch.empty((n, h), dtype=y_dtype, device=x.device)
    _dense("y", y, (n, h), BF16_F32)
    _on_gpu(x, w_gate_up, w_down, bias_down, y)
    _launch("tp_mlp_forward_static", t, n, h, f, _ptr(x), _ld(x), _ptrs(w_gate_up), _ptrs(w_down),
            _ld(w_down[0]), _ptr(bias_down), ACTS[act], MODES[mode], _dt(partial_dtype),
            _ptr(y), _dt(y.dtype), _stream(stream))
    return y


def tp_mlp_host_blocks(n: int, chunks: int) -> List[int]:
    """Boundaries of the row blocks tp_mlp_forward_host runs n tokens in: block b
    covers rows [starts[b], starts[b + 1])."""
    lib = load()
    k = lib.tp_mlp_host_blocks(n, chunks, None, 0)
    if k < 0:
        raise ValueError("n must be >= 0 and chunks in 1..64")
    starts = (ctypes.c_int64 * (k + 1))()
    lib.tp_mlp_host_blocks(n, chunks, starts, k)
    return list(starts)


def tp_mlp_host_workspace_size(t: int, n: int, h: int, f: int, chunks: int, mode: str = "direct",
                               partial_dtype=torch.bfloat16) -> int:
    """Workspace bytes tp_mlp_forward_host needs: one MLP of its tallest row block."""
    s = tp_mlp_host_blocks(n, chunks)
    rows = max((b - a for a, b in zip(s, s[1:])), default=0)
    return tp_mlp_workspace_size(t, rows, h, f, mode, partial_dtype)


def tp_mlp_forward_host(x_host: torch.Tensor, w_gate_up: Sequence[torch.Tensor], w_down: Sequence[torch.Tensor], *,
                        y_host: torch.Tensor, x_dev: torch.Tensor, y_dev: torch.Tensor, workspace: torch.Tensor,
                        bias_down: Optional[torch.Tensor] = None, act: str = "silu", mode: str = "direct",
                        partial_dtype=torch.bfloat16, chunks: int = 2, stream=None, copy_stream=None):
    """tp_mlp_forward on pinned host activations with chunked, overlapped
    copies (see include/tp.h).  The workspace holds one MLP of the tallest
    row block (tp_mlp_host_workspace_size).  Returns y_host; the work is
    complete when `stream` is."""
    if not (isinstance(x_host, torch.Tensor) and isinstance(y_host, torch.Tensor)
            and (x_host.numel() == 0 or x_host.is_pinned()) and (y_host.numel() == 0 or y_host.is_pinned())):
        raise ValueError("x_host and y_host must be page-locked host tensors")
    t, n, h, f = _mlp_args(x_dev, w_gate_up, w_down, bias_down, act, mode)
    _dense("x_host", x_host, (n, h), BF16)
    _dense("x_dev", x_dev, (n, h), BF16)
    _dense("y_host", y_host, (n, h), BF16_F32)
    _dense("y_dev", y_dev, (n, h), (y_host.dtype,))
    _dense("workspace", workspace)
    _on_gpu(x_dev, w_gate_up, w_down, bias_down, y_dev, workspace)
    if copy_stream is None:
        copy_stream = torch.cuda.Stream(device=x_dev.device)
    _launch("tp_mlp_forward_host", t, n, h, f, _ptr(x_host), _ptrs(w_gate_up), _ptrs(w_down), _ld(w_down[0]),
            _ptr(bias_down), ACTS[act], MODES[mode], _dt(partial_dtype), _ptr(x_dev),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(y_dev),
            _ptr(y_host), _dt(y_host.dtype), chunks, _stream(stream), _stream(copy_stream))
    return y_host


def tp_reduce_scatter_rmsnorm(partials: Sequence[torch.Tensor], weight: torch.Tensor, *,
                              residual: Optional[torch.Tensor] = None, eps: float = 1e-6, mode: str = "direct",
                              residual_out: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                              stream=None):
    """Sequence-parallel reduce-scatter + residual add + RMSNorm (all-gather
    in place).  Returns (residual_out or None, out)."""
    t = _shard_count("partials", partials)
    p0 = _dense("partials[0]", partials[0], dtypes=BF16_F32)
    if p0.dim() != 2:
        raise ValueError("partials must be [n, h]")
    n, h = p0.shape
    for r in range(t):
        _dense(("partials", r), partials[r], (n, h), (p0.dtype,))
    if mode not in ("direct", "ring"):
        raise ValueError("mode must be 'direct' or 'ring'")
    _dense("weight", weight, (h,), BF16)
    if residual is not None:
        _dense("residual", residual, (n, h), BF16)
    if residual_out is not None:
        _dense("residual_out", residual_out, (n, h), BF16)
    if out is None:
        out = torch.empty((n, h), dtype=torch.bfloat16, device=partials[0].device)
    _dense("out", out, (n, h), BF16)
    _on_gpu(partials, weight, residual, residual_out, out)
    _launch("tp_reduce_scatter_rmsnorm", t, n, h, _dt(partials[0].dtype), _ptrs(partials), _ptr(residual),
            _ptr(weight), eps, MODES[mode], _ptr(residual_out), _ptr(out),
            _stream(stream))
    return residual_out, out
