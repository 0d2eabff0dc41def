"""Host-side checks of the C ABI: the library loads, exports every function
include/tp.h declares, and rejects invalid arguments on the host, before any
CUDA call (so these run without a GPU)."""

import ctypes
import os
import re

import pytest

from megatron_tensor_layers_gb300 import _lib
from megatron_tensor_layers_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "tp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(names) == sorted(_lib.EXPORTED)


def test_abi_version_and_status_strings(lib):
    assert lib.tp_abi_version() == 1
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.tp_status_string(code).decode() == name


FAKE = 0x10000      # 16-byte aligned non-null address; never dereferenced on rejected calls


def _arr(n, v=FAKE):
    a = (ctypes.c_void_p * n)()
    for i in range(n):
        a[i] = v
    return a


def test_linear_col_rejects_on_host(lib):
    w = _arr(2)
    y = _arr(2)
    ok = dict(t=2, n=8, k=64, out=128, ldx=64, ldw=64, ldy=64)

    def call(**kw):
        a = {**ok, **kw}
        return lib.tp_linear_col(a["t"], a["n"], a["k"], a["out"], kw.get("x", FAKE), a["ldx"], kw.get("w", w),
                                 a["ldw"], None, kw.get("act", 0), 0, y, a["ldy"], kw.get("yd", 0), None)

    assert call(t=0) == 1 and call(t=9) == 1
    assert call(out=129) == 2                      # out_full % t
    assert call(x=FAKE + 2) == 3                   # misaligned pointer
    assert call(ldx=60) == 3                       # ld < in
    assert call(k=60, ldx=64, ldw=64) == 3         # in % 8
    assert call(yd=7) == 4
    assert call(act=9) == 1
    assert call(w=None) == 1


def test_linear_row_and_mlp_reject_on_host(lib):
    two = _arr(2)
    # in_full not divisible by t
    assert lib.tp_linear_row(2, 8, 131, 64, two, 66, two, 66, None, 1, 0, 0, two, 64, FAKE, 64, 0, None) == 2
    # FUSED without reduce_results is meaningless
    assert lib.tp_linear_row(2, 8, 128, 64, two, 64, two, 64, None, 0, 2, 0, two, 64, FAKE, 64, 0, None) == 1
    # workspace too small
    need = lib.tp_mlp_workspace_size(2, 8, 64, 128, 0, 0)
    assert need == 8 * 128 * 2 + 2 * 256 * 4 and need % 256 == 0
    assert lib.tp_mlp_forward(2, 8, 64, 128, FAKE, 64, two, two, 64, None, 1, 0, 0, FAKE, need - 1, FAKE, 0,
                              None) == 7
    assert lib.tp_mlp_forward(2, 8, 64, 128, FAKE, 64, two, two, 64, None, 0, 0, 0, FAKE, need, FAKE, 0,
                              None) == 1              # act NONE is not an MLP
    assert lib.tp_mlp_workspace_size(2, 8, 64, 128, 2, 0) == 8 * 128 * 2   # fused: no partials
    assert lib.tp_mlp_workspace_size(0, 8, 64, 128, 0, 0) == 0


def test_reduce_embed_head_gather_reject_on_host(lib):
    two = _arr(2)
    assert lib.tp_shard_reduce(2, 100, 0, two, None, 0, 0, 1, 0, None) == 1        # nowhere to write
    assert lib.tp_shard_reduce(2, 100, 1, two, FAKE, 1, 1, 0, 0, None) == 4        # bf16 hops on f32 data
    assert lib.tp_shard_reduce(2, 100, 0, two, FAKE, 0, 2, 1, 0, None) == 1        # FUSED is not a reduce mode
    assert lib.vocab_parallel_embed(2, 10, 12, FAKE, 4, two, 0, FAKE, None, None) == 3   # 24-byte rows
    assert lib.vocab_parallel_embed(0, 10, 16, FAKE, 4, two, 0, FAKE, None, None) == 1
    assert lib.vocab_parallel_embed(2, 10, 16, FAKE, 4 * (2 ** 31 - 1) + 1, two, 0, FAKE, None, None) == 1  # grid
    assert lib.vocab_parallel_embed(2, 10, 2 ** 31, FAKE, 4, two, 0, FAKE, None, None) == 1
    assert lib.lm_head_sharded(2, 4, 12, 10, FAKE, 16, two, FAKE, 16, None, 0, None) == 3
    assert lib.lm_head_sharded(2, 4, 16, 10, FAKE, 16, two, None, 0, None, 0, None) == 1
    cols = (ctypes.c_int64 * 2)(3, -1)
    assert lib.tp_shard_gather(2, 4, cols, 0, two, FAKE, None) == 1


def test_tuning_knobs_through_the_binding(lib):
    from megatron_tensor_layers_gb300 import TPError, tp_set_gemm_cta_pair, tp_set_gemm_split, tp_set_gemm_tile_n
    for mode in (1, -1, 0):
        tp_set_gemm_cta_pair(mode)
    for n in (64, 96, 128, 256, 0):
        tp_set_gemm_tile_n(n)
    for mode, cap in ((1, 3), (-1, 0), (0, 0)):
        tp_set_gemm_split(mode, cap)
    with pytest.raises(TPError):
        tp_set_gemm_cta_pair(2)
    with pytest.raises(TPError):
        tp_set_gemm_tile_n(80)
    with pytest.raises(TPError):
        tp_set_gemm_split(2)
    with pytest.raises(TPError):
        tp_set_gemm_split(0, -1)


def test_host_pipeline_rejects_on_host(lib):
    two = _arr(2)
    # missing host buffers, bad chunk counts
    assert lib.tp_mlp_forward_host(2, 8, 64, 128, None, two, two, 64, None, 1, 0, 0, FAKE, FAKE, 1 << 20, FAKE,
                                   FAKE, 0, 1, None, None) == 1
    assert lib.tp_mlp_forward_host(2, 8, 64, 128, FAKE, two, two, 64, None, 1, 0, 0, FAKE, FAKE, 1 << 20, FAKE,
                                   FAKE, 0, 0, None, None) == 1
    # a workspace smaller than one row block
    assert lib.tp_mlp_forward_host(2, 8, 64, 128, FAKE, two, two, 64, None, 1, 0, 0, FAKE, FAKE, 16, FAKE,
                                   FAKE, 0, 2, None, None) == 7
