"""Host-side checks of prepared calls (``prepare``): the entry point's checks run
once and its C calls are recorded, not made; the recorded arguments are the
marshalled ones and keep their own pointer arrays; a failing C call raises
TPError when the prepared call runs.  CPU tensors stand in for device ones
(the device check is switched off), and no recorded call that could reach a
kernel is ever made."""

import ctypes

import pytest
import torch

from megatron_tensor_layers_gb300 import _lib
from megatron_tensor_layers_gb300.build import build


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


@pytest.fixture
def host_tensors(monkeypatch, lib):
    monkeypatch.setattr(_lib, "_on_gpu", lambda *groups: None)
    return lib


def _mlp(t=2, n=8, h=256, f=1024):
    x = torch.zeros((n, h), dtype=torch.bfloat16)
    wgu = [torch.zeros((2 * f // t, h), dtype=torch.bfloat16) for _ in range(t)]
    wd = [torch.zeros((h, f // t), dtype=torch.bfloat16) for _ in range(t)]
    return x, wgu, wd


def test_prepare_records_instead_of_calling(host_tensors):
    """A workspace one byte short is rejected by the C ABI on the host: preparing
    does not reach the C function, running the prepared call does, every time."""
    x, wgu, wd = _mlp()
    need = _lib.tp_mlp_workspace_size(2, 8, 256, 1024, "direct")
    ws = torch.empty(need - 1, dtype=torch.uint8)
    y = torch.empty((8, 256), dtype=torch.bfloat16)
    plan = _lib.prepare(_lib.tp_mlp_forward, x, wgu, wd, workspace=ws, y=y, stream=0)
    assert len(plan) == 1 and plan.result is y
    for _ in range(2):
        with pytest.raises(_lib.TPError) as e:
            plan()
        assert _lib.STATUS_NAMES[e.value.code] == "TP_ERR_WORKSPACE"


def test_prepared_arguments_are_the_marshalled_ones(host_tensors):
    parts = [torch.zeros(4096, dtype=torch.bfloat16) for _ in range(4)]
    out = torch.empty(4096, dtype=torch.float32)
    plan = _lib.prepare(_lib.tp_shard_reduce, parts, out=out, mode="ring", stream=0)
    (name, raw, args), = plan._calls
    assert name == "tp_shard_reduce" and raw.argtypes is None
    decl = _lib.load().tp_shard_reduce.argtypes
    assert len(args) == len(decl)
    t, count, dt, ptrs, optr, odt, mode, hop, rep, stream = args
    assert (t.value, count.value, dt.value) == (4, 4096, _lib.DTYPES[torch.bfloat16])
    assert [ptrs[r] for r in range(4)] == [p.data_ptr() for p in parts]
    assert optr.value == out.data_ptr() and odt.value == _lib.DTYPES[torch.float32]
    assert (mode.value, hop.value, rep.value) == (_lib.MODES["ring"], _lib.DTYPES[torch.float32], 0)
    assert not stream.value
    # later marshalling (the per-thread ring of pointer arrays) leaves the recorded array alone
    others = [torch.zeros(16, dtype=torch.bfloat16) for _ in range(4)]
    for _ in range(3 * _lib._PTR_RING):
        _lib._ptrs(others)
    assert [ptrs[r] for r in range(4)] == [p.data_ptr() for p in parts]


def test_prepare_checks_like_the_entry_point(host_tensors):
    parts = [torch.zeros(64, dtype=torch.bfloat16), torch.zeros(65, dtype=torch.bfloat16)]
    with pytest.raises(ValueError):
        _lib.prepare(_lib.tp_shard_reduce, parts, stream=0)
    assert getattr(_lib._tls, "rec", None) is None
    ok = [torch.zeros(64, dtype=torch.bfloat16) for _ in range(2)]
    plan = _lib.prepare(_lib.tp_shard_reduce, ok, stream=0)
    assert plan.result.shape == (64,) and plan.result.dtype == torch.bfloat16


def test_prepare_does_not_nest(host_tensors):
    ok = [torch.zeros(64, dtype=torch.bfloat16) for _ in range(2)]
    with pytest.raises(RuntimeError):
        _lib.prepare(_lib.prepare, _lib.tp_shard_reduce, ok, stream=0)
    assert getattr(_lib._tls, "rec", None) is None
    with pytest.raises(ValueError):
        _lib.prepare(lambda: None)


def test_prepare_keeps_its_tensors(host_tensors):
    """The prepared call holds the tensors it was prepared with, so their memory
    stays allocated for as long as it can be called."""
    x, wgu, wd = _mlp()
    ws = torch.empty(_lib.tp_mlp_workspace_size(2, 8, 256, 1024, "direct"), dtype=torch.uint8)
    plan = _lib.prepare(_lib.tp_mlp_forward, x, wgu, wd, workspace=ws, stream=0)
    held = plan._keep[0]
    assert held[0] is x and held[1] is wgu and held[2] is wd and plan._keep[1]["workspace"] is ws
    name, raw, args = plan._calls[0]
    assert args[4].value == x.data_ptr() and args[13].value == ws.data_ptr()
    assert isinstance(args[6], ctypes.Array) and args[6][1] == wgu[1].data_ptr()
