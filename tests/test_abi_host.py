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


def test_zero_tokens_on_host(lib):
    """n = 0 is a valid call: data pointers of zero rows may be NULL, the other arguments are
    still checked, and nothing reaches CUDA (these calls run without a GPU)."""
    w, none2 = _arr(2), _arr(2, None)
    assert lib.tp_linear_col(2, 0, 64, 128, None, 64, w, 64, None, 1, 0, none2, 64, 0, None) == 0
    assert lib.tp_linear_col(2, 0, 64, 128, None, 64, w, 64, None, 0, 1, none2, 128, 1, None) == 0
    assert lib.tp_linear_col(0, 0, 64, 128, None, 64, w, 64, None, 1, 0, none2, 64, 0, None) == 1   # t still checked
    assert lib.tp_linear_col(2, 0, 64, 128, None, 64, none2, 64, None, 1, 0, none2, 64, 0, None) == 1   # weights
    for mode in (0, 1, 2):
        assert lib.tp_linear_row(2, 0, 128, 64, none2, 64, w, 64, None, 1, mode, 0, none2, 64, None, 64, 0,
                                 None) == 0
    assert lib.tp_linear_row(2, 0, 131, 64, none2, 66, w, 66, None, 1, 0, 0, none2, 64, None, 64, 0, None) == 2
    assert lib.tp_shard_reduce(2, 0, 0, none2, None, 0, 0, 0, 0, None) == 0
    assert lib.tp_shard_reduce(2, 0, 1, none2, None, 0, 0, 0, 0, None) == 4          # bf16 hops on f32 data
    for mode in (0, 2):
        assert lib.tp_mlp_forward(2, 0, 64, 128, None, 64, w, w, 64, None, 1, mode, 0, None, 0, None, 0, None) == 0
        assert lib.tp_mlp_forward_static(2, 0, 64, 128, None, 64, w, w, 64, None, 1, mode, 0, None, 0, None) == 0
        assert lib.tp_mlp_forward_host(2, 0, 64, 128, None, w, w, 64, None, 1, mode, 0, None, None, 0, None, None,
                                       0, 2, None, None) == 0
    assert lib.tp_mlp_forward(2, 0, 64, 128, None, 64, w, w, 64, None, 0, 0, 0, None, 0, None, 0, None) == 1  # act
    assert lib.tp_mlp_forward_host(2, 0, 64, 128, None, none2, w, 64, None, 1, 0, 0, None, None, 0, None, None,
                                   0, 2, None, None) == 1                            # weights still checked
    assert lib.vocab_parallel_embed(2, 10, 16, None, 0, w, 0, None, none2, None) == 0
    assert lib.vocab_parallel_embed(2, 10, 12, None, 0, w, 0, None, None, None) == 3   # 24-byte rows
    assert lib.lm_head_sharded(2, 0, 16, 10, None, 16, w, None, 0, None, 0, None) == 0
    assert lib.lm_head_sharded(2, 0, 16, 10, None, 16, w, None, 0, none2, 0, None) == 0
    assert lib.lm_head_sharded(2, 0, 12, 10, None, 16, w, None, 0, None, 0, None) == 3  # h % 8
    cols = (ctypes.c_int64 * 2)(3, 5)
    assert lib.tp_shard_gather(2, 0, cols, 0, none2, None, None) == 0
    assert lib.tp_reduce_scatter_rmsnorm(2, 0, 64, 0, none2, None, FAKE, ctypes.c_float(1e-6), 0, None, None,
                                         None) == 0
    assert lib.tp_reduce_scatter_rmsnorm(2, 0, 64, 0, none2, None, None, ctypes.c_float(1e-6), 0, None, None,
                                         None) == 1                                  # the weight is not row data


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
    # a workspace smaller than the tallest row block
    assert lib.tp_mlp_forward_host(2, 8, 64, 128, FAKE, two, two, 64, None, 1, 0, 0, FAKE, FAKE, 16, FAKE,
                                   FAKE, 0, 2, None, None) == 7


def test_host_blocks(lib):
    """The row blocks of tp_mlp_forward_host (host logic): short first and last blocks of
    e = ceil(n / (4 chunks)) rows, rounded up to 128 while at least e rows stay between them,
    and chunks - 1 middle blocks of equal height, rounded up to 128 while the last of them
    keeps rows."""
    def sizes(n, c):
        s = _lib.tp_mlp_host_blocks(n, c)
        return [b - a for a, b in zip(s, s[1:])]
    assert sizes(8192, 1) == [8192]
    assert sizes(8192, 2) == [1024, 6144, 1024]
    assert sizes(8192, 3) == [768, 3328, 3328, 768]
    assert sizes(8192, 4) == [512, 2432, 2432, 2304, 512]
    assert sizes(520, 2) == [128, 264, 128]          # ceil(520 / 8) = 65 -> 128
    assert sizes(40, 5) == [2, 9, 9, 9, 9, 2]        # 128-row edges would leave no middle
    assert sizes(257, 2) == [33, 191, 33]            # nor here more than one row
    assert sizes(3, 2) == [1, 1, 1] and sizes(2, 2) == [2] and sizes(1, 64) == [1] and sizes(0, 2) == []
    for n in (1, 2, 3, 7, 100, 129, 255, 256, 257, 1000, 4099, 8192, 70001):
        for c in (1, 2, 3, 5, 8, 17, 64):
            s = _lib.tp_mlp_host_blocks(n, c)
            b = [y - x for x, y in zip(s, s[1:])]
            assert s[0] == 0 and s[-1] == n and all(v > 0 for v in b), (n, c)
            assert len(b) <= c + 1, (n, c)
            if c > 1 and n >= 3:
                e = -(-n // (4 * c))
                assert len(b) >= 3 and b[0] == b[-1] and b[0] in (e, -(-e // 128) * 128), (n, c)
                assert sum(b[1:-1]) >= b[0] and max(b[1:-1]) - min(b[1:-2] or b[1:2]) <= 128, (n, c)
    # the C query: the count with no buffer, nothing written when the buffer is short, -1 on bad input
    assert lib.tp_mlp_host_blocks(8192, 2, None, 0) == 3
    buf = (ctypes.c_int64 * 4)(-1, -1, -1, -1)
    assert lib.tp_mlp_host_blocks(8192, 2, buf, 2) == 3 and list(buf) == [-1] * 4
    assert lib.tp_mlp_host_blocks(8192, 2, buf, 3) == 3 and list(buf) == [0, 1024, 7168, 8192]
    assert lib.tp_mlp_host_blocks(-1, 2, None, 0) == -1
    assert lib.tp_mlp_host_blocks(8, 0, None, 0) == -1 and lib.tp_mlp_host_blocks(8, 65, None, 0) == -1
    assert _lib.tp_mlp_host_workspace_size(4, 8192, 8192, 28672, 2) == _lib.tp_mlp_workspace_size(4, 6144, 8192, 28672)


def test_gemm_kernel_choice(lib):
    """The host-side plan (no CUDA call) for the shapes whose kernel choice was measured on
    GB300 (152 SMs): the bench prefill, decode, chunked prefill, the tiny MLP, the LM head
    and the 70B attention projections."""
    from megatron_tensor_layers_gb300 import _lib as tp
    plan = tp.tp_debug_gemm_plan
    h, f = 8192, 28672
    # prefill t=4, n=8192: gate_up (gated, 4 shards of 7168 H columns) and down on CTA pairs
    assert plan(8192, f // 4, h, groups=4, gated=True) == ("pair", 256, 0)
    assert plan(8192, h, f // 4, groups=4) == ("pair", 256, 0)
    # fused down at prefill: one output, t K-segments, still pairs
    assert plan(8192, h, f // 4, segs=4) == ("pair", 256, 0)
    # decode t=4: gate_up 128-wide gated tiles (448 tiles), down 256-wide (128 tiles)
    for n in (1, 16, 64):
        assert plan(n, f // 4, h, groups=4, gated=True) == ("single", 128, 0)
        assert plan(n, h, f // 4, groups=4) == ("single", 256, 0)
        # fused reduce at decode: split-K clusters of 4 over 32 tiles of 256
        assert plan(n, h, f // 4, segs=4) == ("split", 256, 4)
    # chunked prefill: pairs from 200 to 256 rows, single CTAs at 128 rows
    assert plan(256, f // 4, h, groups=4, gated=True)[0] == "pair"
    assert plan(200, f // 4, h, groups=4, gated=True)[0] == "pair"
    assert plan(128, f // 4, h, groups=4, gated=True)[0] == "single"
    assert plan(384, h, f // 4, groups=4)[0] == "single"           # pairs would add a wave
    # tiny MLP t=2, n=8: 64-wide gated tiles (96 CTAs), fused down on split-K clusters
    assert plan(8, 1536, 1024, groups=2, gated=True) == ("single", 64, 0)
    assert plan(8, 1024, 1536, segs=2)[0] == "split"
    # 70B attention, t=8 at decode: 96-wide QKV tiles (112 tiles instead of 80 of 128)
    assert plan(1, 1280, h, groups=8) == ("single", 96, 0)
    # LM head t=2, 4096 x 1024 x 151936: pairs
    assert plan(4096, 75968, 1024, groups=2) == ("pair", 256, 0)
    # a gated GEMM never takes the 96-wide tile
    for n in (1, 8, 64):
        assert plan(n, 640, h, groups=8, gated=True)[1] != 96
    assert lib.tp_debug_gemm_plan(0, 1, 1, 1, 1, 0, 152, None, None, None) == 1


def test_mlp_workspace_sizes(lib):
    """tp_mlp_workspace_size: H [n, f] bf16, plus t partials [n, h] unless the reduce
    is fused, each 256-byte aligned; a fused reduce of more than 128 rows adds the
    32 MiB + 4 KiB stream-K area of its down GEMM (optional: tp_mlp_forward also runs
    with the H bytes alone)."""
    al = lambda b: (b + 255) // 256 * 256
    ws = lambda t, n, h, f, mode, pdt: lib.tp_mlp_workspace_size(t, n, h, f, _lib.MODES[mode], pdt)
    tail = 4096 + 128 * 256 * 256 * 4
    t, h, f = 4, 8192, 28672
    for n in (1, 64, 128, 129, 8192):
        hb = al(n * f * 2)
        assert ws(t, n, h, f, "direct", 0) == hb + t * al(n * h * 2)
        assert ws(t, n, h, f, "ring", 1) == hb + t * al(n * h * 4)
        assert ws(t, n, h, f, "fused", 0) == hb + (tail if n > 128 else 0)
    assert ws(0, 8, h, f, "direct", 0) == 0 and ws(4, -1, h, f, "direct", 0) == 0


def test_small_mlp_workspace_sizes(lib):
    """A fused MLP of one to eight tokens with h a multiple of 256 up to 1024 and
    f/t a multiple of 64 (at most 128 slices of 64 columns) runs as one GEMM kernel
    plus an ordered reduce; its workspace holds the slices' fp32 partials
    [f/64][n][h] (optional: with the H bytes alone the two-GEMM path runs)."""
    al = lambda b: (b + 255) // 256 * 256
    ws = lambda t, n, h, f, mode: lib.tp_mlp_workspace_size(t, n, h, f, _lib.MODES[mode], 0)
    for n in range(1, 9):
        assert ws(2, n, 1024, 3072, "fused") == al(48 * n * 1024 * 4)
    assert ws(8, 8, 1024, 8192, "fused") == al(128 * 8 * 1024 * 4)
    assert ws(3, 5, 512, 576, "fused") == al(9 * 5 * 512 * 4)
    hb = lambda n, f: al(n * f * 2)
    assert ws(2, 9, 1024, 3072, "fused") == hb(9, 3072)          # nine tokens
    assert ws(2, 8, 1280, 3072, "fused") == hb(8, 3072)          # h above 1024
    assert ws(2, 8, 640, 3072, "fused") == hb(8, 3072)           # h not a multiple of 256
    assert ws(3, 8, 1024, 3072, "fused") == al(48 * 8 * 1024 * 4)  # three ranks of 1024 columns
    assert ws(2, 8, 1024, 2080, "fused") == hb(8, 2080)          # f/t = 1040, not a multiple of 64
    assert ws(8, 8, 1024, 8704, "fused") == hb(8, 8704)          # 136 slices
    assert ws(2, 8, 1024, 3072, "direct") == hb(8, 3072) + 2 * al(8 * 1024 * 2)
