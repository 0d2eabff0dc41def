"""The multi-rank path of bench.py on CPU: two gloo ranks stand in for two
GPUs (every rank runs an independent replica; the only cross-rank steps are
the barrier and the max over ranks of the timed region)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    elapsed = [0.25, 0.5][rank]                   # rank 1 is the slow one
    m = bench.max_over_ranks(dist, elapsed, torch.device("cpu"))
    out[rank] = (m, bench.whole_job_value(100.0, world, m))
    ref = bench.run_reference(type("A", (), {"ref_rows": 1, "warmup": 0, "steps": 1})(), rank, world) \
        if rank != 0 else "skipped"
    out[10 + rank] = ref
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_whole_job_value():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        for r in range(world):
            m, v = out[r]
            assert m == 0.5                        # both ranks see the slowest rank's time
            assert v == pytest.approx(100.0 * 2 / 0.5)
        assert out[11] is None                     # the reference arm does no work off rank 0


def test_cold_set_count_covers_twice_the_l2():
    """The cold-L2 timings rotate through buffer sets that together hold at
    least twice the L2 (unless the rows cap the count), and never fewer than
    two sets."""
    sys.path.insert(0, ROOT)
    import bench

    class _Props:
        L2_cache_size = 126 * 2 ** 20

    class _Cuda:
        @staticmethod
        def get_device_properties(_):
            return _Props()

    fake_torch = type("T", (), {"cuda": _Cuda})
    l2 = _Props.L2_cache_size
    for set_bytes in (16 << 10, 48 << 10, 3 << 20, 16 << 20, 18_874_368, 300 << 20, 2 << 30):
        n = bench.cold_set_count(fake_torch, set_bytes, 1 << 20)
        assert n >= 2
        assert n * set_bytes >= 2 * l2
        assert (n - 1) * set_bytes < 2 * l2 or n == 2
    assert bench.cold_set_count(fake_torch, 16 << 10, 64) == 64          # capped by the rows available
