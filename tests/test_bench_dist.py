"""Multi-rank logic of bench.py on CPU: two gloo ranks, max-over-ranks timing and
the whole-job aggregate (every rank runs its own copy of the workload)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_time = 1.0 + rank  # rank 1 is the slow one
        t = bench.max_over_ranks(local_time)
        bench.barrier()
        out[rank] = (t, bench.aggregate_value(3.5e12, world, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        t, value = res[r]
        assert t == 2.0
        assert value == pytest.approx(3.5e12 * 2 / 2.0 / 1e12)


def test_single_process_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.aggregate_value(1e12, 1, 0.5) == pytest.approx(2.0)


def test_flop_convention_matches_pages():
    import bench
    p = dict(B=2, H=16, N=8192, d=128, causal=False)
    assert bench.flops(p, "fwd") == 4.0 * 2 * 16 * 8192 ** 2 * 128
    assert bench.flops(dict(p, causal=True), "fwd") == bench.flops(p, "fwd") / 2
    assert bench.flops(p, "fwd_bwd") == 3.5 * bench.flops(p, "fwd")
    assert bench.flops(p, "bwd") == 2.5 * bench.flops(p, "fwd")
