"""The bench's multi-rank arithmetic on CPU: two gloo ranks (127.0.0.1) agree on the max over ranks
of their timed regions, and the whole-job rate counts every rank's units over that time."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.25, 7.5, 1.0][rank]
    got = bench.max_over_ranks(torch, dist, ms, world, "cpu")
    out[rank] = (got, bench.throughput(64, world, got))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_whole_job_rate(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    expect = max([3.25, 7.5, 1.0][:world])
    assert sorted(res) == list(range(world))
    for got, rate in res.values():
        assert got == expect
        assert rate == pytest.approx(64 * world / (expect / 1e3))


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(torch, None, 2.5, 1, "cpu") == 2.5
    assert bench.throughput(64, 1, 0.5) == pytest.approx(128000.0)
