"""The multi-GPU host logic on CPU: two gloo ranks aggregate like replicas.

Each rank reports its own units and time; the job rate is all ranks' units
over the slowest rank's time (the data path has no collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    seconds = 1.0 + rank          # rank 1 is the slow one
    rate, t = bench.whole_job_rate(64 * 100, seconds, world)
    out[rank] = (rate, t, bench.max_over_ranks(float(rank * 10), world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            rate, t, mx = out[r]
            assert t == pytest.approx(2.0)
            assert rate == pytest.approx(2 * 64 * 100 / 2.0)
            assert mx == pytest.approx(10.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(100, 2.0, 1) == (50.0, 2.0)
