"""The multi-rank host logic of bench.py on CPU: two gloo ranks time
different amounts and both see the slowest rank's time; the whole-job value
counts every rank's work.  (The data path itself has no collective.)"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, e2e = bench.reduce_max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")
    out[rank] = (ms, e2e, bench.whole_job_tflops(2.0e12, world, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        ms, e2e, value = res[r]
        assert ms == 2.0 and e2e == 10.0
        assert value == pytest.approx(world * 2.0e12 / 2.0e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max_over_ranks([3.5, 4.5], "cpu") == [3.5, 4.5]
    assert bench.whole_job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)
