"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2): every rank runs its own replica
(no data-path collective), the timing is the max over ranks and `value` counts all ranks' tokens."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 100.0 + 50.0 * rank          # rank 1 is slower
    t = bench.max_over_ranks(local_ms, world, "cpu")
    results[rank] = (t, bench.whole_job_value(6152, 10, world, t))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 150.0
    assert res[0][1] == pytest.approx(2 * 6152 * 10 / 0.150)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.whole_job_value(100, 4, 1, 1000.0) == pytest.approx(400.0)
