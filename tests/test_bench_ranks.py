"""bench.py's multi-rank timing: each rank runs its own replica of the step
(no data-path collective); the reported time is the maximum over ranks.
Checked with two gloo ranks on the CPU."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, values, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank])
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        values = [3.5, 7.25]
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, values, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 7.25, 1: 7.25}


def test_max_over_ranks_without_group():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
