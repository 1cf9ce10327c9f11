"""Multi-process path of bench.py on CPU (gloo, world size 2): every rank runs
its own replica, the timing is the max over ranks and the value aggregates
the units of all ranks (weak scaling)."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    assert bench.dist_env() == (rank, world, rank)
    bench._PG = dist.group.WORLD
    t_ms = bench.max_over_ranks(1.0 + rank)  # rank 1 is the slower one
    bench.barrier()
    value = bench.aggregate(10.0, world, t_ms * 1e-3)
    q.put((rank, t_ms, value))
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_ms, value in out:
        assert t_ms == 2.0                      # max over ranks
        assert abs(value - 10.0 * 2 / 2e-3) < 1e-6   # all ranks' units over the slowest time
