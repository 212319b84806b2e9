"""The N > 1 path of bench.py on CPU: two gloo ranks, each timing its own
replica, agree on the slowest rank's time and report the whole-job rate."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    elapsed = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")  # rank 1 is the slow one
    ms_per_step = elapsed / 5
    q.put((rank, elapsed, bench.job_steps_per_s(ms_per_step, world)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, elapsed, value in res:
        assert elapsed == pytest.approx(20.0)
        assert value == pytest.approx(2 / (4.0 / 1e3))  # 2 replicas, 4 ms per step each
