"""The N > 1 path of bench.py on CPU: two gloo ranks (no GPU) reduce their timings to the
slowest rank and report whole-job throughput over it, as the benchmark does for replicas."""
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


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + rank, 100.0 * (rank + 1), 5.0, 7.0 - rank]
    got = bench.reduce_max(mine, dist, "cpu")
    q.put((rank, got, bench.job_throughput(world, 128, got[1])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, thr in res:
        assert got == [11.0, 200.0, 5.0, 7.0]
        assert abs(thr - 2 * 128 / 0.2) < 1e-9
