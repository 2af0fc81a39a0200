"""The multi-GPU path is replicas only: each rank times its own steps and
the job's throughput is all ranks' work over the slowest rank's time.  The
aggregation runs here on two gloo ranks on the CPU (no GPU)."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _rank(rank, world, port, local_ms, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        total, value = bench.job_throughput(local_ms[rank], 2.0e9, 10, world, dist, torch.device("cpu"))
        q.put((rank, total, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(5.0, 8.0), (8.0, 5.0)])
def test_job_throughput_is_max_over_ranks(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    slowest = max(times)
    for rank, total, value in got:
        assert total == slowest
        # 2 ranks x 10 steps x 2e9 flop over the slowest rank's 8 ms
        assert value == pytest.approx(2 * 10 * 2.0e9 / (slowest * 1e-3) / 1e12)


def test_job_throughput_single_rank():
    import bench
    total, value = bench.job_throughput(4.0, 1.0e9, 4, 1)
    assert total == 4.0 and value == pytest.approx(4 * 1.0e9 / 4e-3 / 1e12)
