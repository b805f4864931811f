"""The N>1 path of bench.py on CPU: two gloo ranks run independent replicas
(distinct chunk seeds, no data-path collective) and the job throughput is all
ranks' chunks over the slowest rank's time."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    def reduce_max(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return t.item()

    local_ms = 1000.0 * (rank + 1)                  # rank 1 is the slow one
    value, ms_step = bench.job_throughput(local_ms, 10, 32, world, reduce_max)
    seeds = [bench.replica_seed(2000, rank, 32) + b for b in range(32)]
    q.put((rank, value, ms_step, seeds))
    dist.destroy_process_group()


def test_two_replicas_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, v0, ms0, s0), (r1, v1, ms1, s1) = res
    assert ms0 == ms1 == pytest.approx(200.0)       # slowest rank: 2000 ms over 10 steps
    assert v0 == v1 == pytest.approx(2 * 32 * 30.0 / 0.2)
    assert not set(s0) & set(s1)                     # the replicas encode disjoint chunks
