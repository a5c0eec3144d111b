"""The bench's multi-rank host logic on CPU with gloo, world size 2: each rank runs its
own batch, the timed total is the maximum over ranks, and the whole-job value counts
every rank's work (weak scaling)."""
import os

import pytest
import torch.multiprocessing as mp


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total = 10.0 + 5.0 * rank          # rank 1 is the slow one
    got = bench.max_over_ranks(total, world, "cpu")
    q.put((rank, got, bench.rank_seeds(rank)))
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1] == 15.0
    # independent batches: the ranks draw different inputs
    assert res[0][2] != res[1][2]
    import bench
    one = bench.weak_scaling_value(1e12, 10, 1, 15.0)
    two = bench.weak_scaling_value(1e12, 10, 2, 15.0)
    assert two == pytest.approx(2 * one)
