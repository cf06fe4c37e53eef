"""Multi-rank host logic on CPU: two gloo ranks shard a batch by rows (every row
exactly once, no overlap) and agree on the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, rows, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from softmax_topk_gb300 import multi
    b, e = multi.shard_rows(rows, rank, world)
    bounds = [None] * world
    dist.all_gather_object(bounds, (b, e))
    slowest = multi.max_over_ranks(1.5 + rank)        # rank 1 is the slow one
    rate = multi.whole_job_rate(units_per_rank=e - b, world=world, max_seconds=slowest)
    out.put((rank, bounds, slowest, rate))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("rows", [0, 1, 7, 4096])
def test_two_gloo_ranks_shard_rows_and_agree_on_time(rows):
    import __graft_entry__
    __graft_entry__._builder().build()   # the package loads the library on import
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, rows, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, bounds, slowest, rate in results:
        covered = [r for b, e in bounds for r in range(b, e)]
        assert covered == list(range(rows))           # every row once, in order
        assert max(e - b for b, e in bounds) - min(e - b for b, e in bounds) <= 1
        assert slowest == 2.5
        assert rate >= 0


def test_shard_rows_rejects_bad_arguments():
    from softmax_topk_gb300 import multi
    with pytest.raises(ValueError):
        multi.shard_rows(10, 2, 2)
    with pytest.raises(ValueError):
        multi.whole_job_rate(1, 1, 0.0)
