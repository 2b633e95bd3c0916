"""The N > 1 bench path on CPU: gloo, world size 2.  Every rank runs its own
replica (no data-path collective); the step time is the max over ranks and the
value counts every rank's rows."""
import os

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]
    agg = bench.max_over_ranks(ms, torch.device("cpu"), world)
    value = bench.layer_queries_per_s(rows=1024, world=world, ms=agg)
    out[rank] = (agg, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_max_time_and_total_rows():
    port = 29000 + os.getpid() % 1000
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        agg, value = out[r]
        assert agg == 5.0
        assert abs(value - 3 * 1024 * 2 / 5e-3) < 1e-6
